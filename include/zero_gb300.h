/*
 * zero_gb300.h -- C ABI of libzero_gb300.so, the GB300 (sm_103a) ZeRO
 * sharded mixed-precision update step.
 *
 * What one step computes.  N data-parallel ranks each hold a gradient buffer
 * for the same flat parameter vector.
 *   1. Reduce-scatter.  Each element's N contributions are added in rank order
 *      0..N-1 in FP32, starting from +0.  The sum is scaled by
 *      fp32(1 / (N * loss_scale)) to the batch mean.
 *   2. Owner update.  Each owner r updates its own slice of the FP32 master
 *      weights and Adam moments m and v with the combined gradient.
 *   3. All-gather.  The updated master is rounded to BF16 (nearest, ties to
 *      even) and written into the one full working-weight view.
 * The N ranks are simulated inside one GPU: the N gradient buffers and the N
 * owners' slices all live in this device's memory, so the collectives are
 * in-device data movement.  Nothing crosses to another GPU.
 *
 * Sources (web pages; section names as printed there):
 *   - lecture deck "RC-T2: sharing data and sharing the duty to store are two
 *     different acts", note N48.  Reduce-scatter adds the contributions of the
 *     same parameter only, scales them to match a batch-mean loss and hands
 *     the result to the slice's owner.  The owner updates with its own master
 *     and m/v.  The next all-gather fetches the updated parameters.
 *   - topic page "Putting the training ledger onto multiple devices",
 *     section "one full ZeRO-3 computation".  Defines all-gather,
 *     reduce-scatter and all-reduce as data semantics, all-reduce being
 *     reduce-scatter followed by all-gather.
 *   - blog post "Data parallelism and ZeRO: how much each of the three stages
 *     saves".  Section "16 bytes per parameter" gives the per-parameter ledger
 *     2 + 2 + 4 + 4 + 4 B.  Section "three stages" and its table cover ZeRO-1/2:
 *     reduce-scatter, an owner step on 1/N of the FP32 state, then an
 *     all-gather of the BF16 weights.  They also give the bytes per parameter
 *     and the communication volume of each stage.
 *   Where the pages say nothing, this library uses these readings:
 *   - Adam with bias correction; eps is added after sqrt(v_hat).
 *   - AdamW's decoupled weight decay, applied to the master weight first.
 *   - The overflow check runs on the scaled FP32 combined gradient.
 *   - The clip coefficient is min(1, max_norm / (norm + 1e-6)).
 *
 * Layout.  The flat vector holds psi parameters, zero-padded to psi_pad, a
 * multiple of N * ZERO_PAD_UNIT.  Owner r holds the contiguous slice
 * [r*S, (r+1)*S), with S = psi_pad / N.
 *
 * Ownership.  The caller allocates and frees every device buffer: the N
 * gradient buffers, master/m/v, the BF16 working weights and the workspace.
 * The step entry points allocate nothing and keep no hidden state between
 * calls.
 *
 * Errors.  Argument errors are detected on the host before any work is
 * enqueued.  The function returns a negative zero_status and modifies
 * nothing.  A CUDA error raised while enqueueing returns ZERO_ERR_CUDA.
 */
#ifndef ZERO_GB300_H
#define ZERO_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ZERO_PAD_UNIT 128      /* psi_pad is a multiple of N * ZERO_PAD_UNIT   */
#define ZERO_MAX_RANKS 64      /* largest N accepted                           */
#define ZERO_ALIGN_BYTES 16    /* every buffer must start on this boundary     */
#define ZERO_BUCKET_ALIGN 8    /* bucket_elems must be a multiple of this      */
/* Largest element count any entry point accepts (psi, psi_pad, a shard, a
 * layer): 2^48, 1 PiB of FP32, past any device's memory.  Larger counts are
 * refused as bad arguments, so no byte size formed from one can overflow. */
#define ZERO_MAX_ELEMS (1LL << 48)

typedef enum {
    ZERO_OK = 0,              /* success; for a step: the update was applied       */
    ZERO_STEP_SKIPPED = 1,    /* the step found a non-finite gradient and skipped  */
    ZERO_ERR_ARG = -1,        /* bad size, count, pointer or hyper-parameter       */
    ZERO_ERR_ALIGN = -2,      /* a buffer not on a ZERO_ALIGN_BYTES boundary       */
    ZERO_ERR_CUDA = -3,       /* a CUDA call failed while enqueueing               */
    ZERO_ERR_TIMEOUT = -4,    /* a bounded wait inside a kernel gave up            */
    ZERO_ERR_WORKSPACE = -5,  /* workspace missing, too small or misaligned        */
    ZERO_ERR_OVERLAP = -6,    /* two buffers that must be disjoint overlap         */
    ZERO_ERR_TOO_LARGE = -7,  /* the step needs more scratch than zero_step_noalloc's
                                 fixed array holds                                 */
    ZERO_ERR_POLICY_WINDOW = -8, /* device policy: the step's t fell outside the window
                                 of bias corrections it was given; nothing changed  */
    ZERO_ERR_BOUNDS = -9      /* debug build only: a kernel found an index outside a
                                 buffer, skipped that access and did not apply the
                                 step (see zero_debug_bounds_violations)            */
} zero_status;

typedef enum {
    ZERO_GRAD_BF16 = 0,       /* gradients as BF16 (2 B per element) */
    ZERO_GRAD_FP32 = 1        /* gradients as FP32 (4 B per element) */
} zero_grad_dtype;

/* The flat layout of a list of tensors (see zero_init_layout). */
typedef struct {
    int64_t psi;        /* parameters: the sum of the tensor sizes       */
    int64_t psi_pad;    /* psi rounded up to a multiple of N * pad_unit  */
    int64_t shard;      /* S = psi_pad / N, the size of one owner's slice */
    int64_t n_tensors;
    int32_t N;          /* data-parallel ranks (the sharding factor)     */
    int32_t pad_unit;   /* ZERO_PAD_UNIT                                 */
} zero_layout;

/* Hyper-parameters of one step.  The Adam scalars are FP64, as a host holds
 * them.  The library rounds each derived scalar once to FP32:
 *   beta1, 1-beta1, beta2, 1-beta2, eps, lr/(1-beta1^t), sqrt(1-beta2^t), 1-lr*wd. */
typedef struct {
    double lr;
    double beta1;
    double beta2;
    double eps;
    double weight_decay;      /* decoupled (AdamW); 0 turns it off                */
    double max_grad_norm;     /* > 0: clip by the global L2 norm; 0: no clipping   */
    int64_t step;             /* t >= 1: count of applied steps including this one */
    int32_t skip_on_overflow; /* 1: any non-finite combined gradient skips the step */
    int32_t micro_batches;    /* k >= 2: the step's gradient is accumulated over k
                                 micro-batches through the plan entry points (each
                                 micro-batch's buckets reduce-scattered as they
                                 arrive); 0 or 1: one batch                         */
    int64_t bucket_elems;     /* > 0: walk the flat vector in buckets of this many
                                 elements (a multiple of ZERO_BUCKET_ALIGN); 0: one
                                 bucket                                            */
} zero_adam_hparams;

/* Outcome of one step, written by the device at the end of the step. */
typedef struct {
    int32_t status;           /* ZERO_OK (applied), ZERO_STEP_SKIPPED, ZERO_ERR_TIMEOUT,
                                 ZERO_ERR_POLICY_WINDOW or (debug build) ZERO_ERR_BOUNDS */
    uint32_t found_nonfinite; /* 1 if any combined gradient element was inf or NaN        */
    float grad_norm;          /* L2 norm of the combined batch-mean gradient, before clip */
    float clip_coef;          /* factor applied to the gradient (1 without clipping)      */
} zero_step_result;

/* Flat layout of n_tensors tensors with the given element counts,
 * concatenated in order with no gaps.  The vector is padded with zeros up to
 * psi_pad, a multiple of N * ZERO_PAD_UNIT, so that every owner's slice has
 * the same size S = psi_pad / N.  That is each rank's 1/N share
 * (RC-T2, slide b1 and note N47; DP-ZeRO blog, "three stages").
 *   tensor_numel    host array of n_tensors sizes (>= 0); may be NULL if n_tensors == 0
 *   N               ranks, 1 .. ZERO_MAX_RANKS
 *   out             host struct, filled on success
 *   tensor_offsets  host array of n_tensors int64 (caller-owned) that receives
 *                   each tensor's start in the flat vector; may be NULL
 * Returns ZERO_OK or ZERO_ERR_ARG (nothing written on error; also when the
 * padded total would exceed ZERO_MAX_ELEMS).  Host only. */
int zero_init_layout(const int64_t* tensor_numel, int64_t n_tensors, int32_t N,
                     zero_layout* out, int64_t* tensor_offsets);

/* Owner r's slice [*begin, *end) of the flat vector.  Host only.
 * Returns ZERO_OK or ZERO_ERR_ARG. */
int zero_shard_range(const zero_layout* layout, int32_t r, int64_t* begin, int64_t* end);

/* Bytes of device workspace a step needs, for the given size and
 * hyper-parameters.  in_place = 1 is for zero_step and 0 for zero_step_into.
 * The workspace holds:
 *   - a 256-byte control block;
 *   - per-CTA partial sums for the norm, shared by the step's launches;
 *   - when the step must see the whole gradient before it may update
 *     anything, an FP32 copy of the combined gradient (psi_pad * 4 bytes).
 *     This is needed with clipping, for an in-place step with
 *     skip_on_overflow, and (as the accumulator) with micro_batches >= 2;
 *   - from the next 256-byte boundary, rows of norm partials: 256 bytes,
 *     then 16 KiB a row.
 *     The size returned has one row per kernel launch of the step's first
 *     pass over the vector (a launch covers at most 2^22 elements of one
 *     hp->bucket_elems bucket), at most 2048.
 * A launch with a row of its own stores its CTAs' sums there; one without
 * adds them to the shared partials after the previous launch has finished,
 * which costs a little time.  So any size down to the part before the rows
 * works, with the rows that fit, and every size gives a result that is the
 * same on every run.  The norm's last bits may depend on how many rows there
 * are.
 * Returns 0 if the arguments are invalid. */
size_t zero_workspace_bytes(int64_t psi_pad, const zero_adam_hparams* hp, int32_t in_place);

/* One ZeRO update step, in place (RC-T2 note N48; DP-ZeRO blog "three stages").
 *   grads        host array of N device pointers.  grads[i] is rank i's
 *                gradient for the whole flat vector: psi_pad elements of
 *                grad_dtype, zero on the padding.  The step only reads them.
 *   grad_dtype   ZERO_GRAD_BF16 or ZERO_GRAD_FP32
 *   master, m, v device FP32 arrays of psi_pad elements, updated in place.
 *                Owner r's slice is [r*S, (r+1)*S).
 *   w_bf16       device array of psi_pad BF16 values (uint16 bit patterns):
 *                the full working-weight view that the all-gather fills
 *   psi_pad, N   sizes; psi_pad must be a multiple of N * ZERO_PAD_UNIT and at
 *                most ZERO_MAX_ELEMS
 *   hp           host pointer to the hyper-parameters
 *   loss_scale   > 0; the gradients hold loss_scale times the true gradient
 *   workspace    device buffer of zero_workspace_bytes(psi_pad, hp, 1) bytes
 *                (fewer work too, down to the part before the rows of norm
 *                partials: see zero_workspace_bytes), 256-byte aligned.  Its
 *                contents need no initialisation.  Calls that share one
 *                workspace must be ordered on one stream.
 *   result       device-accessible zero_step_result (device memory, or pinned
 *                host memory that the device can address), written when the
 *                step completes on `stream`; or NULL.  With NULL the call
 *                waits for the step and returns its status.
 *   stream       cudaStream_t to enqueue on (NULL = the legacy default stream)
 * All device buffers must be ZERO_ALIGN_BYTES-aligned.  None may overlap
 * another: the gradients, master, m, v, w_bf16 and the workspace are checked.
 * With hp->skip_on_overflow set and a non-finite combined gradient, master,
 * m, v and w_bf16 are left bit-for-bit unchanged and the status is
 * ZERO_STEP_SKIPPED.  The step counter and the loss scale are the caller's:
 * this library never changes them.
 * Returns ZERO_OK once the step is enqueued (result != NULL), the step's
 * status (result == NULL), or a negative error code. */
int zero_step(const void* const* grads, int32_t grad_dtype,
              float* master, float* m, float* v, uint16_t* w_bf16,
              int64_t psi_pad, int32_t N, const zero_adam_hparams* hp, float loss_scale,
              void* workspace, size_t workspace_bytes,
              zero_step_result* result, void* stream);

/* The same step, out of place.  It reads master/m/v from src_* and writes the
 * post-step master/m/v and BF16 weights to dst_*.  The caller swaps the two
 * buffer sets between steps.  With skip_on_overflow set, a skipped step
 * copies src to dst (src_w_bf16 to dst_w_bf16 included), so dst always holds
 * the valid post-step state.  Because the old state is never overwritten, the
 * overflow decision needs no second pass over the gradients.  A step with
 * skip_on_overflow and no clipping reads each gradient and state element once
 * and writes each output once.  src_w_bf16 is read only by a skipped step.
 * Other arguments and errors are as for zero_step.  Every dst buffer must be
 * disjoint from every src buffer, from the gradients and from the workspace.
 * The workspace needs zero_workspace_bytes(psi_pad, hp, 0) bytes. */
int zero_step_into(const void* const* grads, int32_t grad_dtype,
                   const float* src_master, const float* src_m, const float* src_v,
                   const uint16_t* src_w_bf16,
                   float* dst_master, float* dst_m, float* dst_v, uint16_t* dst_w_bf16,
                   int64_t psi_pad, int32_t N, const zero_adam_hparams* hp, float loss_scale,
                   void* workspace, size_t workspace_bytes,
                   zero_step_result* result, void* stream);

/* ------------------------------------------------------------------------
 * Bucketed form of the same step.
 *
 * The ledger page, section "one full ZeRO-3 computation", notes two things.
 * Real systems group gradients into buckets and synchronise the ready ones
 * while later layers are still running backward.  The DP-ZeRO blog, section
 * "offloading the shard to the CPU: two buffers", streams gradient chunks
 * through two device slots that alternate: while the kernel reads one, the
 * next chunk is copied into the other.  A plan lets a caller do
 * either.  It enqueues the reduce-scatter one bucket at a time, in flat order,
 * each bucket as soon as its gradients are ready.  A bucket's gradients may sit
 * anywhere, for example in one of two staging slots.  The owner update is
 * committed at the end, once the step-wide checks are known.
 *
 *   zero_plan_init    check and record every argument, as zero_step or
 *                     zero_step_into would (host only, nothing enqueued)
 *   zero_plan_begin   reset the step's control block in the workspace
 *   zero_plan_bucket  enqueue the first pass over [begin, end), the next bucket
 *   zero_plan_end     enqueue the step-wide decision and the commit, then
 *                     report the result as zero_step does
 * zero_step is zero_plan_init, zero_plan_begin, one zero_plan_bucket per
 * bucket and zero_plan_end.  All calls of one step go to one stream.
 * ------------------------------------------------------------------------ */
typedef struct {
    const void* grads[ZERO_MAX_RANKS]; /* rank i's gradient for the whole vector          */
    const float* src_master;
    const float* src_m;
    const float* src_v;
    const uint16_t* src_w_bf16;
    float* dst_master;                 /* == src_master for an in-place step              */
    float* dst_m;
    float* dst_v;
    uint16_t* dst_w_bf16;
    void* workspace;
    size_t workspace_bytes;
    float* grad_accum;                 /* the FP32 combined-gradient buffer of the two-pass
                                          form: NULL = inside the workspace; otherwise the
                                          caller's buffer (see zero_plan_init_ex)          */
    int64_t psi_pad;
    int64_t cursor;                    /* next element a bucket must start at             */
    zero_adam_hparams hp;
    float loss_scale;
    int32_t grad_dtype;
    int32_t N;
    int32_t in_place;
    int32_t two_pass;                  /* 1 if the update waits for a second pass          */
    int32_t state;                     /* 0 unset, 1 initialised, 2 begun                 */
    int32_t micro_batch;               /* micro-batch the next bucket belongs to          */
    int32_t policy_t_count;            /* device policy: size of the t window (0 = none)   */
    int64_t policy_t_first;            /* device policy: first t of the window            */
    void* policy;                      /* device policy (zero_plan_set_device_policy)     */
    int32_t overlap_buckets;           /* 0 (as zero_plan_init leaves it): every bucket
                                          launch waits for all work before it on the
                                          stream.  1: the caller promises to enqueue
                                          nothing on the stream (no kernel, copy or
                                          event wait) between this plan's
                                          zero_plan_bucket calls, so consecutive bucket
                                          launches may overlap (one starts while the
                                          previous drains), as zero_step runs them.
                                          The first bucket of each pass over the vector
                                          never overlaps.                                 */
    int32_t smem_staging;              /* how the one-pass kernel reads its inputs (steps
                                          without micro-batches, clip or in-place skip):
                                          ZERO_STAGING_REGISTERS (0, as zero_plan_init
                                          leaves it) or ZERO_STAGING_TMA.  Set it between
                                          zero_plan_init and the first zero_plan_bucket.  */
    void* current_set;                 /* ping-pong sets (zero_plan_set_pingpong): the
                                          device address of the caller's current-set
                                          word; NULL (as zero_plan_init leaves it) = off */
    int64_t rows_offset;               /* workspace offset of the rows of norm partials */
    int32_t row_capacity;              /* first-pass launches of a step that get a row of
                                          their own (0: the workspace holds no rows)      */
    int32_t rows_used;                 /* rows handed out in the current step             */
    int32_t row_width;                 /* slots of the latest row that count               */
    int32_t shared_slots_used;         /* 1 once a launch of the step had no row of its own */
    const float* policy_table;         /* device policy: the device address of the caller's
                                          table of bias corrections
                                          (zero_plan_set_device_policy_table); NULL (as
                                          zero_plan_init leaves it) = the window passed
                                          with the launch                                 */
} zero_plan;

/* Values of zero_plan.smem_staging.
 *   ZERO_STAGING_REGISTERS  every thread loads its 8-element groups from HBM
 *                           straight into registers, two groups in flight.
 *   ZERO_STAGING_TMA        one thread per CTA copies each tile of T elements
 *                           (the N gradient chunks and the master/m/v chunks)
 *                           into one of two shared-memory stages with TMA bulk
 *                           copies; T / 128 warps compute from shared memory.
 *                           T is 2048, or 1536 for N = 1, 2 or 4 with
 *                           N * g <= 13, where three CTAs then fit an SM.
 *                           Alternating the chunks between two slots, one
 *                           computed from while the other fills, is the DP-ZeRO
 *                           blog's two-buffer pattern.  Needs 2 * T * (N * g + 12)
 *                           bytes of shared memory per CTA, at most 200 KB (g = 2
 *                           for BF16 gradients, 4 for FP32: N <= 18 and N <= 9),
 *                           and the gradients and src master/m/v in device
 *                           memory (the copies read no pinned host or managed
 *                           memory); otherwise zero_plan_bucket returns
 *                           ZERO_ERR_ARG.  Every wait in the kernel gives up
 *                           after about a second: the step then ends with
 *                           status ZERO_ERR_TIMEOUT and is not applied (out of
 *                           place, dst is restored from src; in place, the
 *                           tiles not reached keep their state and the rest
 *                           are updated).
 *   ZERO_STAGING_TMA_TEST_STALL  as ZERO_STAGING_TMA, except that CTA 0 of every
 *                           launch never copies its first tile, so that waits
 *                           run out: for testing the timeout path only.
 * Both forms give the same results bit for bit. */
#define ZERO_STAGING_REGISTERS 0
#define ZERO_STAGING_TMA 1
#define ZERO_STAGING_TMA_TEST_STALL 2

/* Fills *plan from the arguments of zero_step (dst == src) or zero_step_into
 * (dst != src), after the same checks; returns their error codes.  grads is
 * copied, so the caller's array need not outlive the call.  A grads[i] may be
 * NULL if every bucket will pass its own gradient pointers. */
int zero_plan_init(zero_plan* plan, const void* const* grads, int32_t grad_dtype,
                   const float* src_master, const float* src_m, const float* src_v,
                   const uint16_t* src_w_bf16, float* dst_master, float* dst_m, float* dst_v,
                   uint16_t* dst_w_bf16, int64_t psi_pad, int32_t N,
                   const zero_adam_hparams* hp, float loss_scale, void* workspace,
                   size_t workspace_bytes);

/* Bytes of the workspace's control part: what the workspace needs when the
 * combined gradient is kept in a caller buffer (zero_plan_init_ex). */
#define ZERO_WORKSPACE_CONTROL_BYTES 16640

/* zero_plan_init with the owner's FP32 combined gradient (the reduced
 * gradient shard, or the accumulator with micro_batches >= 2) kept in
 * grad_accum.  That is a caller buffer of psi_pad floats, 16-byte aligned and
 * addressable by the device: device memory, or pinned host memory.  With
 * pinned host memory the gradient shard leaves the GPU altogether (DP-ZeRO
 * blog, "offloading the shard to the CPU: two buffers are enough").  The GPU
 * keeps only the buckets in flight, for instance in two staging slots, and
 * the kernels add each reduced bucket into the host shard over NVLink-C2C.
 * A non-NULL grad_accum forces the two-pass form, since the update reads the
 * gradient from there.  The workspace then needs only
 * ZERO_WORKSPACE_CONTROL_BYTES.  NULL behaves as zero_plan_init.  grad_accum
 * must not overlap any other buffer of the step. */
int zero_plan_init_ex(zero_plan* plan, const void* const* grads, int32_t grad_dtype,
                      const float* src_master, const float* src_m, const float* src_v,
                      const uint16_t* src_w_bf16, float* dst_master, float* dst_m, float* dst_v,
                      uint16_t* dst_w_bf16, int64_t psi_pad, int32_t N,
                      const zero_adam_hparams* hp, float loss_scale, void* workspace,
                      size_t workspace_bytes, float* grad_accum);

/* ------------------------------------------------------------------------
 * Device-resident step policy.  The host normally has to read each step's
 * outcome before it can issue the next step: a skipped step leaves t where it
 * was, and the dynamic loss scale reacts to overflow.  With a device policy
 * that bookkeeping stays on the GPU, so the host can issue steps back to back
 * without waiting for any of them.  (Not on the pages; the host-side policy
 * is the same rule.)
 * ------------------------------------------------------------------------ */
typedef struct {
    int64_t t;                 /* steps applied so far; the next applied step uses t + 1 */
    float loss_scale;          /* the scale the next step's gradients carry             */
    int32_t good_steps;        /* clean steps since the scale last changed              */
    int32_t growth_interval;   /* > 0: the scale grows after that many clean steps and
                                  backs off after an overflowing one; 0: static scale   */
    float backoff;             /* e.g. 0.5                                              */
    float growth;              /* e.g. 2.0                                              */
    int32_t last_status;       /* status of the latest step (as zero_step_result.status) */
} zero_device_policy;

#define ZERO_POLICY_WINDOW 16   /* most t values one step can be given */

/* Makes the plan's step take t and the loss scale from *policy instead of
 * hp->step and the loss_scale argument.  *policy is caller-owned and
 * device-addressable: device memory, or pinned host memory the host may read
 * at any time.  When the step ends, the device updates *policy:
 *   - t advances if the step applied;
 *   - with growth_interval > 0, an overflowing step multiplies the scale by
 *     backoff and restarts good_steps; otherwise good_steps counts up and, on
 *     reaching growth_interval, multiplies the scale by growth and restarts;
 *   - last_status is set.
 * The step uses t' = policy->t + 1 at its start.  The bias corrections depend
 * on t', and the host, which may not know t' yet, computes them for every t'
 * in [t_first, t_first + t_count), with 1 <= t_count <= ZERO_POLICY_WINDOW.
 * If t' falls outside that window the step changes nothing and ends with
 * status ZERO_ERR_POLICY_WINDOW.  Call between zero_plan_init(_ex) and
 * zero_plan_begin.  Returns ZERO_OK or ZERO_ERR_ARG. */
int zero_plan_set_device_policy(zero_plan* plan, zero_device_policy* policy, int64_t t_first,
                                int32_t t_count);

/* The bias corrections of a device policy for t = t_first .. t_first +
 * t_count - 1, two floats per t: table[2*i] = lr / (1 - beta1^t) and
 * table[2*i + 1] = sqrt(1 - beta2^t) for t = t_first + i, each rounded once
 * to FP32 from FP64, exactly as a step with hp->step = t rounds them.
 *   hp       host pointer to the hyper-parameters the steps will use (lr,
 *            beta1 and beta2 enter the table)
 *   table    host array of 2 * t_count floats, written on success
 * t_first >= 1, 1 <= t_count and t_first + t_count - 1 <= ZERO_MAX_ELEMS.
 * Returns ZERO_OK or ZERO_ERR_ARG (nothing written).  Host only. */
int zero_policy_table_fill(const zero_adam_hparams* hp, int64_t t_first, int64_t t_count,
                           float* table);

/* zero_plan_set_device_policy with the bias corrections read from a table
 * instead of a window passed with the launch.  table holds 2 * t_count
 * floats filled by zero_policy_table_fill(hp, t_first, t_count, ...) with the
 * plan's lr and betas; it is caller-owned, device-addressable (device memory,
 * or pinned host memory), 8-byte aligned, and must stay unchanged while
 * steps that read it are in flight; 1 <= t_count.  The step reads the entry of
 * t' = policy->t + 1; a t' outside [t_first, t_first + t_count) ends the step
 * with ZERO_ERR_POLICY_WINDOW and changes nothing, as with a window.
 * The launches then carry no value that depends on t, so a step captured in
 * a CUDA graph (its gradients, state sets and policy at fixed addresses) can
 * be replayed once per step for every t the table covers, with t, the loss
 * scale and, with ping-pong sets, the current set all kept on the device.
 * Call between zero_plan_init(_ex) and zero_plan_begin.  Returns ZERO_OK or
 * ZERO_ERR_ARG. */
int zero_plan_set_device_policy_table(zero_plan* plan, zero_device_policy* policy,
                                      const float* table, int64_t t_first, int32_t t_count);

/* ------------------------------------------------------------------------
 * Ping-pong state sets.  An out-of-place step reads one full set of
 * master/m/v/w and writes the other.  Normally the caller swaps the two sets
 * after every step, and a skipped step must therefore copy the old state into
 * the other set (28 bytes per parameter), because the caller will read it
 * from there.  With ping-pong sets the device keeps, in one int32 word, which
 * set is current.  A step reads the current set and writes the other; when
 * the step applies, the device flips the word; when it is skipped (overflow,
 * a t outside the device policy's window, a timed-out wait) the word and the
 * current set stay as they were and nothing is copied.  The skip costs no
 * more than the pass that found the overflow.  (Not on the pages; a skipped
 * step is this library's reading of overflow handling.)
 * ------------------------------------------------------------------------ */

/* Makes the plan's step use ping-pong sets.  Set 0 is the plan's src_* buffers
 * and set 1 its dst_* buffers; both are read and written, so the plan must be
 * out of place with src_w_bf16 given, and no buffer of either set may overlap
 * another buffer of the step.  *current_set is a caller-owned int32 (0 or 1;
 * any non-zero value counts as 1), 4-byte aligned and device-addressable:
 * device memory, or pinned host memory the host may read once the step has
 * completed.  The step reads it once at its start (in zero_plan_begin's
 * prologue) and, if the step applies, stores the other set's index into it
 * when the step ends.  The caller finds the post-step state, and so the
 * current BF16 working-weight view, in the set it names.  Call between
 * zero_plan_init(_ex) and zero_plan_begin.  With ZERO_STAGING_TMA both sets'
 * master/m/v must be in device memory (zero_plan_bucket returns ZERO_ERR_ARG
 * otherwise).  Steps that share a word must be ordered (one stream, or
 * events), since each reads it at its start and may write it at its end; the
 * host must not write the word while such a step is in flight.  Returns
 * ZERO_OK, ZERO_ERR_ARG or ZERO_ERR_OVERLAP. */
int zero_plan_set_pingpong(zero_plan* plan, int32_t* current_set);

/* Starts the step: clears the control block on `stream`.  With a device
 * policy or ping-pong sets it also launches the step's one-thread prologue
 * kernel, which reads them. */
int zero_plan_begin(zero_plan* plan, void* stream);

/* Gradient accumulation (hp->micro_batches = k >= 2; the DP-ZeRO blog,
 * "stacking with other parallelism": under pipeline parallelism gradients
 * arrive micro-batch by micro-batch, so they are reduced chunk by chunk as they
 * go).  The plan then takes k passes of buckets over [0, psi_pad), one per
 * micro-batch, each with that micro-batch's gradients.  Each bucket adds its
 * combined gradient, scaled by fp32(1 / (N * k * loss_scale)), to the owner's
 * FP32 accumulator in the workspace, in micro-batch order, from +0.  The
 * overflow check, the norm, the clip and the update use the accumulated
 * gradient.  When the step needs no second pass (no clip, and no skip of an
 * in-place step) and the accumulator is the workspace's, the last
 * micro-batch's buckets add their part to the accumulator and apply the
 * update in the same pass, leaving the accumulator as the earlier
 * micro-batches left it; the roundings are the same.  zero_step and
 * zero_step_into take one batch only and reject k >= 2.
 *
 * First pass over elements [begin, end) of the flat vector.  begin must equal
 * plan->cursor (buckets arrive in flat order, without gaps).  end is a multiple
 * of ZERO_BUCKET_ALIGN or psi_pad, and begin < end <= psi_pad.
 *   bucket_grads  NULL to read plan->grads[i] + begin; otherwise a host array of
 *                 N device pointers.  bucket_grads[i] points at rank i's
 *                 contribution to element `begin`, and the next end - begin
 *                 elements follow it: a staging slot, say.  Each must be
 *                 ZERO_ALIGN_BYTES-aligned and must not overlap a written buffer.
 * The bucket's gradients are read by the time the stream passes this call, so
 * the buffer may be refilled after an event recorded right after it. */
int zero_plan_bucket(zero_plan* plan, int64_t begin, int64_t end,
                     const void* const* bucket_grads, void* stream);

/* Ends the step once every element has been covered (plan->cursor ==
 * psi_pad), by every micro-batch when accumulating.  It enqueues the step-wide decision and then the commit: the
 * second pass, or the copy of a skipped out-of-place step.  result and the
 * return value are as for zero_step. */
int zero_plan_end(zero_plan* plan, zero_step_result* result, void* stream);

/* ------------------------------------------------------------------------
 * ZeRO-3: per-layer gather of the working weights.
 *
 * Under ZeRO-3 each rank keeps only its 1/N shard of the BF16 working weights.
 * Before a layer runs, its full view is all-gathered into temporary memory and
 * released once the layer has run (RC-T2 slide b2 and note N47; ledger page,
 * "one full ZeRO-3 computation").  Here the N shards are the owners' slices
 * of the flat vector.  A step's all-gather writes them: shard r is
 * w_bf16 + r*S.  They may equally be N separate buffers.
 * ------------------------------------------------------------------------ */

/* Flags of zero3_gather.
 *   ZERO3_GATHER_OVERLAP_PREVIOUS  the gather may start copying while the
 *       kernel enqueued right before it on `stream` drains, without waiting
 *       for it to complete.  Since that kernel may be a gather launched with
 *       this flag too, which did not wait for its own predecessor either, the
 *       kernels that may still be running form a chain back to the last
 *       kernel launched without the flag.  The caller promises that none of
 *       them writes the shards or reads or writes `view`, except those that
 *       an event wait enqueued on `stream` before this gather already orders
 *       before it.  Waits on events stay complete dependencies.  Example: the
 *       gathers of consecutive layers alternating between two views, each
 *       view refilled only after an event wait for the use of its previous
 *       layer (the two-view schedule below).  Without the flag the gather
 *       begins only after everything before it on the stream has completed. */
#define ZERO3_GATHER_OVERLAP_PREVIOUS 1u

/* Copies elements [begin, end) of the full flat view into `view`.  Element j
 * is read from shards[j / shard] at offset j % shard.
 *   shards   host array of N device pointers, each ZERO_ALIGN_BYTES-aligned,
 *            holding `shard` BF16 values
 *   shard    elements per shard, a multiple of ZERO_BUCKET_ALIGN, with N * shard
 *            at most ZERO_MAX_ELEMS (every layout from zero_init_layout
 *            qualifies)
 *   view     device buffer of end - begin BF16 values, ZERO_ALIGN_BYTES-aligned;
 *            it must not overlap a shard
 *   flags    0 or ZERO3_GATHER_OVERLAP_PREVIOUS
 * Any 0 <= begin <= end <= N * shard is accepted.  A begin that is a multiple
 * of ZERO_BUCKET_ALIGN takes a 16-byte vector path; any other begin takes an
 * element-by-element path.  Enqueued on `stream`.  Returns ZERO_OK, or
 * ZERO_ERR_ARG / ZERO_ERR_ALIGN / ZERO_ERR_OVERLAP / ZERO_ERR_CUDA before
 * anything is enqueued. */
int zero3_gather(const uint16_t* const* shards, int32_t N, int64_t shard, int64_t begin,
                 int64_t end, uint16_t* view, uint32_t flags, void* stream);

/* Peak bytes one rank holds under ZeRO-3 when the layers, of layer_numel[i]
 * elements in run order, are gathered one ahead into two BF16 views (one in
 * use, one being prefetched) and each view is released after its layer ran.
 * That is the persistent ZeRO-3 subtotal (zero_ledger(psi, N, 3, ...)) plus 2 B
 * times the largest sum of two neighbouring layers.  The pages stress that the
 * persistent subtotal (32 GB for 8e9 parameters on 4 ranks) is not the peak.
 * Activations and communication buffers are left out, as in the ledger.
 * Host only.  Returns -1 on a bad argument. */
int64_t zero3_peak_bytes(const int64_t* layer_numel, int64_t n_layers, int32_t N,
                         int32_t grad_bytes, int32_t optim_bytes);

/* Persistent bytes one rank holds under a ZeRO stage: 0 = replicated data
 * parallelism, 1 = optimizer state sharded, 2 = also gradients, 3 = also the
 * working weights.  A replicated part counts psi elements.  A sharded part
 * counts ceil(psi / N) elements.  The BF16 working weight is 2 B per
 * parameter, the gradient grad_bytes (2 or 4) and the optimizer state
 * optim_bytes (12 for Adam's FP32 master/m/v, 8 with a first moment only).
 * With grad_bytes = 2 and optim_bytes = 12 this gives 16, 4+12/N, 2+14/N and
 * 16/N bytes per parameter.  See the DP-ZeRO blog's stage table, and RC-T2
 * note N47: 128/56/44/32 GB for 8e9 parameters on 4 ranks.  GB there means
 * 1e9 bytes, counting persistent state only.  Host only.
 * Returns -1 on a bad argument (psi outside 0 .. ZERO_MAX_ELEMS, N < 1, a byte
 * width outside 0 .. 64). */
int64_t zero_ledger(int64_t psi, int32_t N, int32_t stage, int32_t grad_bytes,
                    int32_t optim_bytes);

/* Elements each rank sends per step under a stage, counted as the DP-ZeRO
 * blog's stage table counts them.  Stages 0-2 send 2*psi: one reduce-scatter
 * and one all-gather, i.e. one all-reduce.  Stage 3 sends 3*psi: one more
 * all-gather.  The ledger page warns that this multiple depends on the
 * counting convention.  Host only.  Returns -1 on a bad argument. */
int64_t zero_comm_volume(int64_t psi, int32_t N, int32_t stage);

/* Static text for a zero_status value. */
const char* zero_status_str(int status);

/* Number of kernels this library has launched in this process.  Host only,
 * monotonic, thread-safe.  Memsets and copies are not counted. */
uint64_t zero_launch_count(void);

/* Debug build.  The same sources compiled with -DZERO_DEBUG give
 * libzero_gb300_debug.so, with the same entry points.  There every kernel
 * checks each index range it is about to touch against the lengths of the
 * buffers involved (the state arrays, the gradient buffers or staging slots,
 * the workspace, the shards and the view of a gather).  An access outside
 * them is not made: the kernel skips it and counts it, and a step that saw one
 * ends with status ZERO_ERR_BOUNDS and is not applied: t does not advance, out
 * of place dst is restored from src (with ping-pong sets the current set stays
 * current), and in place the elements reached before may already be updated.
 * No check traps or asserts, so the device stays usable.
 * Returns the number of skipped out-of-range accesses counted on the current
 * device since the previous call, and resets the count; -1 in the release
 * build, which has no checks.  Host only; waits for the device. */
int64_t zero_debug_bounds_violations(void);

/* ------------------------------------------------------------------------
 * zero_step without a caller-provided workspace.  The pages have no
 * counterpart to this entry point: it exists for callers that cannot
 * allocate device memory themselves.  Examples: a host program whose device
 * memory is owned by another allocator or memory pool, a plugin inside a
 * framework that hands it only the tensors it works on, or a control loop
 * where an allocation's implicit device synchronisation is not acceptable.
 *
 * It is the in-place zero_step, with the same arguments, checks, arithmetic
 * and results.  The workspace is a fixed array of ZERO_NOALLOC_SCRATCH_BYTES
 * in device memory, defined inside this library.  Every GPU that loads the
 * library holds that array until the process exits.  The one-pass form (no
 * clipping, no skip_on_overflow) fits at any size.  The two-pass form (with
 * clipping or skip_on_overflow) also keeps the FP32 combined gradient there,
 * so it accepts psi_pad up to ZERO_NOALLOC_MAX_TWO_PASS_ELEMS.  Larger
 * requests return ZERO_ERR_TOO_LARGE before anything is enqueued.
 *
 * The first call on a device looks up the array's device address, with that
 * device current, and keeps it for later calls.  Make that first call before
 * any stream capture.  The call allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine.  It clears, on `stream`, the part
 * of the array each step must start from zero.
 *
 * All calls on a device share the one array, which keeps the last step's
 * contents.  Two calls whose work overlaps on the GPU race on it: from
 * different streams or host threads, order them (one stream, or events)
 * yourself.  Returns as zero_step does, or ZERO_ERR_TOO_LARGE.  zero_step's
 * argument and alignment checks come first: a call they reject gets their
 * ZERO_ERR_ARG or ZERO_ERR_ALIGN whatever its size.  ZERO_ERR_OVERLAP is
 * checked after the size. */
#define ZERO_NOALLOC_MAX_TWO_PASS_ELEMS 4194304
#define ZERO_NOALLOC_SCRATCH_BYTES (16640 + 4 * ZERO_NOALLOC_MAX_TWO_PASS_ELEMS)
int zero_step_noalloc(const void* const* grads, int32_t grad_dtype,
                      float* master, float* m, float* v, uint16_t* w_bf16,
                      int64_t psi_pad, int32_t N, const zero_adam_hparams* hp, float loss_scale,
                      zero_step_result* result, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ZERO_GB300_H */
