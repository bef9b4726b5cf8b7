/*
 * zero_oracle.c -- the CPU oracle for the ZeRO sharded mixed-precision update
 * step.  TEST INFRASTRUCTURE ONLY: only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it.  The product path never does.
 *
 * Plain, slow, obviously correct C.  One element at a time, FP32 operators
 * rounded one by one (build with -ffp-contract=off, no fast-math), FP64 only
 * where a step-wide scalar is formed.  It shares no code, header or constant
 * with the CUDA path.
 *
 * Citation key (the three pages this follows):
 *   [RC-T2]   lecture deck "RC-T2: sharing data and sharing the duty to store
 *             are two different acts" (codingai-lec06.pages.dev/pages/RC-T2.html),
 *             slides b0-b3 and deep-dive notes N46, N47, N48.
 *   [LEDGER]  topic page "Putting the training ledger onto multiple devices"
 *             (codingai-lec06.pages.dev/topics/distributed-training.html),
 *             sections "start from persistent state", "dividing data vs
 *             dividing storage", "one full ZeRO-3 computation".
 *   [DPZERO]  blog post "Data parallelism and ZeRO: how much each of the three
 *             stages saves" (blog.javazero.top/2026/09/05/llm-dp-zero/),
 *             sections "16 bytes per parameter", "three stages" (with its
 *             stage table), "offloading the shard to the CPU: two buffers".
 *
 * Readings taken where the pages are silent (each is also listed with the
 * design notes):
 *   - Adam is the standard bias-corrected Adam; weight decay, when non-zero,
 *     is decoupled (AdamW) and applied to the master weight before the
 *     moment update.  The pages only name "two Adam history statistics".
 *   - The batch-mean scaling is one multiply by fp32(1/(N * loss_scale))
 *     after the FP32 sum of the N contributions taken in rank order 0..N-1,
 *     starting from +0.
 *   - Overflow is detected on that scaled FP32 gradient; a skipped step
 *     leaves every state word and every output weight bit-unchanged.
 *   - The global-norm clip uses coef = min(1, max_norm / (norm + 1e-6)) on the
 *     batch-mean gradient, with the norm summed sequentially in FP64.
 *   - BF16 is round-to-nearest-even on the FP32 bit pattern; a NaN becomes
 *     the quiet NaN 0x7FC0.
 *   - The flat vector is padded with zeros to a multiple of N*128 elements
 *     and owner r holds the contiguous slice [r*S, (r+1)*S), S = psi_pad/N.
 *
 * All-cores timing mode.  Built with -fopenmp, the elementwise loops of the
 * whole-vector step run on all host cores; every element is computed exactly
 * as in the single-thread build.  The step-wide sum of squares is then formed
 * as one FP64 partial per contiguous chunk of the vector (one chunk per
 * thread), each summed in element order, and the partials are added in chunk
 * order: a fixed order for a given thread count.  With one chunk (the
 * single-thread build) it is the sequential sum.  Only the benchmark's CPU
 * baseline uses that build; every pin and parity check uses the plain one.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_BF16 0
#define ORC_FP32 1
#define ORC_PAD_UNIT 128

/* ------------------------------------------------------------------------ */
/* BF16 <-> FP32                                                             */
/* ------------------------------------------------------------------------ */

/* BF16 is the top half of an FP32 word, so widening is exact. */
float orc_bf16_to_f32(uint16_t h)
{
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

/* Round-to-nearest-even of an FP32 value to BF16.  The kept half is the top
 * 16 bits; the dropped half decides: above one half rounds up, below rounds
 * down, exactly one half rounds to the even kept value.  Rounding up past the
 * largest finite BF16 lands on infinity, as IEEE rounding does. */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    uint32_t exponent = (bits >> 23) & 0xffu;
    uint32_t mantissa = bits & 0x7fffffu;
    if (exponent == 0xffu && mantissa != 0u)
        return (uint16_t)0x7fc0u; /* NaN -> quiet NaN */
    uint32_t kept = bits >> 16;
    uint32_t dropped = bits & 0xffffu;
    if (dropped > 0x8000u)
        kept += 1u;
    else if (dropped == 0x8000u && (kept & 1u) != 0u)
        kept += 1u;
    return (uint16_t)kept;
}

void orc_f32_to_bf16_array(const float* in, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_f32_to_bf16(in[i]);
}

/* ------------------------------------------------------------------------ */
/* Flat layout: concatenation, padding and shard slices                      */
/* [RC-T2 b1, N47]: each of the N cards keeps one quarter (1/N) of the state;  */
/* [DPZERO "three stages"]: each card holds 1/N and updates only its piece.   */
/* ------------------------------------------------------------------------ */

/* Returns 0 on success, -1 on a bad argument.  offsets[i] is where tensor i
 * starts in the flat vector; psi is the sum of the sizes; psi_pad rounds psi
 * up to a multiple of N*128; shard = psi_pad / N. */
int orc_layout(const int64_t* numel, int64_t n_tensors, int32_t N,
               int64_t* offsets, int64_t* psi, int64_t* psi_pad, int64_t* shard)
{
    if (N < 1 || n_tensors < 0)
        return -1;
    int64_t total = 0;
    for (int64_t i = 0; i < n_tensors; ++i) {
        if (numel[i] < 0)
            return -1;
        if (offsets)
            offsets[i] = total;
        total += numel[i];
    }
    int64_t unit = (int64_t)N * ORC_PAD_UNIT;
    int64_t units = total / unit;
    if (units * unit < total)
        units += 1;
    *psi = total;
    *psi_pad = units * unit;
    *shard = *psi_pad / N;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Memory ledger and communication volume                                     */
/* [DPZERO "16 bytes per parameter"]: 2 (BF16 weight) + 2 (BF16 grad) +       */
/* 4+4+4 (FP32 master, m, v) = 16 B; FP32 grads add 2 B; a first-moment-only  */
/* optimizer keeps 8 B of optimizer state.  [DPZERO stage table]: DDP 16,     */
/* ZeRO-1 4+12/N, ZeRO-2 2+14/N, ZeRO-3 16/N bytes per parameter.             */
/* [LEDGER "start from persistent state"]: GB = 1e9 bytes, persistent state   */
/* only (no activations, temporaries, buffers or runtime).                    */
/* ------------------------------------------------------------------------ */

static int64_t orc_ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* Persistent bytes held by one rank.  stage 0 is replicated data parallelism;
 * stage 1 shards the optimizer state; stage 2 also the gradient; stage 3
 * also the working weight.  A sharded part of psi elements holds
 * ceil(psi/N) of them per rank.  Returns -1 on a bad argument. */
int64_t orc_ledger_bytes(int64_t psi, int32_t N, int32_t stage,
                         int32_t grad_bytes, int32_t optim_bytes)
{
    const int64_t weight_bytes = 2; /* BF16 working weight */
    if (psi < 0 || N < 1 || grad_bytes < 0 || optim_bytes < 0)
        return -1;
    int64_t sharded = orc_ceil_div(psi, N);
    switch (stage) {
    case 0:
        return (weight_bytes + grad_bytes + optim_bytes) * psi;
    case 1:
        return (weight_bytes + grad_bytes) * psi + optim_bytes * sharded;
    case 2:
        return weight_bytes * psi + (grad_bytes + optim_bytes) * sharded;
    case 3:
        return (weight_bytes + grad_bytes + optim_bytes) * sharded;
    default:
        return -1;
    }
}

/* Elements one rank sends per step.  With ring_exact == 0 this is the
 * pages' count ([DPZERO stage table]): 2*psi for DDP, ZeRO-1 and ZeRO-2
 * (one reduce-scatter plus one all-gather, i.e. one all-reduce) and 3*psi for
 * ZeRO-3 (one more all-gather of the weights).  The ledger page warns that
 * this multiple depends on the counting convention
 * ([LEDGER "one full ZeRO-3 computation"]); ring_exact == 1 gives the count
 * for a ring schedule, where a reduce-scatter or an all-gather has each rank
 * send (N-1) chunks of ceil(psi/N) elements. */
int64_t orc_comm_volume(int64_t psi, int32_t N, int32_t stage, int32_t ring_exact)
{
    if (psi < 0 || N < 1 || stage < 0 || stage > 3)
        return -1;
    int64_t passes = (stage == 3) ? 3 : 2;
    if (!ring_exact)
        return passes * psi;
    return passes * (int64_t)(N - 1) * orc_ceil_div(psi, N);
}

/* ------------------------------------------------------------------------ */
/* ZeRO-3: the working weights persist only as each rank's BF16 shard.  Before */
/* a layer runs, its full view is all-gathered into temporary memory and     */
/* released after use ([RC-T2 b2, N47]; [LEDGER "one full ZeRO-3              */
/* computation"]).                                                           */
/* ------------------------------------------------------------------------ */

/* Elements [begin, end) of the full flat view, gathered from the N ranks'
 * shards of `shard` elements each: element j lives in shard j / shard at
 * offset j % shard. */
int orc_gather_range(const uint16_t* const* shards, int32_t N, int64_t shard, int64_t begin,
                     int64_t end, uint16_t* out)
{
    if (N < 1 || shard < 0 || begin < 0 || end < begin || end > (int64_t)N * shard)
        return -1;
    for (int64_t j = begin; j < end; ++j)
        out[j - begin] = shards[j / shard][j % shard];
    return 0;
}

/* Peak bytes one rank holds under ZeRO-3 when the layers (in run order,
 * layer_numel[i] elements each) are gathered one ahead into two temporary
 * BF16 views -- the current layer's, and the next layer's being gathered
 * ([DPZERO "offloading the shard to the CPU: two buffers"]) -- and each view
 * is released after its layer ran: the persistent ZeRO-3 subtotal plus the
 * largest pair of neighbouring layers alive together.  The pages stress that
 * the persistent subtotal is not the peak ([RC-T2 b2, N47]); activations and
 * communication buffers are left out, as in the ledger. */
int64_t orc_zero3_peak_bytes(const int64_t* layer_numel, int64_t n_layers, int32_t N,
                             int32_t grad_bytes, int32_t optim_bytes)
{
    if (n_layers < 0 || N < 1)
        return -1;
    int64_t psi = 0, live = 0;
    for (int64_t i = 0; i < n_layers; ++i) {
        if (layer_numel[i] < 0)
            return -1;
        psi += layer_numel[i];
        int64_t pair = layer_numel[i] + (i + 1 < n_layers ? layer_numel[i + 1] : 0);
        if (pair > live)
            live = pair;
    }
    int64_t persistent = orc_ledger_bytes(psi, N, 3, grad_bytes, optim_bytes);
    if (persistent < 0)
        return -1;
    return persistent + 2 * live;
}

/* ------------------------------------------------------------------------ */
/* Step-wide scalars                                                          */
/* ------------------------------------------------------------------------ */

typedef struct {
    double lr, beta1, beta2, eps, weight_decay, max_grad_norm;
} orc_hparams;

typedef struct {
    float inv;        /* fp32(1 / (N * loss_scale)): batch mean and unscale */
    float b1, omb1;   /* beta1 and 1 - beta1                                */
    float b2, omb2;   /* beta2 and 1 - beta2                                */
    float eps;
    float step_size;  /* lr / (1 - beta1^t)                                 */
    float sbc2;       /* sqrt(1 - beta2^t)                                  */
    float decay;      /* 1 - lr * weight_decay                              */
    int32_t use_decay;
} orc_scalars;

/* Each scalar is formed in FP64 from the FP64 hyper-parameters and rounded
 * once to FP32.  t is the 1-based count of applied steps including this one. */
void orc_step_scalars(const orc_hparams* hp, int64_t t, int32_t N,
                      double loss_scale, orc_scalars* s)
{
    s->inv = (float)(1.0 / ((double)N * loss_scale));
    s->b1 = (float)hp->beta1;
    s->omb1 = (float)(1.0 - hp->beta1);
    s->b2 = (float)hp->beta2;
    s->omb2 = (float)(1.0 - hp->beta2);
    s->eps = (float)hp->eps;
    double bc1 = 1.0 - pow(hp->beta1, (double)t);
    double bc2 = 1.0 - pow(hp->beta2, (double)t);
    s->step_size = (float)(hp->lr / bc1);
    s->sbc2 = (float)sqrt(bc2);
    s->decay = (float)(1.0 - hp->lr * hp->weight_decay);
    s->use_decay = hp->weight_decay != 0.0;
}

/* ------------------------------------------------------------------------ */
/* Per-element pieces                                                         */
/* ------------------------------------------------------------------------ */

static float orc_load_grad(const void* buf, int32_t dtype, int64_t idx)
{
    if (dtype == ORC_BF16)
        return orc_bf16_to_f32(((const uint16_t*)buf)[idx]);
    return ((const float*)buf)[idx];
}

/* The combined gradient of one parameter: the N ranks' contributions to
 * this same element, added in rank order and scaled to the batch mean.
 * [RC-T2 N48]: the reduction adds contributions of the same parameter only,
 * and a batch-mean loss needs a matching scale at the reduction. */
static float orc_reduce_element(const void* const* grads, int32_t dtype,
                                int32_t N, int64_t idx, float inv)
{
    float a = 0.0f;
    for (int32_t i = 0; i < N; ++i)
        a = a + orc_load_grad(grads[i], dtype, idx);
    return a * inv;
}

static int orc_is_finite(float x)
{
    uint32_t bits;
    memcpy(&bits, &x, sizeof bits);
    return ((bits >> 23) & 0xffu) != 0xffu;
}

/* One mixed-precision Adam update of one element by its owner, with the
 * owner's own FP32 master weight and moments ([RC-T2 N48]; roles of the
 * states: [LEDGER "start from persistent state"]). */
static void orc_adam_element(float g, float* p, float* m, float* v,
                             const orc_scalars* s)
{
    float pp = *p, mm = *m, vv = *v;
    if (s->use_decay)
        pp = pp * s->decay;
    mm = s->b1 * mm + s->omb1 * g;
    vv = s->b2 * vv + s->omb2 * (g * g);
    float den = sqrtf(vv) / s->sbc2 + s->eps;
    pp = pp - s->step_size * (mm / den);
    *p = pp;
    *m = mm;
    *v = vv;
}

/* clip coefficient from the global norm: min(1, max_norm/(norm + 1e-6)),
 * compared in FP64 and rounded once.  A NaN norm compares false and gives 1. */
static float orc_clip_coef(double max_norm, double norm)
{
    double c = max_norm / (norm + 1e-6);
    return (c < 1.0) ? (float)c : 1.0f;
}

/* ------------------------------------------------------------------------ */
/* Collectives, as data semantics ([LEDGER "one full ZeRO-3 computation"]):   */
/* all-gather assembles the shards into a full view at every participant;    */
/* reduce-scatter combines contributions element by element and hands each  */
/* participant its slice; all-reduce gives everyone the full combined result. */
/* ------------------------------------------------------------------------ */

/* Owner r's slice of the combined, batch-mean gradient. */
void orc_reduce_scatter(const void* const* grads, int32_t dtype, int32_t N,
                        int64_t psi_pad, int32_t r, float inv, float* out_shard)
{
    int64_t shard = psi_pad / N;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < shard; ++j)
        out_shard[j] = orc_reduce_element(grads, dtype, N, (int64_t)r * shard + j, inv);
}

/* The full combined, batch-mean gradient, as every participant sees it. */
void orc_all_reduce(const void* const* grads, int32_t dtype, int32_t N,
                    int64_t psi_pad, float inv, float* out_full)
{
    for (int64_t j = 0; j < psi_pad; ++j)
        out_full[j] = orc_reduce_element(grads, dtype, N, j, inv);
}

/* Assemble N FP32 shards of `shard` elements into one full view. */
void orc_all_gather_f32(const float* const* shards, int32_t N, int64_t shard,
                        float* out_full)
{
    for (int32_t r = 0; r < N; ++r)
        for (int64_t j = 0; j < shard; ++j)
            out_full[(int64_t)r * shard + j] = shards[r][j];
}

/* ------------------------------------------------------------------------ */
/* The whole step                                                             */
/* ------------------------------------------------------------------------ */

/* Step-wide overflow flag and sum of squares of g[0..n): one FP64 partial per
 * contiguous chunk, each summed in element order, added in chunk order.  The
 * single-thread build has one chunk, i.e. the plain sequential sum. */
static void orc_check_vector(const float* g, int64_t n, int32_t* bad, double* sumsq)
{
    int chunks = 1;
#ifdef _OPENMP
    chunks = omp_get_max_threads();
    if (chunks < 1)
        chunks = 1;
#endif
    double partial[256];
    int32_t flag[256];
    if (chunks > 256)
        chunks = 256;
#pragma omp parallel for schedule(static, 1) num_threads(chunks)
    for (int c = 0; c < chunks; ++c) {
        int64_t lo = n * c / chunks, hi = n * (c + 1) / chunks;
        double s = 0.0;
        int32_t b = 0;
        for (int64_t j = lo; j < hi; ++j) {
            if (!orc_is_finite(g[j]))
                b = 1;
            s = s + (double)g[j] * (double)g[j];
        }
        partial[c] = s;
        flag[c] = b;
    }
    double total = 0.0;
    int32_t any = 0;
    for (int c = 0; c < chunks; ++c) {
        total = total + partial[c];
        any = any | flag[c];
    }
    *bad = any;
    *sumsq = total;
}

typedef struct {
    int32_t applied;          /* 1 = state updated, 0 = skipped            */
    int32_t found_nonfinite;  /* any non-finite combined gradient element  */
    double sumsq;             /* sum of squares of the combined gradient   */
    float grad_norm;          /* sqrt(sumsq), rounded to FP32              */
    float clip_coef;          /* 1 when clipping is off                    */
} orc_result;

/* ZeRO form ([DPZERO "three stages"], ZeRO-1/2; [RC-T2 N48]; [LEDGER "one full
 * ZeRO-3 computation"]).  Every owner r = 0..N-1 receives its slice of the
 * combined gradient by reduce-scatter, the step-wide checks run over all
 * owners' slices, each owner updates its own slice of master/m/v, and the
 * owners' BF16 slices are all-gathered into the one full working-weight view
 * w.  master, m, v and w are flat arrays of psi_pad elements in which owner r
 * holds [r*S, (r+1)*S).  Returns 0, or -1 on a bad argument or no memory. */
int orc_zero_step(const void* const* grads, int32_t dtype, int32_t N, int64_t psi_pad,
                  float* master, float* m, float* v, uint16_t* w,
                  const orc_hparams* hp, int64_t t, double loss_scale,
                  int32_t skip_on_overflow, orc_result* res)
{
    if (N < 1 || psi_pad < 0 || psi_pad % ((int64_t)N * ORC_PAD_UNIT) != 0)
        return -1;
    int64_t shard = psi_pad / N;
    orc_scalars s;
    orc_step_scalars(hp, t, N, loss_scale, &s);

    float* g = (float*)malloc((size_t)(psi_pad > 0 ? psi_pad : 1) * sizeof(float));
    if (!g)
        return -1;
    /* reduce-scatter into each owner's slice */
    for (int32_t r = 0; r < N; ++r)
        orc_reduce_scatter(grads, dtype, N, psi_pad, r, s.inv, g + (int64_t)r * shard);

    /* step-wide overflow check and sum of squares, over every owner's slice */
    int32_t bad = 0;
    double sumsq = 0.0;
    orc_check_vector(g, psi_pad, &bad, &sumsq);
    res->found_nonfinite = bad;
    res->sumsq = sumsq;
    res->grad_norm = (float)sqrt(sumsq);
    res->clip_coef = 1.0f;
    if (skip_on_overflow && bad) {
        res->applied = 0;
        free(g);
        return 0;
    }
    if (hp->max_grad_norm > 0.0) {
        res->clip_coef = orc_clip_coef(hp->max_grad_norm, sqrt(sumsq));
#pragma omp parallel for schedule(static)
        for (int64_t j = 0; j < psi_pad; ++j)
            g[j] = g[j] * res->clip_coef;
    }
    /* each owner updates its own slice */
    for (int32_t r = 0; r < N; ++r) {
        int64_t lo = (int64_t)r * shard, hi = (int64_t)(r + 1) * shard;
#pragma omp parallel for schedule(static)
        for (int64_t j = lo; j < hi; ++j)
            orc_adam_element(g[j], &master[j], &m[j], &v[j], &s);
    }
    /* all-gather of the owners' BF16 slices into the full view */
    for (int32_t r = 0; r < N; ++r) {
#pragma omp parallel for schedule(static)
        for (int64_t j = 0; j < shard; ++j)
            w[(int64_t)r * shard + j] = orc_f32_to_bf16(master[(int64_t)r * shard + j]);
    }
    res->applied = 1;
    free(g);
    return 0;
}

/* Replicated (DDP) form ([LEDGER "dividing data vs dividing storage"];
 * [RC-T2 N46]): each of the N replicas receives the full combined gradient by
 * all-reduce and updates its own full copy of master/m/v and w.  The
 * replicas' arrays are passed as N pointers each.  A ZeRO step must end in
 * exactly this state ([RC-T2 N48]: all ranks still train one model). */
int orc_ddp_step(const void* const* grads, int32_t dtype, int32_t N, int64_t psi_pad,
                 float* const* master, float* const* m, float* const* v,
                 uint16_t* const* w, const orc_hparams* hp, int64_t t,
                 double loss_scale, int32_t skip_on_overflow, orc_result* res)
{
    if (N < 1 || psi_pad < 0 || psi_pad % ((int64_t)N * ORC_PAD_UNIT) != 0)
        return -1;
    orc_scalars s;
    orc_step_scalars(hp, t, N, loss_scale, &s);
    float* g = (float*)malloc((size_t)(psi_pad > 0 ? psi_pad : 1) * sizeof(float));
    if (!g)
        return -1;
    for (int32_t i = 0; i < N; ++i) {
        /* every replica computes the same all-reduce result for itself */
        orc_all_reduce(grads, dtype, N, psi_pad, s.inv, g);
        int32_t bad = 0;
        double sumsq = 0.0;
        for (int64_t j = 0; j < psi_pad; ++j) {
            if (!orc_is_finite(g[j]))
                bad = 1;
            sumsq = sumsq + (double)g[j] * (double)g[j];
        }
        res->found_nonfinite = bad;
        res->sumsq = sumsq;
        res->grad_norm = (float)sqrt(sumsq);
        res->clip_coef = 1.0f;
        if (skip_on_overflow && bad) {
            res->applied = 0;
            continue;
        }
        if (hp->max_grad_norm > 0.0) {
            res->clip_coef = orc_clip_coef(hp->max_grad_norm, sqrt(sumsq));
            for (int64_t j = 0; j < psi_pad; ++j)
                g[j] = g[j] * res->clip_coef;
        }
        for (int64_t j = 0; j < psi_pad; ++j) {
            orc_adam_element(g[j], &master[i][j], &m[i][j], &v[i][j], &s);
            w[i][j] = orc_f32_to_bf16(master[i][j]);
        }
        res->applied = 1;
    }
    free(g);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Gradient accumulation over micro-batches (the DP-ZeRO blog, "stacking     */
/* with other parallelism": under pipeline parallelism the gradient arrives  */
/* micro-batch by micro-batch, so it is reduced and accumulated chunk by     */
/* chunk instead of once at the end).                                        */
/* Reading: the batch mean covers N * k contributions.  Each micro-batch adds  */
/* its combined gradient, scaled by fp32(1/(N * k * loss_scale)), to the       */
/* owner's FP32 accumulator in micro-batch order, starting from +0.  The      */
/* step-wide checks and the update then use the accumulated gradient.         */
/* ------------------------------------------------------------------------ */

/* grads holds k * N pointers, micro-batch major: grads[mb * N + r]. */
int orc_zero_step_accum(const void* const* grads, int32_t dtype, int32_t N, int32_t k,
                        int64_t psi_pad, float* master, float* m, float* v, uint16_t* w,
                        const orc_hparams* hp, int64_t t, double loss_scale,
                        int32_t skip_on_overflow, orc_result* res)
{
    if (N < 1 || k < 1 || psi_pad < 0 || psi_pad % ((int64_t)N * ORC_PAD_UNIT) != 0)
        return -1;
    orc_scalars s;
    orc_step_scalars(hp, t, N, loss_scale, &s);
    float inv = (float)(1.0 / ((double)N * (double)k * loss_scale));
    float* acc = (float*)malloc((size_t)(psi_pad > 0 ? psi_pad : 1) * sizeof(float));
    if (!acc)
        return -1;
    for (int64_t j = 0; j < psi_pad; ++j)
        acc[j] = 0.0f;
    for (int32_t mb = 0; mb < k; ++mb)
        for (int64_t j = 0; j < psi_pad; ++j)
            acc[j] = acc[j] + orc_reduce_element(grads + (int64_t)mb * N, dtype, N, j, inv);
    int32_t bad = 0;
    double sumsq = 0.0;
    for (int64_t j = 0; j < psi_pad; ++j) {
        if (!orc_is_finite(acc[j]))
            bad = 1;
        sumsq = sumsq + (double)acc[j] * (double)acc[j];
    }
    res->found_nonfinite = bad;
    res->sumsq = sumsq;
    res->grad_norm = (float)sqrt(sumsq);
    res->clip_coef = 1.0f;
    if (skip_on_overflow && bad) {
        res->applied = 0;
        free(acc);
        return 0;
    }
    if (hp->max_grad_norm > 0.0) {
        res->clip_coef = orc_clip_coef(hp->max_grad_norm, sqrt(sumsq));
        for (int64_t j = 0; j < psi_pad; ++j)
            acc[j] = acc[j] * res->clip_coef;
    }
    for (int64_t j = 0; j < psi_pad; ++j) {
        orc_adam_element(acc[j], &master[j], &m[j], &v[j], &s);
        w[j] = orc_f32_to_bf16(master[j]);
    }
    res->applied = 1;
    free(acc);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Windowed form, for vectors too large to hold on the host                   */
/* The step is elementwise once the step-wide flag and norm are known, so a  */
/* window of elements can be stepped on its own, exactly.                     */
/* ------------------------------------------------------------------------ */

/* Pass over n elements (a chunk of the flat vector, given as N pointers to
 * the ranks' contributions for that chunk), carrying the overflow flag and
 * the FP64 sum of squares across calls.  Called on consecutive chunks in
 * order this is the same sequential sum as the whole-vector step takes. */
void orc_check_accumulate(const void* const* grads, int32_t dtype, int32_t N,
                          int64_t n, float inv, int32_t* bad, double* sumsq)
{
    for (int64_t j = 0; j < n; ++j) {
        float g = orc_reduce_element(grads, dtype, N, j, inv);
        if (!orc_is_finite(g))
            *bad = 1;
        *sumsq = *sumsq + (double)g * (double)g;
    }
}

/* Steps a window of n elements given the step-wide outcome: `apply` = 0
 * leaves the window untouched; otherwise each element's combined gradient is
 * scaled by clip_coef (pass 1 when not clipping), and master/m/v/w of the
 * window are updated. */
void orc_step_window(const void* const* grads, int32_t dtype, int32_t N, int64_t n,
                     float* master, float* m, float* v, uint16_t* w,
                     const orc_hparams* hp, int64_t t, double loss_scale,
                     int32_t apply, int32_t clip, float clip_coef)
{
    if (!apply)
        return;
    orc_scalars s;
    orc_step_scalars(hp, t, N, loss_scale, &s);
    for (int64_t j = 0; j < n; ++j) {
        float g = orc_reduce_element(grads, dtype, N, j, s.inv);
        if (clip)
            g = g * clip_coef;
        orc_adam_element(g, &master[j], &m[j], &v[j], &s);
        w[j] = orc_f32_to_bf16(master[j]);
    }
}

/* The clip coefficient the whole-vector step would use for this sum of squares. */
float orc_clip_coef_from_sumsq(double max_norm, double sumsq)
{
    return orc_clip_coef(max_norm, sqrt(sumsq));
}

/* ------------------------------------------------------------------------ */
/* Dynamic loss scale (a host-side policy; not on the pages)                  */
/* On an overflowing step the scale halves and the clean-step count restarts; */
/* after `interval` clean steps in a row the scale doubles.                   */
/* ------------------------------------------------------------------------ */

void orc_loss_scale_update(double* scale, int32_t* good_steps, int32_t found_nonfinite,
                           int32_t interval, double backoff, double growth)
{
    if (found_nonfinite) {
        *scale = *scale * backoff;
        *good_steps = 0;
        return;
    }
    *good_steps = *good_steps + 1;
    if (*good_steps == interval) {
        *scale = *scale * growth;
        *good_steps = 0;
    }
}
