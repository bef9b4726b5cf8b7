// zero_step.cu -- the ZeRO update step on one GB300 (sm_103a).
//
// One step = reduce-scatter of N ranks' gradients with batch-mean scaling,
// owner-local mixed-precision Adam on the FP32 master/m/v slice, BF16 cast and
// all-gather into the full working-weight view.  Sources:
//   - lecture deck "RC-T2", note N48.  The reduction adds contributions of the
//     same parameter only, scaled to match a batch-mean loss.  The owner
//     updates its slice with its own master weight and m/v.  The next
//     all-gather fetches the updated version.
//   - topic page "Putting the training ledger onto multiple devices", section
//     "one full ZeRO-3 computation": reduce-scatter/all-gather as data
//     semantics.
//   - blog post "Data parallelism and ZeRO: how much each of the three stages
//     saves", section "three stages": ZeRO-1/2 reduce-scatter the gradient,
//     step 1/N of the FP32 state, all-gather the BF16 weights.
//
// The N simulated ranks share this device's memory, so a collective is a
// memory access pattern.  For every element j of owner r's slice, the owner
// reads grads[0..N-1][j] (the reduce-scatter).  It writes w[j] into the one
// full-view buffer (the all-gather).  All owners run concurrently: the grid
// walks the whole flat vector, and each 8-element group belongs to exactly
// one owner, because every slice is a multiple of 128 elements.
//
// The path is bound by HBM bandwidth (about 0.5 flop per byte), so nothing
// here uses tensor cores.  The one-pass step has two kernels that give the
// same bits:
//   - zero_fused_kernel: each thread loads 16-byte vectors straight into
//     registers, two 8-element groups in flight, every load of a group issued
//     before its arithmetic;
//   - zero_fused_staged_kernel: one thread per CTA copies each tile into
//     shared memory with TMA bulk copies, and sixteen warps compute from there.
// The arithmetic uses the explicit round-to-nearest intrinsics, so no
// multiply-add is ever contracted: each element is rounded operator by
// operator.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "zero_common.cuh"
#include "zero_elem.cuh"
#include "zero_gb300.h"

namespace {

constexpr int kMaxGrid = 2048;            // CTAs per launch, at most
constexpr int kFinalizeThreads = 256;
constexpr int kMaxWarps = 32;             // finish_cta's per-warp slots: blocks of <= 1024 threads
constexpr size_t kCtrlBytes = 256;
constexpr size_t kPartialsOffset = kCtrlBytes;
constexpr size_t kGradOffset = kPartialsOffset + kMaxGrid * sizeof(double);  // 256-B aligned
// Rows of norm partials (see finish_cta): one row of kMaxGrid FP64 slots per
// first-pass launch, at most kRowCap rows, in an optional area after the part
// of the workspace every step needs.  The area starts with the carry (the sum
// of the rows before the latest), padded to 256 bytes, then the rows.
constexpr int kRowCap = 2048;
constexpr size_t kRowBytes = kMaxGrid * sizeof(double);
constexpr size_t kRowsHeaderBytes = 256;


// Control block at the start of the workspace.  It is zeroed at the start of
// every step.
struct Ctrl {
    unsigned int nonfinite;    // OR over all elements of "combined gradient is inf/NaN"
    int skip;                  // decided by the finalize kernel
    float clip_coef;           // decided by the finalize kernel
    float grad_norm;
    zero_step_result result;   // the outcome, when the caller passes no result pointer
    int policy_error;          // device policy: t fell outside the given window
    unsigned int timeout;      // a bounded wait of the staged kernel gave up
    int cur;                   // ping-pong: the state set this step reads (0 or 1), set
                               // by the prologue from the caller's word
    unsigned int bounds;       // debug build: a kernel skipped an out-of-range access
    Scalars scalars;           // device policy: this step's scalars, set by the prologue
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block");
static_assert(kGradOffset % 256 == 0, "gradient workspace alignment");
static_assert(kGradOffset == ZERO_WORKSPACE_CONTROL_BYTES, "header's control-part size");

struct StepArgs {
    const void* grads[ZERO_MAX_RANKS];
    const float* src_master;
    const float* src_m;
    const float* src_v;
    const uint16_t* src_w;
    float* dst_master;
    float* dst_m;
    float* dst_v;
    uint16_t* dst_w;
    const Scalars* sdev; // device policy: read the step's scalars here instead of s
    float* gws;          // FP32 combined gradient (two-pass form) or accumulator (micro-batches)
    double* partials;    // one FP64 sum of squares per CTA: the shared slots, or this launch's row
    const double* prev_row; // own row: the row of the step's previous launch with a row (or null)
    double* carry;       // own row: the sum of the rows before prev_row, then with it added
    int32_t row_width;   // own row: the slots of this row that count, at least the grid size
    int32_t prev_width;  // own row: the same for prev_row
    int32_t carry_in;    // own row: carry already holds the rows before prev_row
    int32_t partial_mode;// what finish_cta does with the CTA's sum of squares (see there)
    Ctrl* ctrl;
    Scalars s;
    int64_t begin;       // first element of this launch (a multiple of kVec)
    int64_t n8;          // groups of kVec elements in this launch
    int64_t gbase;       // flat index of grads[i][0] (the bucket start for a staging slot)
    int32_t N;
    int32_t clip;        // 1: multiply the gradient by ctrl->clip_coef before Adam
    int32_t acc_first;   // accumulation: this is the first micro-batch (start from +0)
    int32_t acc_last;    // accumulation: the last micro-batch (form the step-wide checks)
    int32_t stages;      // staged kernel: shared-memory stages
    uint32_t stage_bytes;// staged kernel: bytes of one stage (N gradient chunks + 3 state chunks)
    int32_t test_stall;  // staged kernel: CTA 0 never copies its first tile (tests the bounded waits)
    int32_t pingpong;    // 1: read the set ctrl->cur names (0 = src_*, 1 = dst_*), write the other
    int64_t limit;       // elements in every state array and in the workspace gradient (psi_pad)
    int64_t grad_lo;     // flat elements [grad_lo, grad_hi) that the grads[i] buffers hold
    int64_t grad_hi;
};

// The step's scalars: from the kernel arguments, or, under a device policy,
// from the control block where the prologue kernel wrote them.
__device__ __forceinline__ Scalars step_scalars(const StepArgs& a) {
    return a.sdev != nullptr ? *a.sdev : a.s;
}

// Under a device policy a step whose t fell outside its window does nothing.
__device__ __forceinline__ bool policy_off(const StepArgs& a) {
    return a.sdev != nullptr && a.ctrl->policy_error != 0;
}

#ifdef ZERO_DEBUG
constexpr bool kDebugBuild = true;
#else
constexpr bool kDebugBuild = false;
#endif

// Debug build (-DZERO_DEBUG): before touching elements [j, j + len) a kernel
// checks them against the lengths of the buffers involved: the state arrays
// and the workspace gradient hold [0, limit), the gradient buffers (or the
// staging slot) [grad_lo, grad_hi).  An access outside is skipped, counted,
// and makes the step end with ZERO_ERR_BOUNDS; nothing traps.  The release
// build compiles every check to `true`.
#ifdef ZERO_DEBUG
__device__ unsigned long long g_step_bounds_violations;

__device__ __forceinline__ bool range_inside(const StepArgs& a, int64_t j, int64_t len,
                                             bool grads) {
    bool ok = j >= 0 && len >= 0 && j + len <= a.limit;
    if (grads) ok = ok && j >= a.grad_lo && j + len <= a.grad_hi;
    return ok;
}
__device__ __forceinline__ void record_violation(const StepArgs& a) {
    atomicOr(&a.ctrl->bounds, 1u);
    atomicAdd(&g_step_bounds_violations, 1ull);
}
__device__ __forceinline__ bool range_ok(const StepArgs& a, int64_t j, int64_t len, bool grads) {
    const bool ok = range_inside(a, j, len, grads);
    if (!ok) record_violation(a);
    return ok;
}
#else
__device__ __forceinline__ bool range_inside(const StepArgs&, int64_t, int64_t, bool) {
    return true;
}
__device__ __forceinline__ void record_violation(const StepArgs&) {}
__device__ __forceinline__ bool range_ok(const StepArgs&, int64_t, int64_t, bool) { return true; }
#endif

// Ping-pong state sets (zero_plan_set_pingpong).  The plan's src_* buffers
// are set 0 and its dst_* buffers set 1.  A step reads the set the control
// block names and writes the other, so `sw` (set 1 is the current one) swaps
// the two roles.  Without ping-pong sw is false: read src_*, write dst_*.
__device__ __forceinline__ bool sets_swapped(const StepArgs& a) {
    return a.pingpong != 0 && a.ctrl->cur != 0;
}
__device__ __forceinline__ const float* in_master(const StepArgs& a, bool sw) {
    return sw ? a.dst_master : a.src_master;
}
__device__ __forceinline__ const float* in_m(const StepArgs& a, bool sw) {
    return sw ? a.dst_m : a.src_m;
}
__device__ __forceinline__ const float* in_v(const StepArgs& a, bool sw) {
    return sw ? a.dst_v : a.src_v;
}
__device__ __forceinline__ float* out_master(const StepArgs& a, bool sw) {
    return sw ? const_cast<float*>(a.src_master) : a.dst_master;
}
__device__ __forceinline__ float* out_m(const StepArgs& a, bool sw) {
    return sw ? const_cast<float*>(a.src_m) : a.dst_m;
}
__device__ __forceinline__ float* out_v(const StepArgs& a, bool sw) {
    return sw ? const_cast<float*>(a.src_v) : a.dst_v;
}
__device__ __forceinline__ uint16_t* out_w(const StepArgs& a, bool sw) {
    return sw ? const_cast<uint16_t*>(a.src_w) : a.dst_w;
}

// The reduce-scatter of one 8-element group: every rank's contribution to
// these same elements, added in rank order starting from +0.  NT > 0 fixes N
// at compile time (all N loads in flight together); NT == 0 takes a.N.
template <int NT, bool kBF16>
__device__ __forceinline__ void combine(const StepArgs& a, int64_t j, float (&g)[kVec]) {
#pragma unroll
    for (int e = 0; e < kVec; ++e) g[e] = 0.0f;
    if constexpr (NT > 0) {
        GradVec<kBF16> raw[NT];
#pragma unroll
        for (int i = 0; i < NT; ++i) raw[i].load(a.grads[i], j - a.gbase);
#pragma unroll
        for (int i = 0; i < NT; ++i) raw[i].add_to(g);
    } else {
        int i = 0;
        for (; i + 4 <= a.N; i += 4) {
            GradVec<kBF16> raw[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) raw[k].load(a.grads[i + k], j - a.gbase);
#pragma unroll
            for (int k = 0; k < 4; ++k) raw[k].add_to(g);
        }
        for (; i < a.N; ++i) {
            GradVec<kBF16> raw;
            raw.load(a.grads[i], j - a.gbase);
            raw.add_to(g);
        }
    }
}

// End of a CTA's share: publish the overflow flag (one atomic per warp that
// saw a non-finite value) and record the CTA's sum of squares (warp-shuffle
// tree, then the warps in order).  Where it goes is the launch's partial mode:
//   kOwnRow     a row of slots that belongs to this launch alone: a plain
//               store (CTA 0 also zeroes the row's slots past the grid).
//   kSharedSlot the one slot per CTA index that every launch without a row
//               adds to: the add must follow the previous launch's, so thread 0
//               of every CTA first waits for that grid to complete.  While it
//               waits, the CTA keeps its SM slot from the next launch's CTAs.
//   kNoPartial  nothing (the accumulate passes before the last micro-batch).
// Launches get their own rows while the workspace has rows left; the shared
// slots serve the rest.  In the first and last modes only CTA 0 waits for the
// previous grid, at its very end: one waiting CTA is enough to make this grid
// complete after the previous one, so that a pass's last launch completing
// still means the whole pass has, and it holds one SM slot instead of all of
// them.  With a row, CTA 0 then adds the previous launch's row, now complete,
// to the carry: the carry gathers the rows in launch order, and finalize reads
// only the carry and the last row.  Every sum is formed in a fixed order.
constexpr int32_t kNoPartial = 0;
constexpr int32_t kSharedSlot = 1;
constexpr int32_t kOwnRow = 2;

// CTA 0 of a launch with a row, every thread: wait for the previous launch,
// then carry = (carry_in ? carry : 0) + the sum of prev_row's slots (each
// thread its slots in order, the warp-shuffle tree, the warps in order).
__device__ __forceinline__ void carry_previous_row(const StepArgs& a, double* warp_sum) {
    grid_dependency_wait();
    if (a.prev_row == nullptr) return;
    __syncthreads();  // thread 0 has read warp_sum
    const int width = a.prev_width < kMaxGrid ? a.prev_width : kMaxGrid;
    double t = 0.0;
    for (int b = static_cast<int>(threadIdx.x); b < width; b += static_cast<int>(blockDim.x))
        t += a.prev_row[b];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
    if ((threadIdx.x & 31) == 0) warp_sum[threadIdx.x >> 5] = t;
    __syncthreads();
    if (threadIdx.x == 0) {
        double row = 0.0;
        const int warps = static_cast<int>(blockDim.x >> 5);
        for (int w = 0; w < warps; ++w) row += warp_sum[w];
        *a.carry = a.carry_in ? *a.carry + row : row;
    }
}

__device__ __forceinline__ void finish_cta(const StepArgs& a, unsigned bad, double sumsq) {
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(&a.ctrl->nonfinite, 1u);
    if (a.partial_mode == kNoPartial) {
        if (blockIdx.x == 0 && threadIdx.x == 0) grid_dependency_wait();
        return;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sumsq += __shfl_xor_sync(0xffffffffu, sumsq, off);
    __shared__ double warp_sum[kMaxWarps];
    if ((threadIdx.x & 31) == 0) warp_sum[threadIdx.x >> 5] = sumsq;
    const bool row_cta0 = a.partial_mode == kOwnRow && blockIdx.x == 0;
    if (row_cta0) {
        const int width = a.row_width < kMaxGrid ? a.row_width : kMaxGrid;
        for (int b = static_cast<int>(gridDim.x + threadIdx.x); b < width; b += blockDim.x)
            a.partials[b] = 0.0;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        const int warps = static_cast<int>(blockDim.x >> 5);  // whole warps only
        for (int w = 0; w < warps; ++w) t += warp_sum[w];
        if (blockIdx.x >= kMaxGrid) {
            record_violation(a);
        } else if (a.partial_mode == kOwnRow) {
            a.partials[blockIdx.x] = t;
        } else {
            // A bucket launch may start while the previous one drains
            // (programmatic dependent launch).  Its slot update must still
            // come after the previous launch's: wait for that grid to complete
            // first.  Without a programmatic launch this returns at once.
            grid_dependency_wait();
            a.partials[blockIdx.x] += t;
        }
    }
    if (row_cta0) carry_previous_row(a, warp_sum);
}

// ------------------------------------------------------------------ kernels

// One 8-element group: reduce-scatter + scale + check + Adam + BF16 all-gather.
// kAccIn: the last micro-batch of an accumulated step.  The combined gradient
// is this micro-batch's scaled contribution added to the FP32 accumulator the
// earlier micro-batches left in gws (the same two roundings the accumulate
// kernel makes), and is used at once instead of being written back.
template <int NT, bool kBF16, bool kAccIn, int U>
__device__ __forceinline__ void fused_groups(const StepArgs& a, const Scalars& s, bool sw,
                                             const int64_t (&j)[U], unsigned& bad,
                                             double& sumsq) {
    float p[U][kVec], m[U][kVec], v[U][kVec], g[U][kVec];
    float acc[kAccIn ? U : 1][kVec];
    // every load of the U groups is issued before any arithmetic
#pragma unroll
    for (int u = 0; u < U; ++u) {
        load8(in_master(a, sw), j[u], p[u]);
        load8(in_m(a, sw), j[u], m[u]);
        load8(in_v(a, sw), j[u], v[u]);
        if constexpr (kAccIn) load8(a.gws, j[u], acc[u]);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) combine<NT, kBF16>(a, j[u], g[u]);
#pragma unroll
    for (int u = 0; u < U; ++u) {
        float sq = 0.0f;
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
            float gs = __fmul_rn(g[u][e], s.inv);
            if constexpr (kAccIn) gs = __fadd_rn(acc[u][e], gs);
            bad |= is_nonfinite(gs) ? 1u : 0u;
            sq = fmaf(gs, gs, sq);
            adam_element(gs, p[u][e], m[u][e], v[u][e], s);
        }
        sumsq += static_cast<double>(sq);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        store8(out_master(a, sw), j[u], p[u]);
        store8(out_m(a, sw), j[u], m[u]);
        store8(out_v(a, sw), j[u], v[u]);
        store_w8(out_w(a, sw), j[u], p[u]);
    }
}

// One pass: reduce-scatter + scale + check + Adam + BF16 all-gather.  Reads
// src_*, writes dst_* (the same arrays for an in-place step).  Each thread
// keeps two groups (a grid stride apart) in flight: with 128 registers and two
// CTAs per SM that measured faster than one group at 64 registers and four.
template <int NT, bool kBF16, bool kAccIn>
__global__ void __launch_bounds__(kThreads, 2) zero_fused_kernel(const __grid_constant__ StepArgs a) {
    allow_next_launch();
    unsigned bad = 0;
    double sumsq = 0.0;
    const Scalars s = step_scalars(a);
    const bool sw = sets_swapped(a);
    const int64_t n8 = policy_off(a) ? 0 : a.n8;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    int64_t q = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    // FP32 gradients plus the accumulator do not fit two groups in 128
    // registers without spilling: those take one group at a time.
    constexpr bool kPairs = kBF16 || !kAccIn;
    for (; kPairs && q + stride < n8; q += 2 * stride) {
        const int64_t j[2] = {a.begin + q * kVec, a.begin + (q + stride) * kVec};
        if (!range_ok(a, j[0], kVec, true) || !range_ok(a, j[1], kVec, true)) continue;
        fused_groups<NT, kBF16, kAccIn, 2>(a, s, sw, j, bad, sumsq);
    }
    for (; !kPairs && q + stride < n8; q += stride) {
        const int64_t j[1] = {a.begin + q * kVec};
        if (!range_ok(a, j[0], kVec, true)) continue;
        fused_groups<NT, kBF16, kAccIn, 1>(a, s, sw, j, bad, sumsq);
    }
    if (q < n8) {
        const int64_t j[1] = {a.begin + q * kVec};
        if (range_ok(a, j[0], kVec, true)) fused_groups<NT, kBF16, kAccIn, 1>(a, s, sw, j, bad, sumsq);
    }
    finish_cta(a, bad, sumsq);
}

// ------------------------------------------------------------------ staged one-pass kernel
//
// The same one-pass step with each tile of kTile elements staged in shared
// memory.  One producer thread copies a tile's N gradient chunks and its
// master/m/v chunks from HBM into a stage with TMA bulk copies
// (cp.async.bulk), counted in the stage's "full" mbarrier.  Sixteen consumer
// warps wait on it, compute from shared memory, store the results straight to
// HBM and arrive on the stage's "empty" mbarrier, which the producer waits on
// before it refills the stage.  Two stages per CTA: one tile is computed from
// one stage while the next tile streams into the other, the offload pattern's
// pair of alternating slots moved inside a kernel.
//
// Measured on Psi = 1e9, N = 8 BF16 (interleaved runs on one GPU, against the
// register kernel at 5.94 ms per step): 2048-element tiles, 16 consumer warps
// and 2 stages gave 5.89 ms; 8 warps 5.90; 1024-element tiles with 8 warps
// 5.91, with 4 warps 6.03; 3 stages of 1024 with 4 warps 6.21; 4 and 6 stages
// were slower still.  More consumer warps per SM mattered, deeper staging did
// not.
//
// Every wait is bounded by the global timer.  A wait that gives up sets
// ctrl->timeout, and the step ends with ZERO_ERR_TIMEOUT.  Before it leaves,
// the producer always waits (again bounded) for the copies it issued, so that
// no copy is still landing in shared memory when the CTA exits, whether the
// wait that gave up was its own or a consumer's.
//
// Consumer thread c owns the 4-element chunks starting at 4c, 4c + 4C,
// 4c + 8C, ... of a tile (C consumer threads), so each shared-memory load of a
// warp covers consecutive 8- or 16-byte words (no bank conflicts) and each
// global store of a warp is one contiguous run.  The element arithmetic is
// the register kernel's.

constexpr int kTile = 2048;
constexpr int kStagedConsumerWarps = 16;
constexpr int kStagedConsumers = 32 * kStagedConsumerWarps;
constexpr int kStagedThreads = kStagedConsumers + 32;  // + the producer warp
static_assert(kTile % (4 * kStagedConsumers) == 0, "whole 4-element chunks per consumer");
static_assert(kStagedThreads <= 32 * kMaxWarps, "finish_cta's per-warp slots");
constexpr int kMaxStages = 2;
constexpr size_t kStagedSmemLimit = 200 * 1024;  // dynamic shared memory per CTA, at most
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
// Waits for the completion of the barrier's phase of the given parity; false
// if it has not completed within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > kWaitLimitNs) return false;
    return true;
}
// L2 policy for data read exactly once: evict it first.  On Psi = 1e9, N = 8
// the staged step took 5.871 ms with it on the bulk loads and 5.889 ms without.
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    return policy;
}
// A TMA bulk copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from global to this CTA's shared memory, completing on `bar`, with
// the L2 cache policy `policy`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}
// Shared-memory loads, by shared-window address.  The memory clobber keeps
// them after the mbarrier wait that makes the stage's bytes visible.
__device__ __forceinline__ uint2 lds_u2(const void* p) {
    uint2 r;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                 : "=r"(r.x), "=r"(r.y)
                 : "r"(smem_addr(p))
                 : "memory");
    return r;
}
__device__ __forceinline__ float4 lds_f4(const void* p) {
    float4 r;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
                 : "r"(smem_addr(p))
                 : "memory");
    return r;
}

// Consumer work on 4 elements: the tile-relative element e (a multiple of 4)
// of the stage st, flat index j.
template <int NT, bool kBF16>
__device__ __forceinline__ void staged_chunk(const StepArgs& a, const Scalars& s, bool sw,
                                             const unsigned char* st, int e, int64_t j,
                                             unsigned& bad, double& sumsq) {
    constexpr uint32_t gbytes = kBF16 ? 2 : 4;
    const int n = NT > 0 ? NT : a.N;
    float g[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    // rank order from +0, as in the register kernel
#pragma unroll(NT > 0 ? NT : 1)
    for (int i = 0; i < n; ++i) {
        const unsigned char* chunk = st + static_cast<size_t>(i) * kTile * gbytes;
        if constexpr (kBF16) {
            const uint2 r = lds_u2(chunk + e * 2);
            g[0] = __fadd_rn(g[0], bf16_lo(r.x));
            g[1] = __fadd_rn(g[1], bf16_hi(r.x));
            g[2] = __fadd_rn(g[2], bf16_lo(r.y));
            g[3] = __fadd_rn(g[3], bf16_hi(r.y));
        } else {
            const float4 r = lds_f4(chunk + e * 4);
            g[0] = __fadd_rn(g[0], r.x);
            g[1] = __fadd_rn(g[1], r.y);
            g[2] = __fadd_rn(g[2], r.z);
            g[3] = __fadd_rn(g[3], r.w);
        }
    }
    const unsigned char* state = st + static_cast<size_t>(n) * kTile * gbytes;
    const float4 P = lds_f4(state + e * 4);
    const float4 M = lds_f4(state + (kTile + e) * 4);
    const float4 V = lds_f4(state + (2 * kTile + e) * 4);
    float p[4] = {P.x, P.y, P.z, P.w}, m[4] = {M.x, M.y, M.z, M.w}, v[4] = {V.x, V.y, V.z, V.w};
    float sq = 0.0f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float gs = __fmul_rn(g[q], s.inv);
        bad |= is_nonfinite(gs) ? 1u : 0u;
        sq = fmaf(gs, gs, sq);
        adam_element(gs, p[q], m[q], v[q], s);
    }
    sumsq += static_cast<double>(sq);
    __stcs(reinterpret_cast<float4*>(out_master(a, sw) + j), make_float4(p[0], p[1], p[2], p[3]));
    __stcs(reinterpret_cast<float4*>(out_m(a, sw) + j), make_float4(m[0], m[1], m[2], m[3]));
    __stcs(reinterpret_cast<float4*>(out_v(a, sw) + j), make_float4(v[0], v[1], v[2], v[3]));
    __stcs(reinterpret_cast<uint2*>(out_w(a, sw) + j),
           make_uint2(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3])));
}

template <int NT, bool kBF16>
__global__ void __launch_bounds__(kStagedThreads)
    zero_fused_staged_kernel(const __grid_constant__ StepArgs a) {
    allow_next_launch();
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr uint32_t gbytes = kBF16 ? 2 : 4;
    const int n_ranks = NT > 0 ? NT : a.N;
    const int stages = a.stages;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(stages) * a.stage_bytes);
    uint64_t* empty = full + stages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int k = 0; k < stages; ++k) {
            mbar_init(&full[k], 1);                      // the producer's arrive + the bytes
            mbar_init(&empty[k], kStagedConsumerWarps);  // one arrive per consumer warp
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const Scalars s = step_scalars(a);
    const bool sw = sets_swapped(a);
    const int64_t range = (policy_off(a) ? 0 : a.n8) * kVec;  // a multiple of 8
    const int64_t ntiles = (range + kTile - 1) / kTile;
    unsigned bad = 0, timed_out = 0;
    double sumsq = 0.0;
    if (warp == kStagedConsumerWarps) {
        if (lane == 0) {  // the producer
            const uint64_t once = evict_first_policy();
            int64_t k = 0;
            for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++k) {
                const int st_i = static_cast<int>(k % stages);
                if (k >= stages &&
                    !mbar_wait(&empty[st_i], static_cast<uint32_t>((k / stages - 1) & 1))) {
                    timed_out = 1;
                    break;
                }
                if (a.test_stall && blockIdx.x == 0 && k == 0) continue;  // never copied
                const int64_t e0 = t * kTile;
                const int64_t len = (range - e0 < kTile) ? range - e0 : kTile;
                const int64_t j = a.begin + e0;
                if (!range_ok(a, j, len, true)) {
                    // a tile outside the buffers: complete the stage's phase
                    // without copying, and the consumers skip it too
                    mbar_arrive(&full[st_i]);
                    continue;
                }
                unsigned char* st = smem + static_cast<size_t>(st_i) * a.stage_bytes;
                const uint32_t gb = static_cast<uint32_t>(len) * gbytes;
                const uint32_t sb = static_cast<uint32_t>(len) * 4u;
                mbar_arrive_expect_tx(&full[st_i], static_cast<uint32_t>(n_ranks) * gb + 3u * sb);
                for (int i = 0; i < n_ranks; ++i)
                    bulk_load(st + static_cast<size_t>(i) * kTile * gbytes,
                              static_cast<const unsigned char*>(a.grads[i]) + (j - a.gbase) * gbytes,
                              gb, &full[st_i], once);
                unsigned char* state = st + static_cast<size_t>(n_ranks) * kTile * gbytes;
                bulk_load(state, in_master(a, sw) + j, sb, &full[st_i], once);
                bulk_load(state + kTile * 4, in_m(a, sw) + j, sb, &full[st_i], once);
                bulk_load(state + 2 * kTile * 4, in_v(a, sw) + j, sb, &full[st_i], once);
            }
            // Let every copy this thread issued land before the CTA may exit,
            // whichever wait (its own or a consumer's) gave up.  A tile older
            // than the last `stages` was consumed before its stage was refilled,
            // so only those last tiles can still be in flight.  No arrival
            // follows them on their "full" barriers, so on the normal path
            // these waits see phases that have completed or are about to.
            for (int64_t kk = (k > stages ? k - stages : 0); kk < k; ++kk) {
                if (a.test_stall && blockIdx.x == 0 && kk == 0) continue;  // never issued
                mbar_wait(&full[kk % stages], static_cast<uint32_t>((kk / stages) & 1));
            }
        }
    } else {  // the consumers
        const int c = threadIdx.x;  // 0 .. kStagedConsumers - 1
        int64_t k = 0;
        for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++k) {
            const int st_i = static_cast<int>(k % stages);
            if (!mbar_wait(&full[st_i], static_cast<uint32_t>((k / stages) & 1))) {
                timed_out = 1;
                break;
            }
            const int64_t e0 = t * kTile;
            const int64_t len = (range - e0 < kTile) ? range - e0 : kTile;
            const unsigned char* st = smem + static_cast<size_t>(st_i) * a.stage_bytes;
            if (range_inside(a, a.begin + e0, len, true)) {  // as the producer decided
#pragma unroll
                for (int e = 4 * c; e < kTile; e += 4 * kStagedConsumers)
                    if (e < len)
                        staged_chunk<NT, kBF16>(a, s, sw, st, e, a.begin + e0 + e, bad, sumsq);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st_i]);
        }
    }
    if (timed_out) atomicOr(&a.ctrl->timeout, 1u);
    finish_cta(a, bad, sumsq);
}

// U groups of the first pass of the two-pass form.
template <int NT, bool kBF16, int U>
__device__ __forceinline__ void reduce_groups(const StepArgs& a, const Scalars& s,
                                              const int64_t (&j)[U], unsigned& bad,
                                              double& sumsq) {
    float g[U][kVec];
#pragma unroll
    for (int u = 0; u < U; ++u) combine<NT, kBF16>(a, j[u], g[u]);
#pragma unroll
    for (int u = 0; u < U; ++u) {
        float sq = 0.0f;
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
            g[u][e] = __fmul_rn(g[u][e], s.inv);
            bad |= is_nonfinite(g[u][e]) ? 1u : 0u;
            sq = fmaf(g[u][e], g[u][e], sq);
        }
        sumsq += static_cast<double>(sq);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) store8(a.gws, j[u], g[u]);
}

// First pass of the two-pass form: reduce-scatter + scale + check, writing the
// FP32 combined gradient to the workspace.  Two groups per thread in flight,
// as in the fused kernel.
template <int NT, bool kBF16>
__global__ void __launch_bounds__(kThreads, 2) zero_reduce_kernel(const __grid_constant__ StepArgs a) {
    allow_next_launch();
    unsigned bad = 0;
    double sumsq = 0.0;
    const Scalars s = step_scalars(a);
    const int64_t n8 = policy_off(a) ? 0 : a.n8;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    int64_t q = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    for (; q + stride < n8; q += 2 * stride) {
        const int64_t j[2] = {a.begin + q * kVec, a.begin + (q + stride) * kVec};
        if (!range_ok(a, j[0], kVec, true) || !range_ok(a, j[1], kVec, true)) continue;
        reduce_groups<NT, kBF16, 2>(a, s, j, bad, sumsq);
    }
    if (q < n8) {
        const int64_t j[1] = {a.begin + q * kVec};
        if (range_ok(a, j[0], kVec, true)) reduce_groups<NT, kBF16, 1>(a, s, j, bad, sumsq);
    }
    finish_cta(a, bad, sumsq);
}

// U groups of one micro-batch of gradient accumulation: every load first,
// then the arithmetic, then the stores.
template <int NT, bool kBF16, int U>
__device__ __forceinline__ void accum_groups(const StepArgs& a, const Scalars& s,
                                             const int64_t (&j)[U], unsigned& bad,
                                             double& sumsq) {
    float acc[U][kVec], g[U][kVec];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        if (a.acc_first) {
#pragma unroll
            for (int e = 0; e < kVec; ++e) acc[u][e] = 0.0f;
        } else {
            load8(a.gws, j[u], acc[u]);
        }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) combine<NT, kBF16>(a, j[u], g[u]);
#pragma unroll
    for (int u = 0; u < U; ++u) {
        float sq = 0.0f;
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
            acc[u][e] = __fadd_rn(acc[u][e], __fmul_rn(g[u][e], s.inv));
            bad |= is_nonfinite(acc[u][e]) ? 1u : 0u;
            sq = fmaf(acc[u][e], acc[u][e], sq);
        }
        if (a.acc_last) sumsq += static_cast<double>(sq);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) store8(a.gws, j[u], acc[u]);
}

// One micro-batch of gradient accumulation: the reduce-scatter of this
// micro-batch's contributions, scaled to the batch mean over all N * k of them,
// added to the owner's FP32 accumulator.  The last micro-batch also forms the
// overflow flag and the norm of the accumulated gradient.  Two groups per
// thread are in flight, as in the fused kernel.
template <int NT, bool kBF16>
__global__ void __launch_bounds__(kThreads, 2) zero_accum_kernel(const __grid_constant__ StepArgs a) {
    allow_next_launch();
    unsigned bad = 0;
    double sumsq = 0.0;
    const Scalars s = step_scalars(a);
    const int64_t n8 = policy_off(a) ? 0 : a.n8;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    int64_t q = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    for (; q + stride < n8; q += 2 * stride) {
        const int64_t j[2] = {a.begin + q * kVec, a.begin + (q + stride) * kVec};
        if (!range_ok(a, j[0], kVec, true) || !range_ok(a, j[1], kVec, true)) continue;
        accum_groups<NT, kBF16, 2>(a, s, j, bad, sumsq);
    }
    if (q < n8) {
        const int64_t j[1] = {a.begin + q * kVec};
        if (range_ok(a, j[0], kVec, true)) accum_groups<NT, kBF16, 1>(a, s, j, bad, sumsq);
    }
    finish_cta(a, a.acc_last ? bad : 0u, sumsq);
}

__device__ __forceinline__ void copy_state(const StepArgs& a) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; q < a.n8;
         q += stride) {
        const int64_t j = a.begin + q * kVec;
        if (!range_ok(a, j, kVec, false)) continue;
        float x[kVec];
        load8(a.src_master, j, x);
        store8(a.dst_master, j, x);
        load8(a.src_m, j, x);
        store8(a.dst_m, j, x);
        load8(a.src_v, j, x);
        store8(a.dst_v, j, x);
        __stcs(reinterpret_cast<uint4*>(a.dst_w + j),
               __ldcs(reinterpret_cast<const uint4*>(a.src_w + j)));
    }
}

// U groups of the second pass: Adam + BF16 all-gather from the combined
// gradient, clipped by coef when the step clips.
template <int U>
__device__ __forceinline__ void update_groups(const StepArgs& a, const Scalars& s, float coef,
                                              bool sw, const int64_t (&j)[U]) {
    float p[U][kVec], m[U][kVec], v[U][kVec], g[U][kVec];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        load8(in_master(a, sw), j[u], p[u]);
        load8(in_m(a, sw), j[u], m[u]);
        load8(in_v(a, sw), j[u], v[u]);
        load8(a.gws, j[u], g[u]);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
            const float gs = a.clip ? __fmul_rn(g[u][e], coef) : g[u][e];
            adam_element(gs, p[u][e], m[u][e], v[u][e], s);
        }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        store8(out_master(a, sw), j[u], p[u]);
        store8(out_m(a, sw), j[u], m[u]);
        store8(out_v(a, sw), j[u], v[u]);
        store_w8(out_w(a, sw), j[u], p[u]);
    }
}

// Second pass of the two-pass form: Adam + BF16 all-gather from the
// workspace's combined gradient, unless the step was skipped.  A skipped
// out-of-place step copies src to dst instead, except with ping-pong sets,
// where the current set simply stays current.  Two groups per thread in
// flight, as in the fused kernel.
__global__ void __launch_bounds__(kThreads, 2) zero_update_kernel(const __grid_constant__ StepArgs a) {
    allow_next_launch();
    if (a.ctrl->skip) {
        if (a.dst_master != a.src_master && !a.pingpong) copy_state(a);
    } else {
        const float coef = a.ctrl->clip_coef;
        const Scalars s = step_scalars(a);
        const bool sw = sets_swapped(a);
        const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
        int64_t q = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
        for (; q + stride < a.n8; q += 2 * stride) {
            const int64_t j[2] = {a.begin + q * kVec, a.begin + (q + stride) * kVec};
            if (!range_ok(a, j[0], kVec, false) || !range_ok(a, j[1], kVec, false)) continue;
            update_groups<2>(a, s, coef, sw, j);
        }
        if (q < a.n8) {
            const int64_t j[1] = {a.begin + q * kVec};
            if (range_ok(a, j[0], kVec, false)) update_groups<1>(a, s, coef, sw, j);
        }
    }
    // A sub-launch chained to the previous one completes only after it (one
    // waiting CTA is enough): the step's last launch completing then means
    // the whole pass has.
    if (blockIdx.x == 0 && threadIdx.x == 0) grid_dependency_wait();
}

// After a one-pass out-of-place step: a skipped step must leave dst equal to
// src, so copy it; an applied step needs nothing.  Not launched with ping-pong
// sets, where a skipped step leaves the current set current.
__global__ void __launch_bounds__(kThreads) zero_restore_kernel(const __grid_constant__ StepArgs a) {
    if (a.ctrl->skip) copy_state(a);
}

// Step-wide decision: sums the per-CTA partials in a fixed order, forms the
// norm and clip coefficient, decides the skip, and writes the result.  One CTA,
// launched as a programmatic dependent of the step's last first-pass launch, so
// that its launch overlaps that launch's drain; every thread first waits for
// that grid to complete, which (each launch completing after the one before
// it) means every first-pass launch has.  The sum of squares is the carry (the
// rows before the last, gathered by the launches themselves) plus the
// block-wide sum of the shared slots (if any launch added to them) and the
// last row: each thread its slots in order, the warp-shuffle tree, the warps
// in order.
__device__ __forceinline__ void decide(Ctrl* ctrl, double sumsq, double max_norm,
                                       int skip_on_overflow, zero_step_result* result,
                                       zero_device_policy* policy, int32_t* current_set) {
    const double norm = sqrt(sumsq);
    const int nonfinite = ctrl->nonfinite != 0u;
    const int window_miss = (policy != nullptr && ctrl->policy_error) ? 1 : 0;
    const int timeout = ctrl->timeout != 0u;
    const int bounds = ctrl->bounds != 0u;   // debug build only
    const int skip = ((skip_on_overflow && nonfinite) || window_miss || timeout || bounds) ? 1 : 0;
    float coef = 1.0f;
    if (max_norm > 0.0 && !skip) {
        const double c = max_norm / (norm + 1e-6);
        coef = (c < 1.0) ? static_cast<float>(c) : 1.0f;  // a NaN norm compares false
    }
    ctrl->skip = skip;
    ctrl->clip_coef = coef;
    ctrl->grad_norm = static_cast<float>(norm);
    zero_step_result r;
    r.status = bounds        ? ZERO_ERR_BOUNDS
               : timeout     ? ZERO_ERR_TIMEOUT
               : window_miss ? ZERO_ERR_POLICY_WINDOW
               : skip        ? ZERO_STEP_SKIPPED
                             : ZERO_OK;
    r.found_nonfinite = static_cast<uint32_t>(nonfinite);
    r.grad_norm = static_cast<float>(norm);
    r.clip_coef = coef;
    *result = r;
    // ping-pong: an applied step made the other set current.  The step's own
    // kernels read the snapshot in ctrl->cur, never this word, so a second
    // pass after this kernel still reads and writes the right sets.
    if (current_set != nullptr) {
        if (!skip) *current_set = ctrl->cur ^ 1;
        __threadfence_system();
    }
    if (policy != nullptr) {
        // the host-side rule, kept on the device: t counts applied steps; the
        // dynamic scale backs off after an overflow, grows after
        // growth_interval clean steps
        if (!window_miss && !timeout && !bounds) {
            if (!skip) policy->t += 1;
            if (policy->growth_interval > 0) {
                if (nonfinite) {
                    policy->loss_scale *= policy->backoff;
                    policy->good_steps = 0;
                } else if (++policy->good_steps == policy->growth_interval) {
                    policy->loss_scale *= policy->growth;
                    policy->good_steps = 0;
                }
            }
        }
        policy->last_status = r.status;
        __threadfence_system();
    }
}

__global__ void __launch_bounds__(kFinalizeThreads)
zero_finalize_kernel(Ctrl* ctrl, const double* partials, int32_t use_shared,
                     const double* last_row, int32_t last_width, const double* carry,
                     double max_norm, int skip_on_overflow, zero_step_result* result,
                     zero_device_policy* policy, int32_t* current_set) {
    grid_dependency_wait();
    constexpr int T = kFinalizeThreads;
    constexpr int kPer = kMaxGrid / T;
    static_assert(kMaxGrid % T == 0, "whole slots per thread");
    // every load issued before the first add: the shared slots, the last row
    const int width = last_row == nullptr ? 0 : (last_width < kMaxGrid ? last_width : kMaxGrid);
    double x[kPer], y[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int b = static_cast<int>(threadIdx.x) + k * T;
        x[k] = use_shared ? partials[b] : 0.0;
        y[k] = b < width ? last_row[b] : 0.0;
    }
    const double before = (carry != nullptr && threadIdx.x == 0) ? *carry : 0.0;
    double t = 0.0;
#pragma unroll
    for (int k = 0; k < kPer; ++k) t += x[k];
#pragma unroll
    for (int k = 0; k < kPer; ++k) t += y[k];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
    __shared__ double warp_sum[T / 32];
    if ((threadIdx.x & 31) == 0) warp_sum[threadIdx.x >> 5] = t;
    __syncthreads();
    if (threadIdx.x != 0) return;
    double rest = 0.0;
    for (int w = 0; w < T / 32; ++w) rest += warp_sum[w];
    decide(ctrl, before + rest, max_norm, skip_on_overflow, result, policy, current_set);
}

struct PolicyTable {
    float step_size[ZERO_POLICY_WINDOW];  // lr / (1 - beta1^t) for t = t_first + i
    float sbc2[ZERO_POLICY_WINDOW];       // sqrt(1 - beta2^t)
};

// Start of a step that keeps state on the device.
//   - Ping-pong sets: snapshots which set is current into the control block,
//     where every kernel of the step reads it.
//   - Device policy: picks the scalars for t' = policy->t + 1 from the host's
//     window, forms the batch-mean factor from the device's loss scale, and
//     leaves them in the control block for the step's kernels.
__global__ void zero_step_prologue_kernel(const zero_device_policy* policy, Ctrl* ctrl,
                                          Scalars base, PolicyTable table, int64_t t_first,
                                          int32_t t_count, double ranks_times_micro,
                                          const int32_t* current_set) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    if (current_set != nullptr)
        ctrl->cur = *reinterpret_cast<const volatile int32_t*>(current_set) != 0 ? 1 : 0;
    if (policy == nullptr) return;
    const int64_t idx = policy->t + 1 - t_first;
    Scalars s = base;
    if (idx < 0 || idx >= t_count) {
        ctrl->policy_error = 1;  // every kernel of the step then leaves the state alone
    } else {
        s.step_size = table.step_size[idx];
        s.sbc2 = table.sbc2[idx];
    }
    s.inv = static_cast<float>(1.0 / (ranks_times_micro * static_cast<double>(policy->loss_scale)));
    ctrl->scalars = s;
}

// ------------------------------------------------------------------ host side

using StepKernel = void (*)(StepArgs);

template <int NT, bool B>
struct FusedK {
    static constexpr StepKernel fn = zero_fused_kernel<NT, B, false>;
};
template <int NT, bool B>
struct FusedAccK {
    static constexpr StepKernel fn = zero_fused_kernel<NT, B, true>;
};
template <int NT, bool B>
struct ReduceK {
    static constexpr StepKernel fn = zero_reduce_kernel<NT, B>;
};

template <int NT, bool B>
struct StagedK {
    static constexpr StepKernel fn = zero_fused_staged_kernel<NT, B>;
};
template <int NT, bool B>
struct AccumK {
    static constexpr StepKernel fn = zero_accum_kernel<NT, B>;
};

template <template <int, bool> class K>
StepKernel pick(int N, bool bf16) {
    switch (N) {
        case 1: return bf16 ? K<1, true>::fn : K<1, false>::fn;
        case 2: return bf16 ? K<2, true>::fn : K<2, false>::fn;
        case 4: return bf16 ? K<4, true>::fn : K<4, false>::fn;
        case 8: return bf16 ? K<8, true>::fn : K<8, false>::fn;
        default: return bf16 ? K<0, true>::fn : K<0, false>::fn;
    }
}


// Launch shape of a step kernel: the register kernels take one 8-element group
// per thread and no dynamic shared memory; the staged kernel one kTile tile
// per CTA and `smem` bytes of stages.
struct Shape {
    int threads = kThreads;
    size_t smem = 0;
    bool tiles = false;
};

// Persistent grid: as many CTAs as fit on the device at once (a multiple of
// the SM count), fewer if the range is small.
// The grid of a launch with work for every resident CTA: every SM full, at
// most kMaxGrid CTAs.
int full_grid(const void* fn, int device, const Shape& sh = Shape{}) {
    const int64_t full =
        static_cast<int64_t>(sm_count(device)) * resident_ctas(fn, device, sh.threads, sh.smem);
    return full > kMaxGrid ? kMaxGrid : (full < 1 ? 1 : static_cast<int>(full));
}

int grid_for(const void* fn, int device, int64_t n8, const Shape& sh = Shape{}) {
    const int64_t need = sh.tiles ? (n8 * kVec + kTile - 1) / kTile : (n8 + sh.threads - 1) / sh.threads;
    const int full = full_grid(fn, device, sh);
    return need < 1 ? 1 : (need < full ? static_cast<int>(need) : full);
}

// Launches fn over a.n8 groups.  With overlap_previous the launch may begin
// while the kernel before it on the stream drains (programmatic dependent
// launch); only first-pass bucket launches of one step, whose elements are
// disjoint from the previous bucket's, ask for it.
bool launch(StepKernel fn, int device, const StepArgs& a, cudaStream_t stream,
            bool overlap_previous = false, const Shape& sh = Shape{}) {
    const int grid = grid_for(reinterpret_cast<const void*>(fn), device, a.n8, sh);
    if (overlap_previous || sh.smem > 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(static_cast<unsigned>(sh.threads));
        cfg.dynamicSmemBytes = sh.smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = overlap_previous ? 1 : 0;
        if (cudaLaunchKernelEx(&cfg, fn, a) != cudaSuccess) return false;
    } else {
        fn<<<grid, kThreads, 0, stream>>>(a);
    }
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cudaGetLastError() == cudaSuccess;
}

// Largest range one launch covers.  A longer range (a large bucket, or the
// whole vector when the step has one bucket) is split into near-equal
// sub-launches chained by programmatic dependent launch: each one starts
// streaming while the previous drains.  Measured on flat vectors of 1.2e8 to
// 3e9 elements, a cap of 4M elements per launch was the most consistent
// choice, against 6M to 16M.  For Psi = 1e9, N = 8 in 25M buckets it gave
// 6.76 TB/s, against 6.54 TB/s with one launch per bucket.
constexpr int64_t kLaunchElems = int64_t(1) << 22;
constexpr int64_t kLaunchAlignGroups = 32;  // 256 elements

// Launches fn over elements [begin, end) of a (a multiple of kVec long), in
// sub-launches of at most kLaunchElems.  The first sub-launch overlaps the
// kernel before it on the stream only if overlap_first; the others always
// follow a sub-launch of the same range.
// Where the first-pass launches of a step put their norm partials: rows of
// their own while the workspace has rows left (see finish_cta), then the
// shared slots.  rows == nullptr or capacity 0: the shared slots only.
struct RowSource {
    double* rows = nullptr;      // capacity rows of kMaxGrid slots
    double* carry = nullptr;
    int32_t capacity = 0;
    int32_t* used = nullptr;     // rows handed out so far in this step
    int32_t* width = nullptr;    // the slots of the latest row that count
    int32_t* shared = nullptr;   // set to 1 once a launch adds to the shared slots
    int32_t mode_without_row = kSharedSlot;
};

bool launch_range(StepKernel fn, int device, StepArgs a, int64_t begin, int64_t end,
                  cudaStream_t stream, bool overlap_first, const Shape& sh = Shape{},
                  int64_t overrun_groups = 0, RowSource* rs = nullptr) {
    const int64_t groups = (end - begin) / kVec;
    if (groups <= 0) return true;
    const int64_t parts = (groups * kVec + kLaunchElems - 1) / kLaunchElems;
    // Sub-launch sizes are a multiple of kLaunchAlignGroups, so each sub-launch
    // starts as aligned as the range does.  With a range starting on a
    // 512-byte boundary, every warp's 16-byte-per-lane access then covers
    // whole 128-byte lines.  Split at an odd offset instead, each warp access
    // straddles one more line: measured 8-9 % slower.
    int64_t per = (groups + parts - 1) / parts;
    per = (per + kLaunchAlignGroups - 1) / kLaunchAlignGroups * kLaunchAlignGroups;
    for (int64_t k = 0, g0 = 0; g0 < groups; ++k, g0 += per) {
        a.begin = begin + g0 * kVec;
        a.n8 = (groups - g0 < per) ? groups - g0 : per;
        if (g0 + per >= groups) a.n8 += overrun_groups;  // the last launch (debug tests only)
        if (rs != nullptr) {
            if (rs->mode_without_row != kNoPartial && *rs->used < rs->capacity) {
                const int32_t j = *rs->used;
                a.partial_mode = kOwnRow;
                a.partials = rs->rows + static_cast<int64_t>(j) * kMaxGrid;
                // as wide as a full launch of this kernel: a shorter launch
                // zeroes the slots past its grid
                a.row_width = full_grid(reinterpret_cast<const void*>(fn), device, sh);
                a.prev_row = j > 0 ? a.partials - kMaxGrid : nullptr;
                a.prev_width = j > 0 ? *rs->width : 0;
                a.carry = rs->carry;
                a.carry_in = j >= 2 ? 1 : 0;
                *rs->width = a.row_width;
                *rs->used = j + 1;
            } else {
                a.partial_mode = rs->mode_without_row;
                if (a.partial_mode == kSharedSlot) *rs->shared = 1;
            }
        }
        if (!launch(fn, device, a, stream, k > 0 || overlap_first, sh)) return false;
    }
    return true;
}


// The staged kernel's TMA copies read device memory only (not pinned host or
// managed memory, which the register kernels can also read).
bool device_memory(const void* ptr) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
        cudaGetLastError();  // clear the error that query may leave behind
        return false;
    }
    return attr.type == cudaMemoryTypeDevice;
}

// Stages of the staged kernel for N ranks: as many as fit (at most
// kMaxStages) in kStagedSmemLimit, at least two.  Fills a.stages,
// a.stage_bytes and the launch shape; false if two stages do not fit.
bool staged_shape(StepKernel fn, int device, int N, bool bf16, StepArgs& a, Shape& sh) {
    const size_t stage = static_cast<size_t>(N) * kTile * (bf16 ? 2 : 4) + 3 * size_t(kTile) * 4;
    int stages = kMaxStages;
    while (stages >= 2 && stages * (stage + 16) > kStagedSmemLimit) --stages;
    if (stages < 2) return false;
    {
        static std::mutex mu;
        static std::map<std::pair<const void*, int>, bool> opted_in;
        std::lock_guard<std::mutex> lock(mu);
        auto key = std::make_pair(reinterpret_cast<const void*>(fn), device);
        if (!opted_in[key]) {
            if (cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kStagedSmemLimit)) != cudaSuccess)
                return false;
            opted_in[key] = true;
        }
    }
    a.stages = stages;
    a.stage_bytes = static_cast<uint32_t>(stage);
    sh.threads = kStagedThreads;
    sh.smem = stages * stage + 2 * stages * sizeof(uint64_t);
    sh.tiles = true;
    return true;
}

struct Span {
    uintptr_t lo, hi;
    bool written;
};

bool overlaps(const Span& x, const Span& y) { return x.lo < y.hi && y.lo < x.hi; }

bool disjoint(const Span* s, int n) {
    for (int i = 0; i < n; ++i)
        for (int k = i + 1; k < n; ++k) {
            if (!s[i].written && !s[k].written) continue;  // read-only buffers may share memory
            if (overlaps(s[i], s[k])) return false;
        }
    return true;
}

bool valid_hparams(const zero_adam_hparams* hp) {
    if (hp == nullptr) return false;
    auto finite = [](double x) { return std::isfinite(x); };
    return finite(hp->lr) && hp->lr >= 0.0 && finite(hp->beta1) && hp->beta1 >= 0.0 &&
           hp->beta1 < 1.0 && finite(hp->beta2) && hp->beta2 >= 0.0 && hp->beta2 < 1.0 &&
           finite(hp->eps) && hp->eps > 0.0 && finite(hp->weight_decay) &&
           hp->weight_decay >= 0.0 && finite(hp->max_grad_norm) && hp->max_grad_norm >= 0.0 &&
           hp->step >= 1 && (hp->skip_on_overflow == 0 || hp->skip_on_overflow == 1) &&
           hp->micro_batches >= 0 && hp->bucket_elems >= 0 &&
           hp->bucket_elems % ZERO_BUCKET_ALIGN == 0;
}

int32_t micro_batches_of(const zero_adam_hparams* hp) {
    return hp->micro_batches > 1 ? hp->micro_batches : 1;
}

// The update must wait for the step-wide decision: with clipping, or when a
// skipped in-place step would have nothing left to restore from.
bool needs_two_passes(const zero_adam_hparams* hp, bool in_place) {
    return hp->max_grad_norm > 0.0 || (in_place && hp->skip_on_overflow);
}

Scalars make_scalars(const zero_adam_hparams* hp, int32_t N, float loss_scale) {
    Scalars s;
    const double t = static_cast<double>(hp->step);
    // the batch mean covers N ranks times the micro-batches accumulated
    s.inv = static_cast<float>(1.0 / (static_cast<double>(N) * micro_batches_of(hp) *
                                      static_cast<double>(loss_scale)));
    s.b1 = static_cast<float>(hp->beta1);
    s.omb1 = static_cast<float>(1.0 - hp->beta1);
    s.b2 = static_cast<float>(hp->beta2);
    s.omb2 = static_cast<float>(1.0 - hp->beta2);
    s.eps = static_cast<float>(hp->eps);
    s.step_size = static_cast<float>(hp->lr / (1.0 - std::pow(hp->beta1, t)));
    s.sbc2 = static_cast<float>(std::sqrt(1.0 - std::pow(hp->beta2, t)));
    s.decay = static_cast<float>(1.0 - hp->lr * hp->weight_decay);
    s.use_decay = hp->weight_decay != 0.0 ? 1 : 0;
    return s;
}

// The part of the workspace every step needs: the control block and shared
// slots, plus the FP32 combined gradient when the step keeps one.
size_t workspace_bytes(int64_t psi_pad, const zero_adam_hparams* hp, bool in_place) {
    size_t b = kGradOffset;
    if (needs_two_passes(hp, in_place) || micro_batches_of(hp) > 1)
        b += static_cast<size_t>(psi_pad) * sizeof(float);
    return b;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Bytes of a rows area holding `rows` rows: the finalize block sums, then the
// rows.
size_t rows_area_bytes(int64_t rows) {
    if (rows <= 0) return 0;
    return kRowsHeaderBytes + static_cast<size_t>(rows) * kRowBytes;
}

// First-pass launches in one pass over psi_pad elements in buckets of
// hp->bucket_elems (launch_range's split), at most kRowCap.
int64_t launches_per_pass(int64_t psi_pad, const zero_adam_hparams* hp) {
    auto parts = [](int64_t len) -> int64_t {
        const int64_t groups = len / kVec;
        return groups <= 0 ? 0 : (groups * kVec + kLaunchElems - 1) / kLaunchElems;
    };
    if (psi_pad <= 0) return 0;
    const int64_t bucket = hp->bucket_elems > 0 ? hp->bucket_elems : psi_pad;
    const int64_t full = psi_pad / bucket;
    const int64_t total = (full > kRowCap ? kRowCap : full) * parts(bucket) + parts(psi_pad - full * bucket);
    return total > kRowCap ? kRowCap : total;
}

// Rows a rows area of `avail` bytes holds.
int32_t rows_capacity(size_t avail) {
    if (avail <= kRowsHeaderBytes) return 0;
    const int64_t c = static_cast<int64_t>((avail - kRowsHeaderBytes) / kRowBytes);
    return static_cast<int32_t>(c > kRowCap ? kRowCap : c);
}

// The rows area of a plan's workspace.
struct RowArea {
    double* carry = nullptr;
    double* rows = nullptr;
};

RowArea row_area(const zero_plan* p) {
    RowArea r;
    if (p->row_capacity <= 0) return r;
    char* base = static_cast<char*>(p->workspace) + p->rows_offset;
    r.carry = reinterpret_cast<double*>(base);
    r.rows = reinterpret_cast<double*>(base + kRowsHeaderBytes);
    return r;
}

size_t grad_elem_bytes(int32_t dtype) { return dtype == ZERO_GRAD_BF16 ? 2u : 4u; }

// The buffers a step writes, as spans (for the overlap checks).
int written_spans(const zero_plan* p, Span* out) {
    const uintptr_t n = static_cast<uintptr_t>(p->psi_pad);
    int k = 0;
    auto add = [&](const void* ptr, uintptr_t bytes) {
        if (ptr != nullptr)
            out[k++] = Span{reinterpret_cast<uintptr_t>(ptr), reinterpret_cast<uintptr_t>(ptr) + bytes,
                            true};
    };
    add(p->dst_master, 4 * n);
    add(p->dst_m, 4 * n);
    add(p->dst_v, 4 * n);
    add(p->dst_w_bf16, 2 * n);
    // the workspace up to the end of what the step touches (its rows area too)
    const size_t needed = p->grad_accum != nullptr ? kGradOffset
                                                   : workspace_bytes(p->psi_pad, &p->hp, p->in_place != 0);
    const size_t touched = p->row_capacity > 0
                               ? static_cast<size_t>(p->rows_offset) + rows_area_bytes(p->row_capacity)
                               : needed;
    add(p->workspace, touched);
    if (p->grad_accum != nullptr) add(p->grad_accum, 4 * n);
    return k;
}

// Debug builds only, to test the checks: ZERO_DEBUG_TEST_OVERRUN=g makes the
// last launch of each pass over the vector cover g more 8-element groups past
// its end (at most 1024), which the kernels' checks must skip.  The release
// build never overruns.
int64_t debug_test_overrun() {
#ifdef ZERO_DEBUG
    static const int64_t g = [] {
        const char* v = std::getenv("ZERO_DEBUG_TEST_OVERRUN");
        const long long x = v != nullptr ? std::atoll(v) : 0;
        return static_cast<int64_t>(x < 0 ? 0 : (x > 1024 ? 1024 : x));
    }();
    return g;
#else
    return 0;
#endif
}

StepArgs base_args(const zero_plan* p) {
    char* ws = static_cast<char*>(p->workspace);
    StepArgs a{};
    for (int i = 0; i < p->N; ++i) a.grads[i] = p->grads[i];
    a.src_master = p->src_master;
    a.src_m = p->src_m;
    a.src_v = p->src_v;
    a.src_w = p->src_w_bf16;
    a.dst_master = p->dst_master;
    a.dst_m = p->dst_m;
    a.dst_v = p->dst_v;
    a.dst_w = p->dst_w_bf16;
    a.gws = p->grad_accum != nullptr ? p->grad_accum : reinterpret_cast<float*>(ws + kGradOffset);
    a.partials = reinterpret_cast<double*>(ws + kPartialsOffset);
    a.ctrl = reinterpret_cast<Ctrl*>(ws);
    a.s = make_scalars(&p->hp, p->N, p->loss_scale);
    a.sdev = p->policy != nullptr ? &a.ctrl->scalars : nullptr;
    a.N = p->N;
    a.clip = p->hp.max_grad_norm > 0.0 ? 1 : 0;
    a.gbase = 0;
    a.pingpong = p->current_set != nullptr ? 1 : 0;
    a.limit = p->psi_pad;
    a.grad_lo = 0;
    a.grad_hi = p->psi_pad;
    a.partial_mode = kSharedSlot;
    return a;
}

int plan_init(zero_plan* plan, const void* const* grads, int32_t grad_dtype,
              const float* src_master, const float* src_m, const float* src_v,
              const uint16_t* src_w, float* dst_master, float* dst_m, float* dst_v,
              uint16_t* dst_w, int64_t psi_pad, int32_t N, const zero_adam_hparams* hp,
              float loss_scale, void* workspace, size_t workspace_bytes_given,
              bool allow_null_grads, float* grad_accum = nullptr) {
    if (plan == nullptr) return ZERO_ERR_ARG;
    const bool in_place = (dst_master == src_master);
    if (grads == nullptr || N < 1 || N > ZERO_MAX_RANKS || psi_pad < 0 ||
        (grad_dtype != ZERO_GRAD_BF16 && grad_dtype != ZERO_GRAD_FP32) || !valid_hparams(hp) ||
        !(loss_scale > 0.0f) || !std::isfinite(loss_scale))
        return ZERO_ERR_ARG;
    if (psi_pad % (static_cast<int64_t>(N) * ZERO_PAD_UNIT) != 0) return ZERO_ERR_ARG;
    const bool have_data = psi_pad > 0;
    const void* bufs[] = {src_master, src_m, src_v, dst_master, dst_m, dst_v, dst_w};
    for (const void* p : bufs)
        if (have_data && p == nullptr) return ZERO_ERR_ARG;
    if (!in_place && hp->skip_on_overflow && have_data && src_w == nullptr) return ZERO_ERR_ARG;
    if (in_place && (src_m != dst_m || src_v != dst_v)) return ZERO_ERR_ARG;
    for (int i = 0; i < N; ++i) {
        if (have_data && grads[i] == nullptr && !allow_null_grads) return ZERO_ERR_ARG;
        if (!aligned(grads[i], ZERO_ALIGN_BYTES)) return ZERO_ERR_ALIGN;
    }
    for (const void* p : bufs)
        if (!aligned(p, ZERO_ALIGN_BYTES)) return ZERO_ERR_ALIGN;
    if (!aligned(src_w, ZERO_ALIGN_BYTES)) return ZERO_ERR_ALIGN;
    float* accum_dev = nullptr;  // grad_accum as the device addresses it
    if (grad_accum != nullptr) {
        if (!aligned(grad_accum, ZERO_ALIGN_BYTES)) return ZERO_ERR_ALIGN;
        cudaPointerAttributes attr;
        if (cudaPointerGetAttributes(&attr, grad_accum) != cudaSuccess ||
            attr.devicePointer == nullptr) {
            cudaGetLastError();  // clear the error that query may leave behind
            return ZERO_ERR_ARG;
        }
        accum_dev = static_cast<float*>(attr.devicePointer);
    }
    const size_t need = grad_accum != nullptr ? kGradOffset : workspace_bytes(psi_pad, hp, in_place);
    if (workspace == nullptr || workspace_bytes_given < need || !aligned(workspace, 256))
        return ZERO_ERR_WORKSPACE;

    zero_plan p{};
    for (int i = 0; i < N; ++i) p.grads[i] = grads[i];
    p.src_master = src_master;
    p.src_m = src_m;
    p.src_v = src_v;
    p.src_w_bf16 = src_w;
    p.dst_master = dst_master;
    p.dst_m = dst_m;
    p.dst_v = dst_v;
    p.dst_w_bf16 = dst_w;
    p.workspace = workspace;
    p.workspace_bytes = workspace_bytes_given;
    p.psi_pad = psi_pad;
    p.cursor = 0;
    p.hp = *hp;
    p.loss_scale = loss_scale;
    p.grad_dtype = grad_dtype;
    p.N = N;
    p.in_place = in_place ? 1 : 0;
    p.two_pass = (needs_two_passes(hp, in_place) || grad_accum != nullptr) ? 1 : 0;
    p.grad_accum = accum_dev;
    p.state = 1;
    // whatever the workspace holds beyond what the step needs becomes rows of
    // norm partials (see finish_cta)
    p.rows_offset = static_cast<int64_t>(align256(need));
    p.row_capacity = workspace_bytes_given > static_cast<size_t>(p.rows_offset)
                         ? rows_capacity(workspace_bytes_given - static_cast<size_t>(p.rows_offset))
                         : 0;
    p.rows_used = 0;
    p.row_width = 0;
    p.shared_slots_used = 0;

    if (have_data) {
        const uintptr_t n = static_cast<uintptr_t>(psi_pad);
        Span sp[ZERO_MAX_RANKS + 12];  // grads + up to 6 written + 4 read-only
        int k = written_spans(&p, sp);
        auto add = [&](const void* ptr, uintptr_t bytes) {
            if (ptr != nullptr)
                sp[k++] = Span{reinterpret_cast<uintptr_t>(ptr),
                               reinterpret_cast<uintptr_t>(ptr) + bytes, false};
        };
        for (int i = 0; i < N; ++i) add(grads[i], n * grad_elem_bytes(grad_dtype));
        if (!in_place) {
            add(src_master, 4 * n);
            add(src_m, 4 * n);
            add(src_v, 4 * n);
            if (hp->skip_on_overflow) add(src_w, 2 * n);
        }
        if (!disjoint(sp, k)) return ZERO_ERR_OVERLAP;
    }
    *plan = p;
    return ZERO_OK;
}

int plan_begin(zero_plan* p, void* stream) {
    NvtxRange range("zero_plan_begin");
    if (p == nullptr || p->state < 1) return ZERO_ERR_ARG;
    if (cudaMemsetAsync(p->workspace, 0, kGradOffset, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return ZERO_ERR_CUDA;
    if (p->policy != nullptr || p->current_set != nullptr) {
        PolicyTable table{};
        zero_adam_hparams hp = p->hp;
        for (int32_t i = 0; i < p->policy_t_count; ++i) {
            hp.step = p->policy_t_first + i;
            const Scalars si = make_scalars(&hp, p->N, p->loss_scale);
            table.step_size[i] = si.step_size;
            table.sbc2[i] = si.sbc2;
        }
        const Scalars base = make_scalars(&p->hp, p->N, p->loss_scale);
        zero_step_prologue_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
            static_cast<const zero_device_policy*>(p->policy),
            reinterpret_cast<Ctrl*>(p->workspace), base, table, p->policy_t_first,
            p->policy_t_count, static_cast<double>(p->N) * micro_batches_of(&p->hp),
            static_cast<const int32_t*>(p->current_set));
        g_launches.fetch_add(1, std::memory_order_relaxed);
        if (cudaGetLastError() != cudaSuccess) return ZERO_ERR_CUDA;
    }
    p->cursor = 0;
    p->micro_batch = 0;
    p->rows_used = 0;
    p->row_width = 0;
    p->shared_slots_used = 0;
    p->state = 2;
    return ZERO_OK;
}

int plan_bucket(zero_plan* p, int64_t begin, int64_t end, const void* const* bucket_grads,
                void* stream) {
    NvtxRange range("zero_plan_bucket");
    if (p == nullptr || p->state != 2) return ZERO_ERR_ARG;
    if (begin != p->cursor || end <= begin || end > p->psi_pad ||
        (end % ZERO_BUCKET_ALIGN != 0 && end != p->psi_pad))
        return ZERO_ERR_ARG;
    StepArgs a = base_args(p);
    if (bucket_grads != nullptr) {
        Span written[6];
        const int nw = written_spans(p, written);
        const uintptr_t bytes = static_cast<uintptr_t>(end - begin) * grad_elem_bytes(p->grad_dtype);
        for (int i = 0; i < p->N; ++i) {
            if (bucket_grads[i] == nullptr) return ZERO_ERR_ARG;
            if (!aligned(bucket_grads[i], ZERO_ALIGN_BYTES)) return ZERO_ERR_ALIGN;
            const Span g{reinterpret_cast<uintptr_t>(bucket_grads[i]),
                         reinterpret_cast<uintptr_t>(bucket_grads[i]) + bytes, false};
            for (int k = 0; k < nw; ++k)
                if (overlaps(g, written[k])) return ZERO_ERR_OVERLAP;
            a.grads[i] = bucket_grads[i];
        }
        a.gbase = begin;
        a.grad_lo = begin;   // a staging slot holds this bucket only
        a.grad_hi = end;
    } else {
        for (int i = 0; i < p->N; ++i)
            if (p->grads[i] == nullptr) return ZERO_ERR_ARG;
    }
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return ZERO_ERR_CUDA;
    const bool bf16 = p->grad_dtype == ZERO_GRAD_BF16;
    const int32_t k = micro_batches_of(&p->hp);
    if (p->smem_staging < ZERO_STAGING_REGISTERS || p->smem_staging > ZERO_STAGING_TMA_TEST_STALL)
        return ZERO_ERR_ARG;
    StepKernel fn;
    Shape shape;
    if (k == 1 && !p->two_pass && p->smem_staging != ZERO_STAGING_REGISTERS) {
        fn = pick<StagedK>(p->N, bf16);
        if (!staged_shape(fn, device, p->N, bf16, a, shape)) return ZERO_ERR_ARG;
        // the plan's own gradient buffers once per pass (at its first bucket),
        // a bucket's own pointers every time
        if (bucket_grads != nullptr || begin == 0)
            for (int i = 0; i < p->N; ++i)
                if (!device_memory(a.grads[i])) return ZERO_ERR_ARG;
        if (begin == 0 && bucket_grads != nullptr)
            for (int i = 0; i < p->N; ++i)
                if (p->grads[i] != nullptr && !device_memory(p->grads[i])) return ZERO_ERR_ARG;
        if (begin == 0 &&
            (!device_memory(p->src_master) || !device_memory(p->src_m) || !device_memory(p->src_v)))
            return ZERO_ERR_ARG;
        // with ping-pong sets the copies may read either set
        if (begin == 0 && p->current_set != nullptr &&
            (!device_memory(p->dst_master) || !device_memory(p->dst_m) || !device_memory(p->dst_v)))
            return ZERO_ERR_ARG;
        a.test_stall = p->smem_staging == ZERO_STAGING_TMA_TEST_STALL ? 1 : 0;
    } else if (k > 1 && p->micro_batch == k - 1 && !p->two_pass) {
        // the last micro-batch of a step with no second pass: accumulate and
        // update in one pass, without writing the accumulator back
        fn = pick<FusedAccK>(p->N, bf16);
    } else if (k > 1) {
        fn = pick<AccumK>(p->N, bf16);
        a.acc_first = p->micro_batch == 0 ? 1 : 0;
        a.acc_last = p->micro_batch == k - 1 ? 1 : 0;
    } else {
        fn = p->two_pass ? pick<ReduceK>(p->N, bf16) : pick<FusedK>(p->N, bf16);
    }
    // Overlap with the previous bucket only when that launch is the one right
    // before this on the stream.  The caller promises that by setting
    // overlap_buckets (zero_step does).  A bucket read from a staging slot
    // follows the wait for that slot's copy, so that caller leaves the flag at
    // 0.  The first bucket of a pass (begin == 0) never overlaps: when
    // accumulating it reads what the previous micro-batch wrote.
    const bool overlap = p->overlap_buckets != 0 && begin > 0;
    // the launches' norm partials: rows of their own while the workspace has
    // rows left; the accumulate passes before the last micro-batch have none
    const RowArea ra = row_area(p);
    RowSource rs;
    rs.rows = ra.rows;
    rs.carry = ra.carry;
    rs.capacity = p->row_capacity;
    rs.used = &p->rows_used;
    rs.width = &p->row_width;
    rs.shared = &p->shared_slots_used;
    rs.mode_without_row = (k > 1 && p->micro_batch < k - 1) ? kNoPartial : kSharedSlot;
    if (!launch_range(fn, device, a, begin, end, static_cast<cudaStream_t>(stream), overlap, shape,
                      end == p->psi_pad ? debug_test_overrun() : 0, &rs))
        return ZERO_ERR_CUDA;
    p->cursor = end;
    // accumulating: a micro-batch that covered the vector hands over to the
    // next, whose first bucket starts at 0 again.  That first bucket is never
    // overlapped (begin == 0), because it reads what this micro-batch wrote.
    if (p->cursor == p->psi_pad && p->micro_batch < k - 1) {
        p->micro_batch += 1;
        p->cursor = 0;
    }
    return ZERO_OK;
}

int plan_end(zero_plan* p, zero_step_result* result, void* stream_handle) {
    NvtxRange range("zero_plan_end");
    if (p == nullptr || p->state != 2 || p->cursor != p->psi_pad ||
        p->micro_batch != micro_batches_of(&p->hp) - 1)
        return ZERO_ERR_ARG;
    zero_step_result* result_dev = nullptr;
    if (result != nullptr) {
        cudaPointerAttributes attr;
        if (cudaPointerGetAttributes(&attr, result) != cudaSuccess || attr.devicePointer == nullptr) {
            cudaGetLastError();  // clear the error that query may leave behind
            return ZERO_ERR_ARG;
        }
        result_dev = static_cast<zero_step_result*>(attr.devicePointer);
    }
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return ZERO_ERR_CUDA;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_handle);
    StepArgs a = base_args(p);
    Ctrl* ctrl = a.ctrl;
    if (result_dev == nullptr) result_dev = &ctrl->result;

    {
        // A programmatic dependent of whatever kernel precedes it on the stream
        // (normally the last bucket's last launch); it waits for that grid to
        // complete before it reads anything.
        const RowArea ra = row_area(p);
        const int32_t n_rows = p->rows_used;
        const double* last_row = n_rows > 0 ? ra.rows + static_cast<int64_t>(n_rows - 1) * kMaxGrid
                                            : nullptr;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1);
        cfg.blockDim = dim3(kFinalizeThreads);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, zero_finalize_kernel, ctrl, static_cast<const double*>(a.partials),
                               p->shared_slots_used, last_row, n_rows > 0 ? p->row_width : 0,
                               static_cast<const double*>(n_rows >= 2 ? ra.carry : nullptr),
                               p->hp.max_grad_norm, static_cast<int>(p->hp.skip_on_overflow),
                               result_dev, static_cast<zero_device_policy*>(p->policy),
                               static_cast<int32_t*>(p->current_set)) != cudaSuccess)
            return ZERO_ERR_CUDA;
    }
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (cudaGetLastError() != cudaSuccess) return ZERO_ERR_CUDA;

    if (p->two_pass) {
        // the first update launch waits for the finalize kernel in stream order
        if (!launch_range(zero_update_kernel, device, a, 0, p->psi_pad, stream, false, Shape{},
                          debug_test_overrun()))
            return ZERO_ERR_CUDA;
    } else if (!p->in_place && p->current_set == nullptr &&
               (p->hp.skip_on_overflow || p->policy != nullptr ||
                p->smem_staging != ZERO_STAGING_REGISTERS || kDebugBuild)) {
        // a skipped step (overflow, a t outside the policy's window, a timed-out
        // staged wait, or in a debug build an access the checks skipped) must
        // leave dst equal to src.  With ping-pong sets the current set stays
        // current instead, and nothing is copied.
        a.begin = 0;
        a.n8 = p->psi_pad / kVec + debug_test_overrun();
        if (!launch(zero_restore_kernel, device, a, stream)) return ZERO_ERR_CUDA;
    }
    p->state = 1;

    if (result == nullptr) {
        zero_step_result host;
        if (cudaMemcpyAsync(&host, &ctrl->result, sizeof host, cudaMemcpyDeviceToHost, stream) !=
                cudaSuccess ||
            cudaStreamSynchronize(stream) != cudaSuccess)
            return ZERO_ERR_CUDA;
        return host.status;
    }
    return ZERO_OK;
}

// zero_step and zero_step_into: one plan, walked bucket by bucket.
int run_step(const void* const* grads, int32_t grad_dtype, const float* src_master,
             const float* src_m, const float* src_v, const uint16_t* src_w, float* dst_master,
             float* dst_m, float* dst_v, uint16_t* dst_w, int64_t psi_pad, int32_t N,
             const zero_adam_hparams* hp, float loss_scale, void* workspace,
             size_t workspace_bytes_given, zero_step_result* result, void* stream) {
    NvtxRange range("zero_step");
    if (hp != nullptr && micro_batches_of(hp) > 1) return ZERO_ERR_ARG;  // one batch only
    zero_plan plan;
    int rc = plan_init(&plan, grads, grad_dtype, src_master, src_m, src_v, src_w, dst_master, dst_m,
                       dst_v, dst_w, psi_pad, N, hp, loss_scale, workspace, workspace_bytes_given,
                       false);
    if (rc != ZERO_OK) return rc;
    plan.overlap_buckets = 1;  // the buckets below are launched back to back
    if ((rc = plan_begin(&plan, stream)) != ZERO_OK) return rc;
    const int64_t bucket = hp->bucket_elems > 0 ? hp->bucket_elems : psi_pad;
    for (int64_t b0 = 0; b0 < psi_pad; b0 += bucket) {
        const int64_t b1 = (psi_pad - b0 > bucket) ? b0 + bucket : psi_pad;
        if ((rc = plan_bucket(&plan, b0, b1, nullptr, stream)) != ZERO_OK) return rc;
    }
    return plan_end(&plan, result, stream);
}

}  // namespace

extern "C" size_t zero_workspace_bytes(int64_t psi_pad, const zero_adam_hparams* hp,
                                       int32_t in_place) {
    if (psi_pad < 0 || hp == nullptr) return 0;
    return align256(workspace_bytes(psi_pad, hp, in_place != 0)) +
           rows_area_bytes(launches_per_pass(psi_pad, hp));
}

extern "C" int zero_step(const void* const* grads, int32_t grad_dtype, float* master, float* m,
                         float* v, uint16_t* w_bf16, int64_t psi_pad, int32_t N,
                         const zero_adam_hparams* hp, float loss_scale, void* workspace,
                         size_t workspace_bytes_given, zero_step_result* result, void* stream) {
    if (master == nullptr && psi_pad > 0) return ZERO_ERR_ARG;
    return run_step(grads, grad_dtype, master, m, v, w_bf16, master, m, v, w_bf16, psi_pad, N, hp,
                    loss_scale, workspace, workspace_bytes_given, result, stream);
}

extern "C" int zero_step_into(const void* const* grads, int32_t grad_dtype,
                              const float* src_master, const float* src_m, const float* src_v,
                              const uint16_t* src_w_bf16, float* dst_master, float* dst_m,
                              float* dst_v, uint16_t* dst_w_bf16, int64_t psi_pad, int32_t N,
                              const zero_adam_hparams* hp, float loss_scale, void* workspace,
                              size_t workspace_bytes_given, zero_step_result* result,
                              void* stream) {
    if (psi_pad > 0 && (src_master == nullptr || dst_master == nullptr)) return ZERO_ERR_ARG;
    if (psi_pad > 0 && static_cast<const void*>(src_master) == static_cast<const void*>(dst_master))
        return ZERO_ERR_OVERLAP;
    return run_step(grads, grad_dtype, src_master, src_m, src_v, src_w_bf16, dst_master, dst_m,
                    dst_v, dst_w_bf16, psi_pad, N, hp, loss_scale, workspace,
                    workspace_bytes_given, result, stream);
}

extern "C" int zero_plan_init(zero_plan* plan, const void* const* grads, int32_t grad_dtype,
                              const float* src_master, const float* src_m, const float* src_v,
                              const uint16_t* src_w_bf16, float* dst_master, float* dst_m,
                              float* dst_v, uint16_t* dst_w_bf16, int64_t psi_pad, int32_t N,
                              const zero_adam_hparams* hp, float loss_scale, void* workspace,
                              size_t workspace_bytes_given) {
    if (psi_pad > 0 && (src_master == nullptr || dst_master == nullptr)) return ZERO_ERR_ARG;
    return plan_init(plan, grads, grad_dtype, src_master, src_m, src_v, src_w_bf16, dst_master,
                     dst_m, dst_v, dst_w_bf16, psi_pad, N, hp, loss_scale, workspace,
                     workspace_bytes_given, true);
}

extern "C" int zero_plan_init_ex(zero_plan* plan, const void* const* grads, int32_t grad_dtype,
                                 const float* src_master, const float* src_m, const float* src_v,
                                 const uint16_t* src_w_bf16, float* dst_master, float* dst_m,
                                 float* dst_v, uint16_t* dst_w_bf16, int64_t psi_pad, int32_t N,
                                 const zero_adam_hparams* hp, float loss_scale, void* workspace,
                                 size_t workspace_bytes_given, float* grad_accum) {
    if (psi_pad > 0 && (src_master == nullptr || dst_master == nullptr)) return ZERO_ERR_ARG;
    return plan_init(plan, grads, grad_dtype, src_master, src_m, src_v, src_w_bf16, dst_master,
                     dst_m, dst_v, dst_w_bf16, psi_pad, N, hp, loss_scale, workspace,
                     workspace_bytes_given, true, grad_accum);
}

extern "C" int zero_plan_set_device_policy(zero_plan* plan, zero_device_policy* policy,
                                           int64_t t_first, int32_t t_count) {
    if (plan == nullptr || plan->state != 1 || policy == nullptr || t_first < 1 || t_count < 1 ||
        t_count > ZERO_POLICY_WINDOW || !aligned(policy, 8))
        return ZERO_ERR_ARG;
    // An in-place one-pass step cannot leave its state alone once it has run,
    // so a window miss must be caught before: only the plan's kernels check
    // it, and they all do.  The policy must be device-addressable.
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, policy) != cudaSuccess || attr.devicePointer == nullptr) {
        cudaGetLastError();
        return ZERO_ERR_ARG;
    }
    plan->policy = attr.devicePointer;
    plan->policy_t_first = t_first;
    plan->policy_t_count = t_count;
    return ZERO_OK;
}

extern "C" int zero_plan_set_pingpong(zero_plan* plan, int32_t* current_set) {
    if (plan == nullptr || plan->state != 1 || current_set == nullptr || !aligned(current_set, 4))
        return ZERO_ERR_ARG;
    // Both sets are read and written, so the step must be out of place, the
    // src set complete, and every buffer of both sets disjoint from the rest.
    if (plan->in_place) return ZERO_ERR_ARG;
    if (plan->psi_pad > 0) {
        if (plan->src_w_bf16 == nullptr) return ZERO_ERR_ARG;
        const uintptr_t n = static_cast<uintptr_t>(plan->psi_pad);
        Span sp[ZERO_MAX_RANKS + 12];
        int k = written_spans(plan, sp);
        auto add = [&](const void* ptr, uintptr_t bytes, bool written) {
            if (ptr != nullptr)
                sp[k++] = Span{reinterpret_cast<uintptr_t>(ptr),
                               reinterpret_cast<uintptr_t>(ptr) + bytes, written};
        };
        add(plan->src_master, 4 * n, true);
        add(plan->src_m, 4 * n, true);
        add(plan->src_v, 4 * n, true);
        add(plan->src_w_bf16, 2 * n, true);
        for (int i = 0; i < plan->N; ++i) add(plan->grads[i], n * grad_elem_bytes(plan->grad_dtype), false);
        if (!disjoint(sp, k)) return ZERO_ERR_OVERLAP;
    }
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, current_set) != cudaSuccess ||
        attr.devicePointer == nullptr) {
        cudaGetLastError();
        return ZERO_ERR_ARG;
    }
    plan->current_set = attr.devicePointer;
    return ZERO_OK;
}

extern "C" int zero_plan_begin(zero_plan* plan, void* stream) { return plan_begin(plan, stream); }

extern "C" int zero_plan_bucket(zero_plan* plan, int64_t begin, int64_t end,
                                const void* const* bucket_grads, void* stream) {
    return plan_bucket(plan, begin, end, bucket_grads, stream);
}

extern "C" int zero_plan_end(zero_plan* plan, zero_step_result* result, void* stream) {
    return plan_end(plan, result, stream);
}

namespace zero_internal {
std::atomic<uint64_t> g_launches{0};
}  // namespace zero_internal

extern "C" uint64_t zero_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" int64_t zero_debug_bounds_violations(void) {
#ifdef ZERO_DEBUG
    if (cudaDeviceSynchronize() != cudaSuccess) return -1;
    unsigned long long n = 0;
    const unsigned long long zero = 0;
    if (cudaMemcpyFromSymbol(&n, g_step_bounds_violations, sizeof n) != cudaSuccess ||
        cudaMemcpyToSymbol(g_step_bounds_violations, &zero, sizeof zero) != cudaSuccess)
        return -1;
    const int64_t g = zero_internal::gather_bounds_violations_take();
    return g < 0 ? -1 : static_cast<int64_t>(n) + g;
#else
    return -1;
#endif
}

// ------------------------------------------------------------------ no-allocation entry point
//
// For callers that cannot allocate device memory: zero_step with its
// workspace in a fixed array defined here.  The array lives in every GPU that
// loads this library until the process exits.  Host code must not pass the
// array's name to a kernel.  On the host that name stands for a host-side
// copy, so the address a kernel may use is looked up per device below.

static __device__ __align__(256) unsigned char g_noalloc_scratch[ZERO_NOALLOC_SCRATCH_BYTES];
static_assert(ZERO_NOALLOC_SCRATCH_BYTES == kGradOffset + 4 * ZERO_NOALLOC_MAX_TWO_PASS_ELEMS,
              "header size of the no-allocation scratch");

namespace {

constexpr int kMaxDevices = 256;

// Device address of g_noalloc_scratch on the current device.  It is looked
// up on the first call per device, with that device current, and then
// cached.  Returns nullptr if the lookup fails.
void* noalloc_scratch(int device) {
    static std::mutex mu;
    static void* addr[kMaxDevices] = {};
    if (device < 0 || device >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[device] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();  // leave no error behind for the caller's next call
            return nullptr;
        }
        addr[device] = p;
    }
    return addr[device];
}

}  // namespace

extern "C" int zero_step_noalloc(const void* const* grads, int32_t grad_dtype, float* master,
                                 float* m, float* v, uint16_t* w_bf16, int64_t psi_pad, int32_t N,
                                 const zero_adam_hparams* hp, float loss_scale,
                                 zero_step_result* result, void* stream) {
    // zero_step's own argument and alignment checks come first, on the host.
    // Run without a workspace, a call whose arguments pass them all stops at
    // the workspace check; only then is the size held against the array.
    if (master == nullptr && psi_pad > 0) return ZERO_ERR_ARG;
    if (hp == nullptr || micro_batches_of(hp) > 1) return ZERO_ERR_ARG;
    {
        zero_plan probe;
        const int rc = plan_init(&probe, grads, grad_dtype, master, m, v, w_bf16, master, m, v,
                                 w_bf16, psi_pad, N, hp, loss_scale, nullptr, 0, false);
        if (rc != ZERO_ERR_WORKSPACE) return rc;
    }
    if (workspace_bytes(psi_pad, hp, true) > ZERO_NOALLOC_SCRATCH_BYTES) return ZERO_ERR_TOO_LARGE;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return ZERO_ERR_CUDA;
    void* scratch = noalloc_scratch(device);
    if (scratch == nullptr) return ZERO_ERR_CUDA;
    return zero_step(grads, grad_dtype, master, m, v, w_bf16, psi_pad, N, hp, loss_scale, scratch,
                     ZERO_NOALLOC_SCRATCH_BYTES, result, stream);
}
