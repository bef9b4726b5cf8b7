// zero_kernels.cuh -- the device side of the ZeRO update step on one GB300 (sm_103a).
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
//     shared memory with TMA bulk copies, and 12 or 16 warps compute from there.
// The arithmetic uses the explicit round-to-nearest intrinsics, so no
// multiply-add is ever contracted: each element is rounded operator by
// operator.
//
// This header holds the control block and the per-launch arguments, the
// per-element and per-CTA helpers, and every kernel of the step (one-pass
// register and TMA-staged, the two-pass reduce and update, the micro-batch
// accumulation, restore, finalize and the step prologue).  zero_step.cu, the
// only file that includes it, holds the host side.  The profile summaries'
// kernel-code hash covers this file, zero_elem.cuh and zero_common.cuh, so
// that host-side changes leave the DRAM figures they report standing.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

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

// One 8-element group's combined gradient, formed as fused_groups forms it.
template <int NT, bool kBF16, bool kAccIn>
__device__ __forceinline__ void combined_gradient(const StepArgs& a, const Scalars& s, int64_t j,
                                                  float (&g)[kVec]) {
    float acc[kVec];
    if constexpr (kAccIn) load8(a.gws, j, acc);
    combine<NT, kBF16>(a, j, g);
#pragma unroll
    for (int e = 0; e < kVec; ++e) {
        g[e] = __fmul_rn(g[e], s.inv);
        if constexpr (kAccIn) g[e] = __fadd_rn(acc[e], g[e]);
    }
}

// One 8-element group: reduce-scatter + scale + check + Adam + BF16 all-gather.
// kAccIn: the last micro-batch of an accumulated step.  The combined gradient
// is this micro-batch's scaled contribution added to the FP32 accumulator the
// earlier micro-batches left in gws (the same two roundings the accumulate
// kernel makes), and is used at once instead of being written back.
template <int NT, bool kBF16, bool kAccIn, int U>
__device__ __forceinline__ void fused_groups(const StepArgs& a, const Scalars& s, bool sw,
                                             const int64_t (&j)[U], unsigned& bad,
                                             double& sumsq, unsigned& extreme) {
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
        // out of range: the kernel sums this thread's groups again, scaled
        extreme |= squares_in_range(sq) ? 0u : 1u;
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
    unsigned extreme = 0;
    const int64_t q0 = q;
    for (; kPairs && q + stride < n8; q += 2 * stride) {
        const int64_t j[2] = {a.begin + q * kVec, a.begin + (q + stride) * kVec};
        if (!range_ok(a, j[0], kVec, true) || !range_ok(a, j[1], kVec, true)) continue;
        fused_groups<NT, kBF16, kAccIn, 2>(a, s, sw, j, bad, sumsq, extreme);
    }
    for (; !kPairs && q + stride < n8; q += stride) {
        const int64_t j[1] = {a.begin + q * kVec};
        if (!range_ok(a, j[0], kVec, true)) continue;
        fused_groups<NT, kBF16, kAccIn, 1>(a, s, sw, j, bad, sumsq, extreme);
    }
    if (q < n8) {
        const int64_t j[1] = {a.begin + q * kVec};
        if (range_ok(a, j[0], kVec, true))
            fused_groups<NT, kBF16, kAccIn, 1>(a, s, sw, j, bad, sumsq, extreme);
    }
    if (extreme) {
        // The same groups in the same order, their combined gradient formed
        // again from the inputs (which this kernel only reads), summed scaled.
        sumsq = 0.0;
        float g[kVec];
        for (q = q0; kPairs && q + stride < n8; q += 2 * stride) {
            const int64_t j[2] = {a.begin + q * kVec, a.begin + (q + stride) * kVec};
            if (!range_ok(a, j[0], kVec, true) || !range_ok(a, j[1], kVec, true)) continue;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                combined_gradient<NT, kBF16, kAccIn>(a, s, j[u], g);
                sumsq += sum_of_squares(g);
            }
        }
        for (; !kPairs && q + stride < n8; q += stride) {
            if (!range_ok(a, a.begin + q * kVec, kVec, true)) continue;
            combined_gradient<NT, kBF16, kAccIn>(a, s, a.begin + q * kVec, g);
            sumsq += sum_of_squares(g);
        }
        if (q < n8 && range_ok(a, a.begin + q * kVec, kVec, true)) {
            combined_gradient<NT, kBF16, kAccIn>(a, s, a.begin + q * kVec, g);
            sumsq += sum_of_squares(g);
        }
    }
    finish_cta(a, bad, sumsq);
}

// ------------------------------------------------------------------ staged one-pass kernel
//
// The same one-pass step with each tile of T::kTile elements staged in shared
// memory.  One producer thread copies a tile's N gradient chunks and its
// master/m/v chunks from HBM into a stage with TMA bulk copies
// (cp.async.bulk), counted in the stage's "full" mbarrier.  The consumer
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

// The tile, per kernel instance: 2048 elements and 16 consumer warps, or 1536
// and 12 where an element's bytes (N*g + 12) are at most 25, so that three
// CTAs of two stages fit one SM's shared memory instead of two.  Measured
// interleaved on one GPU: GPT-2 small, N = 4 BF16, 0.621 ms per step against
// 0.637 with 2048; ragged 6B, N = 4, 29.12 ms against 29.52; Psi = 1e9, N = 8
// (57 KB stages either way two CTAs) 6.020 against 6.018; 1280 and 10 warps
// (three CTAs for N = 8) 6.034.  A runtime rank count (NT = 0) keeps 2048.
constexpr int staged_tile(int nt, bool bf16) {
    return (nt > 0 && nt * (bf16 ? 2 : 4) + 12 <= 25) ? 1536 : 2048;
}
template <int NT, bool kBF16>
struct Staged {
    static constexpr int kTile = staged_tile(NT, kBF16);
    static constexpr int kWarps = kTile / 128;        // consumer warps: 4 elements a thread
    static constexpr int kConsumers = 32 * kWarps;
    static constexpr int kThreads = kConsumers + 32;  // + the producer warp
    static_assert(kTile % (4 * kConsumers) == 0, "whole 4-element chunks per consumer");
    static_assert(kThreads <= 32 * kMaxWarps, "finish_cta's per-warp slots");
};
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
        const unsigned char* chunk = st + static_cast<size_t>(i) * Staged<NT, kBF16>::kTile * gbytes;
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
    constexpr int kTile = Staged<NT, kBF16>::kTile;
    const unsigned char* state = st + static_cast<size_t>(n) * kTile * gbytes;
    const float4 P = lds_f4(state + e * 4);
    const float4 M = lds_f4(state + (kTile + e) * 4);
    const float4 V = lds_f4(state + (2 * kTile + e) * 4);
    float p[4] = {P.x, P.y, P.z, P.w}, m[4] = {M.x, M.y, M.z, M.w}, v[4] = {V.x, V.y, V.z, V.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float gs = __fmul_rn(g[q], s.inv);
        bad |= is_nonfinite(gs) ? 1u : 0u;
        g[q] = gs;
        adam_element(gs, p[q], m[q], v[q], s);
    }
    sumsq += sum_of_squares(g);
    __stcs(reinterpret_cast<float4*>(out_master(a, sw) + j), make_float4(p[0], p[1], p[2], p[3]));
    __stcs(reinterpret_cast<float4*>(out_m(a, sw) + j), make_float4(m[0], m[1], m[2], m[3]));
    __stcs(reinterpret_cast<float4*>(out_v(a, sw) + j), make_float4(v[0], v[1], v[2], v[3]));
    __stcs(reinterpret_cast<uint2*>(out_w(a, sw) + j),
           make_uint2(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3])));
}

template <int NT, bool kBF16>
__global__ void __launch_bounds__(Staged<NT, kBF16>::kThreads)
    zero_fused_staged_kernel(const __grid_constant__ StepArgs a) {
    allow_next_launch();
    constexpr int kTile = Staged<NT, kBF16>::kTile;
    constexpr int kStagedConsumerWarps = Staged<NT, kBF16>::kWarps;
    constexpr int kStagedConsumers = Staged<NT, kBF16>::kConsumers;
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

// U groups of the first pass of the two-pass form.  The squares are summed
// unscaled; a group whose FP32 sum is out of range sets `extreme`, and the
// kernel then sums this thread's groups again, scaled (sum_of_squares), from
// the combined gradient it wrote.  That keeps the common loop free of a branch.
template <int NT, bool kBF16, int U>
__device__ __forceinline__ void reduce_groups(const StepArgs& a, const Scalars& s,
                                              const int64_t (&j)[U], unsigned& bad,
                                              double& sumsq, unsigned& extreme) {
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
        extreme |= squares_in_range(sq) ? 0u : 1u;
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
    unsigned extreme = 0;
    const int64_t q0 = q;
    for (; q + stride < n8; q += 2 * stride) {
        const int64_t j[2] = {a.begin + q * kVec, a.begin + (q + stride) * kVec};
        if (!range_ok(a, j[0], kVec, true) || !range_ok(a, j[1], kVec, true)) continue;
        reduce_groups<NT, kBF16, 2>(a, s, j, bad, sumsq, extreme);
    }
    if (q < n8) {
        const int64_t j[1] = {a.begin + q * kVec};
        if (range_ok(a, j[0], kVec, true)) reduce_groups<NT, kBF16, 1>(a, s, j, bad, sumsq, extreme);
    }
    if (extreme) {
        // the same groups in the same order, from the values this thread stored
        sumsq = 0.0;
        float g[kVec];
        for (q = q0; q + stride < n8; q += 2 * stride) {
            const int64_t j[2] = {a.begin + q * kVec, a.begin + (q + stride) * kVec};
            if (!range_ok(a, j[0], kVec, true) || !range_ok(a, j[1], kVec, true)) continue;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                load8(a.gws, j[u], g);
                sumsq += sum_of_squares(g);
            }
        }
        if (q < n8 && range_ok(a, a.begin + q * kVec, kVec, true)) {
            load8(a.gws, a.begin + q * kVec, g);
            sumsq += sum_of_squares(g);
        }
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
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
            acc[u][e] = __fadd_rn(acc[u][e], __fmul_rn(g[u][e], s.inv));
            bad |= is_nonfinite(acc[u][e]) ? 1u : 0u;
        }
        if (a.acc_last) sumsq += sum_of_squares(acc[u]);
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
//     window (the launch's `window`), or from the caller's table in memory
//     (`table`: step_size and sbc2 for each t, in pairs), forms the
//     batch-mean factor from the device's loss scale, and leaves them in the
//     control block for the step's kernels.
__global__ void zero_step_prologue_kernel(const zero_device_policy* policy, Ctrl* ctrl,
                                          Scalars base, PolicyTable window, const float* table,
                                          int64_t t_first, int64_t t_count,
                                          double ranks_times_micro, const int32_t* current_set) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    if (current_set != nullptr)
        ctrl->cur = *reinterpret_cast<const volatile int32_t*>(current_set) != 0 ? 1 : 0;
    if (policy == nullptr) return;
    const int64_t idx = policy->t + 1 - t_first;
    Scalars s = base;
    if (idx < 0 || idx >= t_count) {
        ctrl->policy_error = 1;  // every kernel of the step then leaves the state alone
    } else if (table != nullptr) {
        s.step_size = table[2 * idx];
        s.sbc2 = table[2 * idx + 1];
    } else {
        s.step_size = window.step_size[idx];
        s.sbc2 = window.sbc2[idx];
    }
    s.inv = static_cast<float>(1.0 / (ranks_times_micro * static_cast<double>(policy->loss_scale)));
    ctrl->scalars = s;
}

}  // namespace
