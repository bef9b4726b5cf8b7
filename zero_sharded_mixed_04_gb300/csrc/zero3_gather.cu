// zero3_gather.cu -- ZeRO-3 per-layer gather of the working weights on one
// GB300 (sm_103a).
//
// Under ZeRO-3 each rank keeps only its 1/N shard of the BF16 working weights;
// before a layer runs, its full view is all-gathered into temporary memory and
// released after use (lecture deck "RC-T2", slide b2 and note N47; topic page
// "Putting the training ledger onto multiple devices", section "one full
// ZeRO-3 computation").
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>

#include "zero_common.cuh"
#include "zero_gb300.h"

// ------------------------------------------------------------------ ZeRO-3 layer gather
//
// The full view of a layer, assembled from the owners' BF16 shards: the
// all-gather before a layer runs under ZeRO-3.  Pure data movement: 2 B read
// and 2 B written per element.

namespace {

struct GatherArgs {
    const uint16_t* shards[ZERO_MAX_RANKS];
    uint16_t* view;
    int64_t shard;  // elements per shard (a multiple of kVec)
    int64_t begin;  // first element of the range in the full view
    int64_t n;      // elements in the range
    // The range cut at shard boundaries (vector path): segment s copies
    // seg_len[s] elements from shard seg_shard[s] at seg_src[s] to the view at
    // seg_dst[s].  At most one segment per shard.
    int64_t seg_src[ZERO_MAX_RANKS];
    int64_t seg_dst[ZERO_MAX_RANKS];
    int64_t seg_len[ZERO_MAX_RANKS];
    int32_t seg_shard[ZERO_MAX_RANKS];
    int32_t segments;
    int32_t wait_previous;  // 0 under ZERO3_GATHER_OVERLAP_PREVIOUS
    int32_t N;              // shards
};

// Debug build (-DZERO_DEBUG): each segment (vector path) or element (element
// path) is checked against the shard it reads and the view it writes before
// it is copied; one outside them is skipped and counted.
#ifdef ZERO_DEBUG
__device__ unsigned long long g_gather_bounds_violations;
__device__ __forceinline__ bool gather_ok(bool ok) {
    if (!ok) atomicAdd(&g_gather_bounds_violations, 1ull);
    return ok;
}
#else
__device__ __forceinline__ bool gather_ok(bool) { return true; }
#endif

// 16-byte vectors in flight per thread, and CTAs of kThreads per SM at most.
// Measured as CUDA-graph replays of the two-view pass: 2 and 6 gave 0.090 ms
// per GPT-2-small pass and 0.666 ms per pass of twenty 50M-element layers,
// against 0.097 and 0.671 ms with 4 vectors and every resident CTA (6 per SM);
// 1, 4 and 8 vectors with 2 to 8 CTAs per SM were no better.
constexpr int kGatherUnroll = 2;
constexpr int kGatherCtasPerSm = 6;

// The gathers are launched as programmatic dependents of whatever precedes
// them on the stream, so their CTAs are scheduled while that kernel drains.
// Unless the caller declared that kernel independent of this gather
// (ZERO3_GATHER_OVERLAP_PREVIOUS), every thread waits for it to complete
// before its first access, which keeps the plain stream order.
__device__ __forceinline__ void gather_prologue(const GatherArgs& g) {
    allow_next_launch();
    if (g.wait_previous) grid_dependency_wait();
}

// begin is a multiple of kVec, so every segment is a whole number of 8-element
// groups on both sides; the last segment may end with n % 8 single elements.
__global__ void __launch_bounds__(kThreads) zero3_gather_vec_kernel(const __grid_constant__ GatherArgs g) {
    gather_prologue(g);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    for (int s = 0; s < g.segments; ++s) {
        if (!gather_ok(g.seg_shard[s] >= 0 && g.seg_shard[s] < g.N && g.seg_src[s] >= 0 &&
                       g.seg_dst[s] >= 0 && g.seg_len[s] >= 0 &&
                       g.seg_src[s] + g.seg_len[s] <= g.shard &&
                       g.seg_dst[s] + g.seg_len[s] <= g.n))
            continue;
        const uint4* src = reinterpret_cast<const uint4*>(g.shards[g.seg_shard[s]] + g.seg_src[s]);
        uint4* dst = reinterpret_cast<uint4*>(g.view + g.seg_dst[s]);
        const int64_t n8 = g.seg_len[s] / kVec;
        int64_t q = tid;
        for (; q + (kGatherUnroll - 1) * stride < n8; q += kGatherUnroll * stride) {
            uint4 x[kGatherUnroll];
#pragma unroll
            for (int u = 0; u < kGatherUnroll; ++u) x[u] = __ldcs(src + q + u * stride);
#pragma unroll
            for (int u = 0; u < kGatherUnroll; ++u) __stcs(dst + q + u * stride, x[u]);
        }
        for (; q < n8; q += stride) __stcs(dst + q, __ldcs(src + q));
        const int64_t tail = g.seg_len[s] - n8 * kVec;  // only the last segment has one
        if (tid < tail) {
            const int64_t i = n8 * kVec + tid;
            g.view[g.seg_dst[s] + i] = g.shards[g.seg_shard[s]][g.seg_src[s] + i];
        }
    }
}

// Any begin: element by element (a layer that starts at an odd offset).
__global__ void __launch_bounds__(kThreads) zero3_gather_elem_kernel(const __grid_constant__ GatherArgs g) {
    gather_prologue(g);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < g.n; i += stride) {
        const int64_t j = g.begin + i;
        const int64_t r = j / g.shard;
        if (!gather_ok(r >= 0 && r < g.N)) continue;
        g.view[i] = g.shards[r][j - r * g.shard];
    }
}

}  // namespace

extern "C" int zero3_gather(const uint16_t* const* shards, int32_t N, int64_t shard, int64_t begin,
                            int64_t end, uint16_t* view, uint32_t flags, void* stream) {
    NvtxRange range("zero3_gather");
    if (shards == nullptr || N < 1 || N > ZERO_MAX_RANKS || shard < 0 || shard % kVec != 0 ||
        shard > ZERO_MAX_ELEMS / N || begin < 0 || end < begin ||
        end > static_cast<int64_t>(N) * shard ||
        (flags & ~ZERO3_GATHER_OVERLAP_PREVIOUS) != 0)
        return ZERO_ERR_ARG;
    const int64_t n = end - begin;
    if (n == 0) return ZERO_OK;
    if (view == nullptr) return ZERO_ERR_ARG;
    if (!aligned(view, ZERO_ALIGN_BYTES)) return ZERO_ERR_ALIGN;
    GatherArgs g{};
    const uintptr_t vlo = reinterpret_cast<uintptr_t>(view), vhi = vlo + 2 * static_cast<uintptr_t>(n);
    for (int i = 0; i < N; ++i) {
        if (shards[i] == nullptr) return ZERO_ERR_ARG;
        if (!aligned(shards[i], ZERO_ALIGN_BYTES)) return ZERO_ERR_ALIGN;
        const uintptr_t lo = reinterpret_cast<uintptr_t>(shards[i]);
        const uintptr_t hi = lo + 2 * static_cast<uintptr_t>(shard);
        if (lo < vhi && vlo < hi) return ZERO_ERR_OVERLAP;
        g.shards[i] = shards[i];
    }
    g.view = view;
    g.N = N;
    g.shard = shard;
    g.begin = begin;
    g.n = n;
    g.wait_previous = (flags & ZERO3_GATHER_OVERLAP_PREVIOUS) ? 0 : 1;
    // cut [begin, end) at shard boundaries
    g.segments = 0;
    for (int64_t at = begin; at < end;) {
        const int64_t r = at / shard;
        const int64_t stop = (end < (r + 1) * shard) ? end : (r + 1) * shard;
        g.seg_shard[g.segments] = static_cast<int32_t>(r);
        g.seg_src[g.segments] = at - r * shard;
        g.seg_dst[g.segments] = at - begin;
        g.seg_len[g.segments] = stop - at;
        ++g.segments;
        at = stop;
    }
#ifdef ZERO_DEBUG
    // Debug builds only, to test the checks: ZERO_DEBUG_TEST_OVERRUN=g makes the
    // last segment g 8-element groups longer than the range, which the
    // kernel's check must skip.
    if (const char* v = std::getenv("ZERO_DEBUG_TEST_OVERRUN")) {
        const long long x = std::atoll(v);
        g.seg_len[g.segments - 1] += 8 * (x < 0 ? 0 : (x > 1024 ? 1024 : x));
    }
#endif
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return ZERO_ERR_CUDA;
    const bool vec = begin % kVec == 0;
    const void* fn = vec ? reinterpret_cast<const void*>(zero3_gather_vec_kernel)
                         : reinterpret_cast<const void*>(zero3_gather_elem_kernel);
    const int64_t units = vec ? (n + kVec * kGatherUnroll - 1) / (kVec * kGatherUnroll) : n;
    const int64_t full = static_cast<int64_t>(sm_count(device)) * resident_ctas(fn, device, kThreads);
    int64_t grid = (units + kThreads - 1) / kThreads;
    if (grid > full) grid = full;
    const int64_t cap = static_cast<int64_t>(kGatherCtasPerSm) * sm_count(device);
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t err = vec ? cudaLaunchKernelEx(&cfg, zero3_gather_vec_kernel, g)
                                : cudaLaunchKernelEx(&cfg, zero3_gather_elem_kernel, g);
    if (err != cudaSuccess) return ZERO_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cudaGetLastError() == cudaSuccess ? ZERO_OK : ZERO_ERR_CUDA;
}


int64_t zero_internal::gather_bounds_violations_take() {
#ifdef ZERO_DEBUG
    unsigned long long n = 0;
    const unsigned long long zero = 0;
    if (cudaMemcpyFromSymbol(&n, g_gather_bounds_violations, sizeof n) != cudaSuccess ||
        cudaMemcpyToSymbol(g_gather_bounds_violations, &zero, sizeof zero) != cudaSuccess)
        return -1;
    return static_cast<int64_t>(n);
#else
    return 0;
#endif
}
