// zero_common.cuh -- what the kernel files of libzero_gb300.so share: launch
// shapes, the launch counter, occupancy queries, programmatic dependent
// launch and NVTX ranges.  Internal to the library.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>

#include <nvtx3/nvToolsExt.h>

namespace zero_internal {
// Kernels this library has launched in this process (zero_launch_count).
extern std::atomic<uint64_t> g_launches __attribute__((visibility("hidden")));
// Debug build: out-of-range accesses the gather kernels skipped on the current
// device since the last call, read and reset (-1 on a CUDA error).
__attribute__((visibility("hidden"))) int64_t gather_bounds_violations_take();
}  // namespace zero_internal

namespace {

using zero_internal::g_launches;

constexpr int kThreads = 256;             // threads per CTA of the streaming kernels
constexpr int kVec = 8;                   // elements per thread per group (16 B of BF16)

// NVTX range around a host entry point, so that profilers show which step,
// bucket or gather enqueued the kernels that follow it.  Without a profiler
// attached this costs a check of one pointer.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

// Programmatic dependent launch.  Consecutive bucket launches of one step
// touch disjoint elements, so launch k+1 may start streaming while launch k
// drains.  Every CTA allows the next launch to be scheduled as soon as it
// starts.  The one write that needs ordering (the CTA's norm slot) waits for
// the previous grid to complete.  The next grid's CTAs can only be scheduled
// once every CTA of this grid is resident, so that wait always ends.
__device__ __forceinline__ void allow_next_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// CTAs per SM for a kernel on a device with the given dynamic shared memory,
// measured once and cached.
inline int resident_ctas(const void* fn, int device, int threads, size_t smem = 0) {
    static std::mutex mu;
    static std::map<std::tuple<const void*, int, size_t>, int> cache;
    std::lock_guard<std::mutex> lock(mu);
    auto key = std::make_tuple(fn, device, smem);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess || n < 1)
        n = 1;
    cache[key] = n;
    return n;
}

inline int sm_count(int device) {
    static std::mutex mu;
    static std::map<int, int> cache;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(device);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n < 1)
        n = 1;
    cache[device] = n;
    return n;
}

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
