// zero_elem.cuh -- the per-element arithmetic of the ZeRO update step, shared
// by the kernel files of libzero_gb300.so: the step's FP32 scalars, the owner's
// Adam update of one element, BF16 widening and rounding, and the 16-byte
// vector loads and stores of 8-element groups.  Internal to the library.
//
// Every operator is an explicit round-to-nearest intrinsic, so no multiply-add
// is ever contracted and each element is rounded operator by operator, in the
// order the oracle takes.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "zero_common.cuh"

namespace {

// Per-step FP32 scalars, each rounded once from FP64.
struct Scalars {
    float inv;        // 1 / (N * loss_scale)
    float b1, omb1;   // beta1, 1 - beta1
    float b2, omb2;   // beta2, 1 - beta2
    float eps;
    float step_size;  // lr / (1 - beta1^t)
    float sbc2;       // sqrt(1 - beta2^t)
    float decay;      // 1 - lr * weight_decay
    int use_decay;
};

// ------------------------------------------------------------------ element math

__device__ __forceinline__ bool is_nonfinite(float x) {
    return (__float_as_uint(x) & 0x7f800000u) == 0x7f800000u;
}

// Sum of squares of K values, in FP64, without the overflow (|x| >= 2^64) or
// underflow (|x| < 2^-75) that squaring in FP32 meets.  The values are
// multiplied by one power of two, 2^-e, where 2^e is the binade of their
// largest magnitude (clamped so that 2^-e stays a normal FP32 number).  The
// scaled squares are summed in FP32 in order, by multiply-add, and the sum is
// multiplied by 2^(2e) in FP64, exactly.  Multiplying by a power of two
// commutes with rounding in the normal range, so wherever the unscaled squares
// neither overflow nor underflow this gives the bits of summing them unscaled.
// A NaN or an infinity reaches the result through its own square.
template <int K>
__device__ __forceinline__ double sum_of_squares_scaled(const float (&x)[K]) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < K; ++i) amax = fmaxf(amax, fabsf(x[i]));
    int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 127;
    e = e < -126 ? -126 : (e > 126 ? 126 : e);
    const float s = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    float sq = 0.0f;
#pragma unroll
    for (int i = 0; i < K; ++i) {
        const float y = __fmul_rn(x[i], s);
        sq = fmaf(y, y, sq);
    }
    return static_cast<double>(sq) *
           __longlong_as_double(static_cast<long long>(1023 + 2 * e) << 52);
}

// The same sum, unscaled where that is as accurate.  A finite FP32 sum means
// no partial sum overflowed.  The multiply-add forms each square exactly, so
// the only coarse rounding a small value can meet is that of a partial sum in
// the subnormal range, off by at most 2^-150.  Against a final sum of at least
// 2^-40, whose half unit in the last place is 2^-65 or more, that gives the
// scaled sum's bits unless the exact sum lies within 2^-150 of a rounding
// boundary, and one unit in the last place at worst.  Other groups, rare, take
// the scaled sum.  Either way the result is a fixed function of the values.
__device__ __forceinline__ bool squares_in_range(float sq) {
    return sq >= 0x1p-40f && sq < INFINITY;
}

template <int K>
__device__ __forceinline__ double sum_of_squares(const float (&x)[K]) {
    float sq = 0.0f;
#pragma unroll
    for (int i = 0; i < K; ++i) sq = fmaf(x[i], x[i], sq);
    if (squares_in_range(sq)) return static_cast<double>(sq);
    return sum_of_squares_scaled(x);
}

// BF16 is the top half of an FP32 word; element 2q of a 16-byte vector is the
// low half of 32-bit word q.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // round to nearest, ties to even
    return *reinterpret_cast<uint32_t*>(&h);
}

// Owner update of one element: AdamW with bias correction, every operator
// rounded to FP32 on its own.
__device__ __forceinline__ void adam_element(float g, float& p, float& m, float& v,
                                             const Scalars& s) {
    if (s.use_decay) p = __fmul_rn(p, s.decay);
    m = __fadd_rn(__fmul_rn(s.b1, m), __fmul_rn(s.omb1, g));
    v = __fadd_rn(__fmul_rn(s.b2, v), __fmul_rn(s.omb2, __fmul_rn(g, g)));
    const float den = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), s.sbc2), s.eps);
    p = __fsub_rn(p, __fmul_rn(s.step_size, __fdiv_rn(m, den)));
}

// ------------------------------------------------------------------ vector loads
//
// Global memory only: __ldcs / __stcs are the global-space cache-streaming
// forms (ld.global.cs / st.global.cs).  Shared-memory stages are read with
// lds_u2 / lds_f4 below.

template <bool kBF16>
struct GradVec;

template <>
struct GradVec<true> {
    uint4 r;
    __device__ __forceinline__ void load(const void* base, int64_t j) {
        r = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + j));
    }
    __device__ __forceinline__ void add_to(float (&g)[kVec]) const {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            g[2 * q] = __fadd_rn(g[2 * q], bf16_lo(w[q]));
            g[2 * q + 1] = __fadd_rn(g[2 * q + 1], bf16_hi(w[q]));
        }
    }
};

template <>
struct GradVec<false> {
    float4 a, b;
    __device__ __forceinline__ void load(const void* base, int64_t j) {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + j);
        a = __ldcs(p);
        b = __ldcs(p + 1);
    }
    __device__ __forceinline__ void add_to(float (&g)[kVec]) const {
        g[0] = __fadd_rn(g[0], a.x); g[1] = __fadd_rn(g[1], a.y);
        g[2] = __fadd_rn(g[2], a.z); g[3] = __fadd_rn(g[3], a.w);
        g[4] = __fadd_rn(g[4], b.x); g[5] = __fadd_rn(g[5], b.y);
        g[6] = __fadd_rn(g[6], b.z); g[7] = __fadd_rn(g[7], b.w);
    }
};

__device__ __forceinline__ void load8(const float* base, int64_t j, float (&x)[kVec]) {
    const float4* p = reinterpret_cast<const float4*>(base + j);
    const float4 u = __ldcs(p), w = __ldcs(p + 1);
    x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
    x[4] = w.x; x[5] = w.y; x[6] = w.z; x[7] = w.w;
}

__device__ __forceinline__ void store8(float* base, int64_t j, const float (&x)[kVec]) {
    float4* p = reinterpret_cast<float4*>(base + j);
    __stcs(p, make_float4(x[0], x[1], x[2], x[3]));
    __stcs(p + 1, make_float4(x[4], x[5], x[6], x[7]));
}

__device__ __forceinline__ void store_w8(uint16_t* base, int64_t j, const float (&p)[kVec]) {
    const uint4 packed = make_uint4(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]),
                                    pack_bf16x2(p[4], p[5]), pack_bf16x2(p[6], p[7]));
    __stcs(reinterpret_cast<uint4*>(base + j), packed);
}

}  // namespace
