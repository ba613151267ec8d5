// Shared device helpers of the sparse attention kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sfa.h"

namespace sfa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------------------
// Element type traits: 16-bit storage, fp32 arithmetic.

struct F16 {
    using T = __half;
    static __device__ __forceinline__ float to_f(T x) { return __half2float(x); }
    static __device__ __forceinline__ T from_f(float x) { return __float2half_rn(x); }
    // two packed elements (low = first) -> two floats
    static __device__ __forceinline__ float2 unpack2(uint32_t u) {
        __half2 h = *reinterpret_cast<__half2*>(&u);
        return __half22float2(h);
    }
    static __device__ __forceinline__ uint32_t pack2(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
};

struct BF16 {
    using T = __nv_bfloat16;
    static __device__ __forceinline__ float to_f(T x) { return __bfloat162float(x); }
    static __device__ __forceinline__ T from_f(float x) { return __float2bfloat16_rn(x); }
    static __device__ __forceinline__ float2 unpack2(uint32_t u) {
        return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
    }
    static __device__ __forceinline__ uint32_t pack2(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
};

// 8-bit floating point (E4M3 when E5 is false, else E5M2), two elements at
// a time: the first in the low byte.  Packing rounds to nearest even and
// saturates to the largest finite value; unpacking is exact (every E4M3 and
// E5M2 value is an fp16 value).
template <bool E5>
__device__ __forceinline__ uint32_t f8_pack2(float first, float second) {
    uint16_t r;
    if constexpr (E5)
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(second), "f"(first));
    else
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(second), "f"(first));
    return r;
}

template <bool E5>
__device__ __forceinline__ float2 f8_unpack2(uint32_t two) {
    const uint16_t in = (uint16_t)two;
    uint32_t h2;
    if constexpr (E5)
        asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h2) : "h"(in));
    else
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    __half2 h = *reinterpret_cast<__half2*>(&h2);
    return __half22float2(h);
}

// ---------------------------------------------------------------------------
// Asynchronous global -> shared copies (16 bytes per thread, L2 only).

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async_16(void* smem_dst, const void* gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem_dst)),
                 "l"(gmem_src)
                 : "memory");
}

// Zero-fill variant: src_bytes == 0 writes 16 zero bytes and reads nothing.
__device__ __forceinline__ void cp_async_16_zfill(void* smem_dst, const void* gmem_src,
                                                  int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem_dst)),
                 "l"(gmem_src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------
// Warp reductions.

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// exp2 with -inf -> 0 (ex2.approx already maps -inf to +0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// plan()'s logits_soft_cap in log2 units: a logit u = x * log2(e) becomes
// capl2 * tanh(u / capl2) with capl2 = cap * log2(e), i.e. cap * tanh(x / cap)
// scaled to log2 units (tanhf: the accurate library function).
__device__ __forceinline__ float soft_cap_log2(float u, float capl2, float inv_capl2) {
    return capl2 * tanhf(u * inv_capl2);
}

// Rescale factor exp2(m_old - m_new) of an online softmax, defined as 1 when
// both maxima are still -inf (no visible slot yet).
__device__ __forceinline__ float rescale_factor(float m_old, float m_new) {
    return (m_new == -INFINITY) ? 1.0f : fast_exp2(m_old - m_new);
}

}  // namespace sfa
