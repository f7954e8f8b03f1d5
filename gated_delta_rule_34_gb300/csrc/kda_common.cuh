// kda_common.cuh -- small device helpers shared by the KDA kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

// Lower bound of the per-channel log-decay: g = g_min * sigmoid(exp(A) * z)
// with g_min = -5 ("How Kimi K3 is built: 2.8 trillion parameters, linear attention and agents for a million tokens",
// section "Sequence: three KDA to one global MLA").
// The chunked kernels rely on it: across 16 tokens the decay spans at most
// e^80, inside the fp32/bf16 exponent range.
constexpr float kGMin = -5.0f;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// sigmoid from its definition 1 / (1 + e^-x), with CUDA's expf; the result is
// clamped to [g_min, 0] so that rounding can never leave the bound that the
// chunked form depends on.
__device__ __forceinline__ float gate_accurate(float expA, float z) {
    const float x = expA * z;
    const float s = 1.0f / (1.0f + expf(-x));
    return fminf(fmaxf(kGMin * s, kGMin), 0.0f);
}

// Same definition with the fast intrinsics (__expf, __fdividef); used where
// the gate sits on the throughput-critical path of bf16 prefill.
__device__ __forceinline__ float gate_fast(float expA, float z) {
    const float x = expA * z;
    const float s = __fdividef(1.0f, 1.0f + __expf(-x));
    return fminf(fmaxf(kGMin * s, kGMin), 0.0f);
}

// Two fp32 lanes in one 64-bit register (element 0 in the low half) and the
// packed arithmetic on them (fma.rn.f32x2, mul.rn.f32x2): each lane rounds
// exactly like the scalar fmaf / multiply, one instruction for both.
__device__ __forceinline__ uint64_t f2_pack(float x, float y) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
    return x;
}

// Sequence bounds for sequence n: packed (cu != nullptr) or fixed length T.
// Offsets are clamped into [0, T_total] so that malformed cu_seqlens can
// never move an access outside the buffers.
__device__ __forceinline__ void seq_bounds(const int32_t* cu, int n, int64_t T, int64_t T_total,
                                           int64_t& bos, int64_t& eos) {
    if (cu) {
        int64_t b = cu[n], e = cu[n + 1];
        b = b < 0 ? 0 : (b > T_total ? T_total : b);
        e = e < b ? b : (e > T_total ? T_total : e);
        bos = b;
        eos = e;
    } else {
        bos = (int64_t)n * T;
        eos = bos + T;
    }
}

}  // namespace kda
