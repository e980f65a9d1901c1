// Per-element helpers shared by the kernels: loads and stores of C (and of
// the bias) in its dtype with one round-to-nearest-even, and the GeluTanh
// activation of the fused epilogue.
#pragma once
#include "../../include/tcgemm.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace tc {

__device__ __forceinline__ uint32_t pack2(float x, float y, int c_dtype)
{
    if (c_dtype == TC_BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __half2 h = __floats2half2_rn(x, y);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float load_c(const void *C, long long off, int c_dtype)
{
    if (c_dtype == TC_F32) return static_cast<const float *>(C)[off];
    const uint16_t bits = static_cast<const uint16_t *>(C)[off];
    if (c_dtype == TC_BF16) return __bfloat162float(__ushort_as_bfloat16(bits));
    return __half2float(__ushort_as_half(bits));
}

__device__ __forceinline__ void store_c1(void *C, long long off, float v, int c_dtype)
{
    if (c_dtype == TC_F32) {
        static_cast<float *>(C)[off] = v;
    } else if (c_dtype == TC_BF16) {
        static_cast<__nv_bfloat16 *>(C)[off] = __float2bfloat16_rn(v);
    } else {
        static_cast<__half *>(C)[off] = __float2half_rn(v);
    }
}

// Fused epilogue (tessl architecture.md, "Fused Epilogue"): activation(y +
// bias[col]) in fp32 on the value y = alpha * acc + beta * C_old.
// GeluTanh: 0.5 x (1 + tanh(z)), z = sqrt(2/pi) (x + 0.044715 x^3),
// evaluated through the identity 1 + tanh(z) = 2 / (1 + exp(-2z)) as
// x / (1 + 2^u) with u = -2 z log2(e) = x (K1 + K2 x^2): three multiply-adds,
// the PTX approximate base-2 exponential and reciprocal, one add and one
// multiply.  The two approximate instructions run on the SM's special
// function unit (16 results per clock), which bounds the epilogue of a
// large tile; the constants are folded so that the rest is as short as it
// can be.  Relative error about 1e-6 (the exponential's error, damped by
// e / (1 + e)).  Large positive x gives x; large negative x overflows 2^u
// to +inf and gives -0.
__device__ __forceinline__ float gelu_tanh(float x)
{
    constexpr float K1 = -2.0f * 0.7978845608028654f * 1.4426950408889634f;
    constexpr float K2 = K1 * 0.044715f;
    const float u = x * fmaf(K2, x * x, K1);
    float e, r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(u));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
    return x * r;
}

}  // namespace tc
