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
// x / (1 + exp(-2z)) with the __expf intrinsic: a few instructions, and a
// relative error of about 1e-6 (the intrinsic's error in exp, damped by
// e / (1 + e)).  Large positive z gives x; large negative z overflows exp to
// +inf and gives -0.
__device__ __forceinline__ float gelu_tanh(float x)
{
    const float z = 0.7978845608028654f * fmaf(0.044715f * x, x * x, x);
    return __fdividef(x, 1.0f + __expf(-2.0f * z));
}

}  // namespace tc
