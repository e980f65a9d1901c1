// Operand repacking for inputs that TMA cannot read in place.
//
// A TMA tensor copy needs a 16-byte aligned base address and row strides
// that are multiples of 16 bytes.  A contiguous f16/bf16 matrix with an odd
// row length (the ragged shapes of the tessl architecture.md "Edge-Slice
// Support" discussion) breaks the second rule.  Such an operand is copied
// once, in the same layout, into a workspace whose rows are padded to a
// multiple of 8 elements; the tensor-core kernel then reads the copy.  The
// padding is never read: the TMA descriptor keeps the logical extent and
// fills out-of-bounds elements with zeros.
#include "internal.h"

namespace tc {
namespace {

__global__ void __launch_bounds__(256) pack_kernel(const PackArgs p)
{
    const long long groups = (p.cols + 7) / 8;           // 8 elements -> one 16-byte store
    const long long per_mat = groups * p.rows;
    const long long total = per_mat * p.batch;
    for (long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x; g < total;
         g += (long long)gridDim.x * blockDim.x) {
        const long long b = g / per_mat;
        const long long rem = g - b * per_mat;
        const long long r = rem / groups;
        const long long c = (rem - r * groups) * 8;
        const uint16_t *s = p.src + b * p.stride_src + r * p.ld_src + c;
        uint16_t v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = (c + i < p.cols) ? s[i] : (uint16_t)0;
        uint4 w;
        w.x = (uint32_t)v[0] | ((uint32_t)v[1] << 16);
        w.y = (uint32_t)v[2] | ((uint32_t)v[3] << 16);
        w.z = (uint32_t)v[4] | ((uint32_t)v[5] << 16);
        w.w = (uint32_t)v[6] | ((uint32_t)v[7] << 16);
        *reinterpret_cast<uint4 *>(p.dst + b * p.stride_dst + r * p.ld_dst + c) = w;
    }
}

}  // namespace

cudaError_t launch_pack(const PackArgs &p, cudaStream_t st)
{
    const long long total = ((p.cols + 7) / 8) * p.rows * p.batch;
    long long blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    pack_kernel<<<(unsigned)blocks, 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace tc
