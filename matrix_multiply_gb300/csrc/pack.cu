// Operand repacking for inputs that TMA cannot read in place.
//
// A TMA tensor copy needs a 16-byte aligned base address and row strides
// that are multiples of 16 bytes.  A contiguous f16/bf16 matrix with an odd
// row length (the ragged shapes of the tessl architecture.md "Edge-Slice
// Support" discussion) breaks the second rule.  Such an operand is copied
// once, in the same layout, into a workspace whose rows are padded to a
// multiple of 64 elements (128 bytes, so every TMA box row starts on a
// cache-line boundary); the tensor-core kernel then reads the copy.  The
// padding is never read: the TMA descriptor keeps the logical extent and
// fills out-of-bounds elements with zeros.
#include "internal.h"

namespace tc {
namespace {

// One CTA row of 256 threads copies 256 consecutive elements of a row, so
// each warp instruction reads and writes one contiguous 64-byte segment;
// every thread handles four rows per iteration (four loads in flight).
// Only the logical columns are written: TMA never reads the padding.
__global__ void __launch_bounds__(256) pack_kernel(const PackArgs p)
{
    const long long c = (long long)blockIdx.x * 256 + threadIdx.x;
    if (c >= p.cols) return;
    const long long step = (long long)gridDim.y * 4;
    for (int b = 0; b < p.batch; ++b) {
        const uint16_t *src = p.src + b * p.stride_src + c;
        uint16_t *dst = p.dst + b * p.stride_dst + c;
        for (long long r0 = (long long)blockIdx.y * 4; r0 < p.rows; r0 += step) {
            uint16_t v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (r0 + q < p.rows) v[q] = src[(r0 + q) * p.ld_src];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (r0 + q < p.rows) dst[(r0 + q) * p.ld_dst] = v[q];
        }
    }
}

}  // namespace

cudaError_t launch_pack(const PackArgs &p, cudaStream_t st)
{
    const long long gx = (p.cols + 255) / 256;
    const long long rows4 = (p.rows + 3) / 4;
    long long gy = (2048 + gx - 1) / gx;           // about 2048 CTAs in total
    if (gy > rows4) gy = rows4;
    if (gy > 65535) gy = 65535;
    if (gy < 1) gy = 1;
    if (gx > 0x7fffffffLL) return cudaErrorInvalidValue;
    pack_kernel<<<dim3((unsigned)gx, (unsigned)gy, 1), 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace tc
