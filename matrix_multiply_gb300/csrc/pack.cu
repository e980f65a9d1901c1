// Operand preparation: repacking of inputs that TMA cannot read in place,
// and the bf16 copies of the relaxed-fp32 and int8 paths.
//
// Repacking: a TMA tensor copy needs a 16-byte aligned base address and row strides
// that are multiples of 16 bytes.  A contiguous f16/bf16 matrix with an odd
// row length (the ragged shapes of the tessl architecture.md "Edge-Slice
// Support" discussion) breaks the second rule.  Such an operand is copied
// once, in the same layout, into a workspace whose rows are padded to a
// multiple of 64 elements (128 bytes, so every TMA box row starts on a
// cache-line boundary); the tensor-core kernel then reads the copy.  The
// padding is never read: the TMA descriptor keeps the logical extent and
// fills out-of-bounds elements with zeros.
//
// One launch repacks every operand of a call (a whole group of problems):
// the CTAs are split between the operands by a prefix table.
#include "internal.h"

#include <cuda_bf16.h>

#include <algorithm>

namespace tc {
namespace {

constexpr int PACK_THREADS = 256;
constexpr int PACK_ITEMS = 8;      // 16-byte output chunks per thread (loads in flight)

__device__ __forceinline__ uint32_t fsr(uint32_t lo, uint32_t hi, uint32_t sh) { return __funnelshift_r(lo, hi, sh); }

// The 16 bytes at byte offset `off` (even, 0..14) of the 32-byte window a|b.
__device__ __forceinline__ uint4 window16(const uint4 &a, const uint4 &b, uint32_t off)
{
    const uint32_t sh = (off & 2u) * 8u;
    uint4 o;
    switch (off >> 2) {
    case 0: o = make_uint4(fsr(a.x, a.y, sh), fsr(a.y, a.z, sh), fsr(a.z, a.w, sh), fsr(a.w, b.x, sh)); break;
    case 1: o = make_uint4(fsr(a.y, a.z, sh), fsr(a.z, a.w, sh), fsr(a.w, b.x, sh), fsr(b.x, b.y, sh)); break;
    case 2: o = make_uint4(fsr(a.z, a.w, sh), fsr(a.w, b.x, sh), fsr(b.x, b.y, sh), fsr(b.y, b.z, sh)); break;
    default: o = make_uint4(fsr(a.w, b.x, sh), fsr(b.x, b.y, sh), fsr(b.y, b.z, sh), fsr(b.z, b.w, sh)); break;
    }
    return o;
}

// Each thread moves PACK_ITEMS chunks of 8 elements; consecutive threads
// take consecutive chunks of a row, so loads and stores are contiguous
// across a warp.  A source chunk that is not 16-byte aligned is read as the
// one or two aligned 16-byte words that hold its valid elements (each word
// read holds at least one of them) and shifted into place.  The 16-byte
// store may write past the row's last column into the row padding, which
// nothing reads.  Index = 32-bit unsigned when every copy has fewer than
// 2^31 chunks (the divisions dominate the instruction count), else 64-bit.
template <typename Index>
__global__ void __launch_bounds__(PACK_THREADS) pack_kernel(const __grid_constant__ PackBatch pb)
{
    // the copy this CTA works on: the last e with block_begin[e] <= blockIdx.x
    int lo = 0, hi = pb.count - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pb.block_begin[mid] <= (long long)blockIdx.x)
            lo = mid;
        else
            hi = mid - 1;
    }
    const PackArgs &p = pb.seg[lo];
    const Index chunks = (Index)((p.cols + 7) / 8);
    const Index rows = (Index)p.rows;
    const Index per_entry = rows * chunks;
    const Index items = per_entry * (Index)p.batch;
    Index it = (Index)((long long)blockIdx.x - pb.block_begin[lo]) * (PACK_THREADS * PACK_ITEMS) + (Index)threadIdx.x;
    if (it >= items) return;

    // (entry, row, chunk) of the first item, then stepped by PACK_THREADS
    // chunks per item without further divisions
    Index b = 0, rem = it;
    if (p.batch > 1) {
        b = it / per_entry;
        rem = it - b * per_entry;
    }
    Index r = rem / chunks, ch = rem - r * chunks;
    const Index dr = PACK_THREADS / chunks, dc = PACK_THREADS - dr * chunks;

    uint4 q0[PACK_ITEMS], q1[PACK_ITEMS];
    uint32_t off[PACK_ITEMS];
    uint16_t *dst[PACK_ITEMS];
#pragma unroll
    for (int k = 0; k < PACK_ITEMS; ++k) {
        dst[k] = nullptr;
        if (it < items) {
            const Index c = ch * 8;
            const uint16_t *s = p.src + (long long)b * p.stride_src + (long long)r * p.ld_src + c;
            const int valid = (int)min((long long)8, p.cols - (long long)c);
            const uintptr_t addr = reinterpret_cast<uintptr_t>(s);
            off[k] = (uint32_t)(addr & 15u);
            const uint4 *w = reinterpret_cast<const uint4 *>(addr - off[k]);
            q0[k] = __ldg(w);
            q1[k] = (off[k] + 2u * (uint32_t)valid > 16u) ? __ldg(w + 1) : make_uint4(0u, 0u, 0u, 0u);
            dst[k] = p.dst + (long long)b * p.stride_dst + (long long)r * p.ld_dst + c;
        }
        it += PACK_THREADS;
        r += dr;
        ch += dc;
        if (ch >= chunks) {
            ch -= chunks;
            ++r;
        }
        if (r >= rows) {     // into a later batch entry (rows * chunks items each)
            const Index q = r / rows;
            b += q;
            r -= q * rows;
        }
    }
#pragma unroll
    for (int k = 0; k < PACK_ITEMS; ++k)
        if (dst[k]) *reinterpret_cast<uint4 *>(dst[k]) = window16(q0[k], q1[k], off[k]);
}

// Relaxed fp32 (split into bf16 parts): x = hi + lo + e with hi = bf16(x),
// lo = bf16(x - hi) (x - hi is exact in fp32), |e| <= 2^-16 |x|.  One thread
// per element; consecutive threads take consecutive columns, so the fp32
// loads and the three bf16 stores are contiguous across a warp.
__global__ void __launch_bounds__(256) split_kernel(const SplitArgs a)
{
    const long long total = a.rows * a.cols;
    for (long long i = (long long)blockIdx.x * 256 + threadIdx.x; i < total; i += (long long)gridDim.x * 256) {
        const long long r = i / a.cols, c = i - r * a.cols;
        const float x = __ldg(a.src + r * a.ld_src + c);
        const __nv_bfloat16 hi = __float2bfloat16_rn(x);
        const __nv_bfloat16 lo = __float2bfloat16_rn(x - __bfloat162float(hi));
        const uint16_t part[2] = {__bfloat16_as_ushort(hi), __bfloat16_as_ushort(lo)};
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const long long off = a.k_along_cols ? r * a.ld_dst + j * a.cols + c : (j * a.rows + r) * a.ld_dst + c;
            a.dst[off] = part[a.parts[j]];
        }
    }
}

// int8 -> bf16 (every int8 value is exact in bf16), four consecutive
// columns per thread: four byte loads, one 8-byte store when the row has
// all four.
__global__ void __launch_bounds__(256) widen_kernel(const WidenArgs a)
{
    const long long groups = (a.cols + 3) / 4, total = a.rows * groups;
    for (long long i = (long long)blockIdx.x * 256 + threadIdx.x; i < total; i += (long long)gridDim.x * 256) {
        const long long r = i / groups, c = (i - r * groups) * 4;
        const int8_t *src = a.src + r * a.ld_src + c;
        uint16_t *dst = a.dst + r * a.ld_dst + c;
        const int n = (int)min(4LL, a.cols - c);
        uint16_t h[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float x = j < n ? (float)__ldg(src + j) : 0.0f;
            h[j] = a.to_f16 ? __half_as_ushort(__float2half_rn(x)) : __bfloat16_as_ushort(__float2bfloat16_rn(x));
        }
        if (n == 4) {
            *reinterpret_cast<uint2 *>(dst) = make_uint2(h[0] | (uint32_t)h[1] << 16, h[2] | (uint32_t)h[3] << 16);
        } else {
            for (int j = 0; j < n; ++j) dst[j] = h[j];
        }
    }
}

}  // namespace

cudaError_t launch_widen(const WidenArgs &a, cudaStream_t st)
{
    if (a.rows < 1 || a.cols < 1 || (a.ld_dst % 64) || (reinterpret_cast<uintptr_t>(a.dst) & 255u))
        return cudaErrorInvalidValue;
    const long long total = a.rows * ((a.cols + 3) / 4);
    const long long grid = std::min<long long>((total + 255) / 256, 152LL * 16);
    widen_kernel<<<(unsigned)grid, 256, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_split(const SplitArgs &a, cudaStream_t st)
{
    if (a.rows < 1 || a.cols < 1) return cudaErrorInvalidValue;
    const long long total = a.rows * a.cols;
    const long long grid = std::min<long long>((total + 255) / 256, 152LL * 16);
    split_kernel<<<(unsigned)grid, 256, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_pack(PackBatch &pb, cudaStream_t st)
{
    if (pb.count < 1 || pb.count > PACK_MAX) return cudaErrorInvalidValue;
    long long blocks = 0;
    bool narrow = true;
    for (int i = 0; i < pb.count; ++i) {
        const PackArgs &p = pb.seg[i];
        if ((reinterpret_cast<uintptr_t>(p.dst) & 15u) || (p.ld_dst % 8) || (p.stride_dst % 8))
            return cudaErrorInvalidValue;
        const long long items = p.rows * ((p.cols + 7) / 8) * p.batch;
        // 32-bit indices: every item index, plus one CTA's span, below 2^31
        if (items + PACK_THREADS * PACK_ITEMS >= (1LL << 31)) narrow = false;
        pb.block_begin[i] = blocks;
        blocks += (items + PACK_THREADS * PACK_ITEMS - 1) / (PACK_THREADS * PACK_ITEMS);
    }
    pb.block_begin[pb.count] = blocks;
    if (blocks < 1 || blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    if (narrow)
        pack_kernel<uint32_t><<<(unsigned)blocks, PACK_THREADS, 0, st>>>(pb);
    else
        pack_kernel<unsigned long long><<<(unsigned)blocks, PACK_THREADS, 0, st>>>(pb);
    return cudaGetLastError();
}

}  // namespace tc
