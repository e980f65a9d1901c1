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
#include "ptx.cuh"

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
    griddep_launch_dependents();     // the GEMM launched next may start its set-up
    griddep_wait();                  // (no-op: this kernel is launched in the ordinary way)
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
// lo = bf16(x - hi) (x - hi is exact in fp32), |e| <= 2^-16 |x|.  Each thread
// takes four consecutive columns of a row: one 16-byte load and three 8-byte
// stores when the row's addresses allow, element by element otherwise.
// Consecutive threads take consecutive groups, so loads and stores are
// contiguous across a warp.  Index = 32-bit unsigned when the group count
// allows (the division per group dominates the index arithmetic).
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

template <typename Index>
__global__ void __launch_bounds__(256) split_kernel(const SplitArgs a)
{
    griddep_launch_dependents();     // the GEMM launched next may start its set-up
    griddep_wait();                  // (no-op: this kernel is launched in the ordinary way)
    const Index gpr = (Index)((a.cols + 3) / 4), total = (Index)a.rows * gpr;
    const bool vec = ((reinterpret_cast<uintptr_t>(a.src) & 15u) == 0) && (a.ld_src % 4 == 0) &&
                     ((reinterpret_cast<uintptr_t>(a.dst) & 7u) == 0) && (a.ld_dst % 4 == 0) &&
                     (!a.k_along_cols || a.cols % 4 == 0);
    for (Index i = (Index)blockIdx.x * 256 + threadIdx.x; i < total; i += (Index)gridDim.x * 256) {
        const Index r = i / gpr;
        const long long c = (long long)(i - r * gpr) * 4;
        const float *src = a.src + (long long)r * a.ld_src + c;
        const int n = (int)min(4LL, a.cols - c);
        float x[4];
        if (vec && n == 4) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(src));
            x[0] = v.x, x[1] = v.y, x[2] = v.z, x[3] = v.w;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) x[j] = j < n ? __ldg(src + j) : 0.0f;
        }
        float hi[4], lo[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            hi[j] = __bfloat162float(__float2bfloat16_rn(x[j]));
            lo[j] = x[j] - hi[j];
        }
        const uint2 part[2] = {make_uint2(pack_bf16x2(hi[0], hi[1]), pack_bf16x2(hi[2], hi[3])),
                               make_uint2(pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]))};
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const long long off = a.k_along_cols ? (long long)r * a.ld_dst + j * a.cols + c
                                                 : (j * a.rows + (long long)r) * a.ld_dst + c;
            const uint2 v = part[a.parts[j]];
            if (vec && n == 4) {
                *reinterpret_cast<uint2 *>(a.dst + off) = v;
            } else {
                const uint16_t e[4] = {(uint16_t)(v.x & 0xffffu), (uint16_t)(v.x >> 16), (uint16_t)(v.y & 0xffffu),
                                       (uint16_t)(v.y >> 16)};
                for (int q = 0; q < n; ++q) a.dst[off + q] = e[q];
            }
        }
    }
}

// int8 -> bf16 or f16 (every int8 value is exact in both).  Each thread takes
// 16 consecutive columns of a row: one 16-byte load and two 16-byte stores
// when the row's addresses allow (the destination rows are 64-element
// padded and 256-byte aligned), element by element otherwise.
template <typename Index>
__global__ void __launch_bounds__(256) widen_kernel(const WidenArgs a)
{
    griddep_launch_dependents();     // launched as a programmatic dependent (see launch_dependent)
    griddep_wait();
    const Index gpr = (Index)((a.cols + 15) / 16), total = (Index)a.rows * gpr;
    const bool vec_src = ((reinterpret_cast<uintptr_t>(a.src) & 15u) == 0) && (a.ld_src % 16 == 0);
    for (Index i = (Index)blockIdx.x * 256 + threadIdx.x; i < total; i += (Index)gridDim.x * 256) {
        const Index r = i / gpr;
        const long long c = (long long)(i - r * gpr) * 16;
        const int8_t *src = a.src + (long long)r * a.ld_src + c;
        uint16_t *dst = a.dst + (long long)r * a.ld_dst + c;
        const int n = (int)min(16LL, a.cols - c);
        int8_t b[16];
        if (vec_src && n == 16) {
            const int4 v = __ldg(reinterpret_cast<const int4 *>(src));
            *reinterpret_cast<int4 *>(b) = v;
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) b[j] = j < n ? __ldg(src + j) : (int8_t)0;
        }
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float x0 = (float)b[2 * j], x1 = (float)b[2 * j + 1];
            if (a.to_f16) {
                const __half2 h = __floats2half2_rn(x0, x1);
                w[j] = *reinterpret_cast<const uint32_t *>(&h);
            } else {
                w[j] = pack_bf16x2(x0, x1);
            }
        }
        // the destination row is padded to a multiple of 64 elements: a
        // 16-column group never straddles its end, so whole stores are safe
        // (columns past `cols` land in the padding, which nothing reads)
        *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4 *>(dst + 8) = make_uint4(w[4], w[5], w[6], w[7]);
    }
}

}  // namespace

cudaError_t launch_widen(const WidenArgs &a, cudaStream_t st)
{
    if (a.rows < 1 || a.cols < 1 || (a.ld_dst % 64) || (reinterpret_cast<uintptr_t>(a.dst) & 255u))
        return cudaErrorInvalidValue;
    const long long total = a.rows * ((a.cols + 15) / 16);
    const long long grid = std::min<long long>((total + 255) / 256, 152LL * 16);
    if (total + (long long)grid * 256 < (1LL << 31))
        return launch_dependent(widen_kernel<uint32_t>, dim3((unsigned)grid), dim3(256), 0, st, 1u, a);
    return launch_dependent(widen_kernel<unsigned long long>, dim3((unsigned)grid), dim3(256), 0, st, 1u, a);
}

cudaError_t launch_split(const SplitArgs &a, cudaStream_t st)
{
    if (a.rows < 1 || a.cols < 1) return cudaErrorInvalidValue;
    const long long total = a.rows * ((a.cols + 3) / 4);
    const long long grid = std::min<long long>((total + 255) / 256, 152LL * 16);
    // an ordinary launch (as a dependent: relaxed fp32 4096^3 ~2 us slower a
    // step, its CTAs placed beside the previous GEMM's); the widening pass
    // gains from one (int8 4096^3: 164.2 against 166.3 us)
    if (total + (long long)grid * 256 < (1LL << 31))
        split_kernel<uint32_t><<<(unsigned)grid, 256, 0, st>>>(a);
    else
        split_kernel<unsigned long long><<<(unsigned)grid, 256, 0, st>>>(a);
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
    // an ordinary launch: as a dependent of the GEMM before it, its many
    // small CTAs would be placed beside that GEMM's and crowd the SMs (the
    // 64-problem ragged batch: 720.8 us a step against 710)
    if (narrow)
        pack_kernel<uint32_t><<<(unsigned)blocks, PACK_THREADS, 0, st>>>(pb);
    else
        pack_kernel<unsigned long long><<<(unsigned)blocks, PACK_THREADS, 0, st>>>(pb);
    return cudaGetLastError();
}

}  // namespace tc
