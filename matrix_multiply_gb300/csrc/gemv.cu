// Skinny products: Out = alpha * (X W^T) (* scale per W row) + beta * Out_old
// for X with at most 16 rows.  This is the decode shape of the pages: the
// tensorcore gemm.md "Kernel variants" table's M <= 4 GEMV (fp16 out) and
// the Foundry metal.md "Custom Compute Kernels" int8-weight products
// (fm_matvec_q8, fm_sgemm_q8: each weight row scaled by its own factor).
//
// Every weight byte is read once, so the product is bound by HBM, not by
// arithmetic.  Both kernels are built around the weight stream:
//   * a warp owns 16 rows of W; each lane streams 16-byte pieces of two rows
//     (rows g and g + 8 of the warp's 16, g = lane / 4), four lanes covering
//     64 contiguous bytes of a row per step;
//   * the 8 warps of a CTA interleave along K over the same rows; the CTA
//     adds their partial sums in warp order through shared memory.
// The row-range kernel (aligned rows, enough rows for every CTA): one
// persistent grid of two CTAs per SM, each owning an equal range of W rows
// (so no CTA waits on a partial last wave), each warp streaming its pieces
// of W and of X through a ring of cp.async slots in shared memory several
// steps ahead of its multiplies.  The cluster kernel (unaligned rows, or too
// few rows to give every SM some): one CTA per 16-row block and K slice,
// the slices of a block forming a cluster of up to 8 CTAs whose sums are
// added in rank order through distributed shared memory.  Fixed orders
// everywhere, so the result is deterministic.
// The multiply-adds run on mma.sync m16n8k16 (fp32 accumulation) with W as
// the 16-row operand and X^T as the 8-column operand: the K order inside one
// lane's piece is remapped the same way for both operands, so the fragments
// come straight from the loaded registers.  On CUDA cores the same work
// would need a type conversion and M fused multiply-adds per weight, which
// for int8 weights at M = 4 comes close to the FFMA peak at HBM speed.
// int8 weights are widened exactly in registers (byte permutes into the
// mantissa of a half, then one subtraction).
#include "elem.cuh"
#include "internal.h"
#include "ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

namespace tc {
namespace {

constexpr int GV_WARPS = 8;
constexpr int GV_UNROLL = 4;      // cluster kernel: steps in flight per warp

// 16 bytes global -> shared without passing through registers (cp.async,
// L2 only); src_bytes = 0 writes zeros
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
// the same through L1 (X is read by every CTA of the SM: L1 keeps it)
__device__ __forceinline__ void cp_async16_l1(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// D(16x8, f32) += A(16x16) * B(16x8), A row-major, B column-major
template <bool BF16>
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    if constexpr (BF16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}

// 16 bytes of the weight stream: read once, so kept out of L1
__device__ __forceinline__ uint4 ld_stream16(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 16 bytes of X, re-read by every CTA: through L1
__device__ __forceinline__ uint4 ld_reuse16(const void *p) { return __ldg(reinterpret_cast<const uint4 *>(p)); }

// Elements [k, k + E) of a row of 2-byte or 1-byte elements as 16 bytes,
// zero beyond `kend`; element by element (an unaligned row or the K tail).
template <int ESZ>
__device__ __forceinline__ uint4 ld_partial(const uint8_t *row, long long k, long long kend)
{
    constexpr int E = 16 / ESZ;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int j = 0; j < E; ++j) {
        if (k + j < kend) {
            uint32_t v = ESZ == 2 ? (uint32_t)reinterpret_cast<const uint16_t *>(row)[k + j]
                                  : (uint32_t)(uint8_t)row[k + j];
            w[(j * ESZ) / 4] |= v << (8 * ((j * ESZ) % 4));
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Four int8 values (one 32-bit word) -> two half2 / bf16x2 words, exactly.
// half: 0x6400 | (b + 128) is the half 1024 + b + 128; subtracting 1152
// leaves b.  bf16 has too few mantissa bits for that, so each byte goes
// through fp32 the same way (0x4B000000 | (b + 128) is 2^23 + b + 128) and
// the exact small integers are packed to bf16.
template <bool BF16>
__device__ __forceinline__ void widen4(uint32_t v, uint32_t &lo, uint32_t &hi)
{
    const uint32_t u = v ^ 0x80808080u;          // b + 128 in every byte
    if constexpr (!BF16) {
        const uint32_t p0 = __byte_perm(u, 0x64646464u, 0x4140u);
        const uint32_t p1 = __byte_perm(u, 0x64646464u, 0x4342u);
        const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6480u));   // 1152
        __half2 h0 = __hsub2(*reinterpret_cast<const __half2 *>(&p0), bias);
        __half2 h1 = __hsub2(*reinterpret_cast<const __half2 *>(&p1), bias);
        lo = *reinterpret_cast<uint32_t *>(&h0);
        hi = *reinterpret_cast<uint32_t *>(&h1);
    } else {
        float f[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            f[j] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440u | (uint32_t)j)) - 8388736.0f;
        __nv_bfloat162 b0 = __floats2bfloat162_rn(f[0], f[1]);
        __nv_bfloat162 b1 = __floats2bfloat162_rn(f[2], f[3]);
        lo = *reinterpret_cast<uint32_t *>(&b0);
        hi = *reinterpret_cast<uint32_t *>(&b1);
    }
}

// One slab of the product: lane (g, t) holds K values [k, k + WK) of W rows
// g and g + 8 (w0, w1) and of X rows nt * 8 + g (xv); MMA j takes pairs
// 4j..4j+1 as the fragments' columns 2t..2t+1 and pairs 4j+2..4j+3 as
// columns 2t+8..2t+9, for W and X alike.  Every lane of the warp calls it.
template <bool BF16, bool W8, int NT>
__device__ __forceinline__ void slab_mma(float (&acc)[NT][4], const uint4 &w0, const uint4 &w1,
                                         const uint4 (&xv)[NT][W8 ? 2 : 1])
{
    constexpr int WK = W8 ? 16 : 8;
    constexpr int XL = W8 ? 2 : 1;
    uint32_t h0[WK / 2], h1[WK / 2];
    if constexpr (W8) {
        const uint32_t r0[4] = {w0.x, w0.y, w0.z, w0.w};
        const uint32_t r1[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            widen4<BF16>(r0[q], h0[2 * q], h0[2 * q + 1]);
            widen4<BF16>(r1[q], h1[2 * q], h1[2 * q + 1]);
        }
    } else {
        h0[0] = w0.x, h0[1] = w0.y, h0[2] = w0.z, h0[3] = w0.w;
        h1[0] = w1.x, h1[1] = w1.y, h1[2] = w1.z, h1[3] = w1.w;
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        uint32_t x[WK / 2];
#pragma unroll
        for (int q = 0; q < XL; ++q) {
            x[4 * q + 0] = xv[nt][q].x;
            x[4 * q + 1] = xv[nt][q].y;
            x[4 * q + 2] = xv[nt][q].z;
            x[4 * q + 3] = xv[nt][q].w;
        }
#pragma unroll
        for (int j = 0; j < WK / 4; ++j) {
            const uint32_t afrag[4] = {h0[2 * j], h1[2 * j], h0[2 * j + 1], h1[2 * j + 1]};
            mma_16816<BF16>(acc[nt], afrag, x[2 * j], x[2 * j + 1]);
        }
    }
}

// alpha * (v * scale[n]) + beta * C_old, one rounding, for W row n and X row c
__device__ __forceinline__ void gemv_out(const GemvArgs &a, long long n, int c, float v)
{
    if (a.scale) v *= a.scale[n];
    const long long off = (long long)c * a.c_sx + n * a.c_sw;
    v = (a.beta != 0.0f) ? fmaf(a.beta, load_c(a.C, off, a.c_dtype), a.alpha * v) : a.alpha * v;
    store_c1(a.C, off, v, a.c_dtype);
}

// BF16: X (and W unless W8) are bf16, else f16.  W8: W is int8.  NT: n8
// tiles of X rows (1: at most 8 rows, 2: at most 16).
// The cluster kernel: one CTA per (16-row block, K slice), the K slices of a
// block one cluster of a.ksplit CTAs.  Each warp issues the weight loads of
// GV_UNROLL steps before their multiplies; unaligned rows and the K tail
// are read element by element.  Two CTAs per SM (at most 128 registers).
template <bool BF16, bool W8, int NT>
__global__ void __launch_bounds__(GV_WARPS * 32, 2) gemv_kernel(const GemvArgs a)
{
    constexpr int WK = W8 ? 16 : 8;             // weights per 16-byte load
    constexpr int SLAB = 4 * WK;                // K values per warp step (4 lanes per row)
    constexpr int XL = W8 ? 2 : 1;              // 16-byte X loads per weight load
    constexpr int WSZ = W8 ? 1 : 2;
    constexpr int COLS = NT * 8;                // X rows covered
    __shared__ float red[GV_WARPS][16][COLS + 1];
    __shared__ float sums[COLS][16];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int KS = a.ksplit;
    const int rb = blockIdx.x / KS;
    const int kr = blockIdx.x - rb * KS;       // rank in the cluster (consecutive CTAs)
    const long long n0 = (long long)rb * 16;
    const long long K = a.K;
    const long long nslab = (K + SLAB - 1) / SLAB;
    const long long s0 = (long long)kr * nslab / KS, s1 = (long long)(kr + 1) * nslab / KS;
    griddep_launch_dependents();     // a dependent launched next may start its set-up
    griddep_wait();                  // (no-op: this kernel is launched in the ordinary way)

    const uint8_t *W = static_cast<const uint8_t *>(a.W);
    const uint8_t *X = static_cast<const uint8_t *>(a.X);
    const bool r0ok = n0 + g < a.rows_w, r1ok = n0 + g + 8 < a.rows_w;
    const uint8_t *wrow0 = W + (r0ok ? (n0 + g) * a.ldw * WSZ : 0);
    const uint8_t *wrow1 = W + (r1ok ? (n0 + g + 8) * a.ldw * WSZ : 0);
    const uint8_t *xrow[NT];
    bool xok[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        xok[nt] = nt * 8 + g < a.rows_x;
        xrow[nt] = X + (xok[nt] ? (long long)(nt * 8 + g) * a.ldx * 2 : 0);
    }

    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;

    auto load_w = [&](const uint8_t *row, bool ok, long long k) -> uint4 {
        if (!ok) return make_uint4(0u, 0u, 0u, 0u);
        if (a.w_vec && k + WK <= K) return ld_stream16(row + k * WSZ);
        return ld_partial<WSZ>(row, k, K);
    };
    auto load_x = [&](int nt, long long k) -> uint4 {
        if (!xok[nt]) return make_uint4(0u, 0u, 0u, 0u);
        if (a.x_vec && k + 8 <= K) return ld_reuse16(xrow[nt] + k * 2);
        return ld_partial<2>(xrow[nt], k, K);
    };

    // One slab: lane (g, t) holds K values [k, k + WK) of rows g and g + 8
    // (w0, w1) and of X rows g (and 8 + g); MMA j takes pairs 4j..4j+1 as
    // the fragments' columns 2t..2t+1 and pairs 4j+2..4j+3 as columns
    // 2t+8..2t+9, for W and X alike.  X is read as it is needed (it stays in
    // L1).  Every lane of the warp calls it.
    auto mma_slab = [&](const uint4 &w0, const uint4 &w1, long long k) {
        uint4 xv[NT][XL];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int q = 0; q < XL; ++q) xv[nt][q] = load_x(nt, k + 8 * q);
        slab_mma<BF16, W8, NT>(acc, w0, w1, xv);
    };

    for (long long s = s0 + warp; s < s1; s += (long long)GV_WARPS * GV_UNROLL) {
        uint4 wv[GV_UNROLL][2];
#pragma unroll
        for (int u = 0; u < GV_UNROLL; ++u) {
            const long long sl = s + (long long)u * GV_WARPS;     // warp-uniform
            const long long k = sl * SLAB + t * WK;
            if (sl < s1) {
                wv[u][0] = load_w(wrow0, r0ok, k);
                wv[u][1] = load_w(wrow1, r1ok, k);
            } else {
                wv[u][0] = wv[u][1] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int u = 0; u < GV_UNROLL; ++u) {
            const long long sl = s + (long long)u * GV_WARPS;
            if (sl >= s1) break;                                     // warp-uniform
            mma_slab(wv[u][0], wv[u][1], sl * SLAB + t * WK);
        }
    }

    // D fragment: acc[nt][e] is (W row g, X row nt*8 + 2t + e), acc[nt][2 + e]
    // is (W row g + 8, same X row)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        red[warp][g][nt * 8 + 2 * t] = acc[nt][0];
        red[warp][g][nt * 8 + 2 * t + 1] = acc[nt][1];
        red[warp][g + 8][nt * 8 + 2 * t] = acc[nt][2];
        red[warp][g + 8][nt * 8 + 2 * t + 1] = acc[nt][3];
    }
    __syncthreads();
    const int r = threadIdx.x & 15, c = threadIdx.x >> 4;      // W row r, X row c
    float v = 0.0f;
    if (c < COLS) {
#pragma unroll
        for (int w = 0; w < GV_WARPS; ++w) v += red[w][r][c];
    }
    if (KS > 1) {
        // the cluster's K ranges, added in rank order by rank 0
        if (c < COLS) sums[c][r] = v;
        cluster_sync();
        if (kr == 0 && c < COLS) {
            const uint32_t off = smem_u32(&sums[c][r]);
            float part[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (q < KS) part[q] = ld_shared_cluster_f32(mapa_shared(off, (uint32_t)q));
            v = part[0];
#pragma unroll
            for (int q = 1; q < 8; ++q)
                if (q < KS) v += part[q];
        }
    }
    const long long n = n0 + r;
    if (kr == 0 && c < COLS && c < a.rows_x && n < a.rows_w) gemv_out(a, n, c, v);
    if (KS > 1) cluster_sync();      // peers keep their shared memory until rank 0 has read it
}

// ------------------------------------------------------------ row-range kernel
// gridDim.x persistent CTAs; CTA c owns W rows [c N / G, (c + 1) N / G),
// taken 16 at a time.  Warp w streams steps w, w + 8, ... of each 16-row
// block through its own ring of GV_RR_RING bytes: per step and lane one
// slot holds its 16 bytes of rows g and g + 8 and of X rows nt * 8 + g,
// copied with cp.async (bytes past K or past the rows read as zeros; X
// through L1, since every CTA of the SM reads the same X rows) and
// read back by the same lane only, so a lane needs nothing but its own copy
// groups.  The ring runs on across block boundaries; after a block's last
// step the warps' sums are added in warp order and written.
constexpr int GV_RR_RING = 12 * 1024;      // bytes of ring per warp

template <bool W8, int NT>
__host__ __device__ constexpr int rr_slot() { return (2 + NT * (W8 ? 2 : 1)) * 32 * 16; }
template <bool W8, int NT>
__host__ __device__ constexpr int rr_stages() { return GV_RR_RING / rr_slot<W8, NT>(); }

template <bool BF16, bool W8, int NT>
__global__ void __launch_bounds__(GV_WARPS * 32, 2) gemv_rr_kernel(const GemvArgs a)
{
    constexpr int WK = W8 ? 16 : 8;
    constexpr int SLAB = 4 * WK;
    constexpr int XL = W8 ? 2 : 1;
    constexpr int WSZ = W8 ? 1 : 2;
    constexpr int COLS = NT * 8;
    constexpr int SLOT = rr_slot<W8, NT>();
    constexpr int S = rr_stages<W8, NT>();
    static_assert(S >= 3, "ring depth");
    extern __shared__ __align__(16) uint8_t rr_ring[];
    __shared__ float red[GV_WARPS][16][COLS + 1];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const long long K = a.K;
    griddep_launch_dependents();     // launched as a programmatic dependent (see launch_dependent)
    griddep_wait();
    long long r_lo, r_hi;
    if (a.block_rows) {
        const long long nb = ((long long)a.rows_w + 15) / 16;
        r_lo = 16 * ((long long)blockIdx.x * nb / gridDim.x);
        r_hi = min((long long)a.rows_w, 16 * ((long long)(blockIdx.x + 1) * nb / gridDim.x));
    } else {
        r_lo = (long long)blockIdx.x * a.rows_w / gridDim.x;
        r_hi = (long long)(blockIdx.x + 1) * a.rows_w / gridDim.x;
    }
    const int nblk = (int)((r_hi - r_lo + 15) / 16);
    const int nslab = (int)((K + SLAB - 1) / SLAB);
    const int per = warp < nslab ? (nslab - warp + GV_WARPS - 1) / GV_WARPS : 0;   // this warp's steps per block
    const int items = nblk * per;
    const uint8_t *W = static_cast<const uint8_t *>(a.W);
    const uint8_t *X = static_cast<const uint8_t *>(a.X);
    const uint32_t ring = smem_u32(rr_ring) + (uint32_t)(warp * GV_RR_RING + lane * 16);
    // Per-lane copy state for the next item to issue (block ib, step ij of
    // this warp, ring slot is): source pointers advanced by additions, byte
    // counts fixed per block except in the step that reaches past K.
    const long long wrow = a.ldw * WSZ;                 // bytes between W rows
    constexpr int WADV = GV_WARPS * SLAB * WSZ;         // bytes between two steps of a warp (W)
    constexpr int XADV = GV_WARPS * SLAB * 2;           // the same for X
    const int kbase = warp * SLAB + t * WK;             // this lane's first K
    const uint8_t *xbase[NT];
    uint32_t xfull[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const bool ok = nt * 8 + g < a.rows_x;
        xfull[nt] = ok ? 16u : 0u;
        xbase[nt] = ok ? X + ((long long)(nt * 8 + g) * a.ldx + kbase) * 2 : X;
    }
    int ib = 0, ij = 0, is = 0, kq = kbase;
    const uint8_t *wp0 = W, *wp1 = W;
    const uint8_t *xp[NT];
    uint32_t w0full = 0, w1full = 0;
    auto start_block = [&]() {
        const long long n0 = r_lo + 16LL * ib;
        const bool ok0 = n0 + g < r_hi, ok1 = n0 + g + 8 < r_hi;
        w0full = ok0 ? 16u : 0u;
        w1full = ok1 ? 16u : 0u;
        wp0 = ok0 ? W + (n0 + g) * wrow + (long long)kbase * WSZ : W;
        wp1 = ok1 ? W + (n0 + g + 8) * wrow + (long long)kbase * WSZ : W;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) xp[nt] = xbase[nt];
        kq = kbase;
    };
    if (per > 0) start_block();
    auto issue = [&]() {
        const uint32_t slot = ring + (uint32_t)(is * SLOT);
        if ((warp + GV_WARPS * ij + 1) * SLAB <= K) {        // the whole step is inside K (warp-uniform)
            cp_async16(slot, wp0, w0full);
            cp_async16(slot + 512, wp1, w1full);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int q = 0; q < XL; ++q) cp_async16_l1(slot + (2 + nt * XL + q) * 512, xp[nt] + 16 * q, xfull[nt]);
        } else {                                              // the step reaching past K
            const int kw = (int)min(16LL, max(0LL, (K - kq) * WSZ));
            cp_async16(slot, kw ? wp0 : W, w0full ? (uint32_t)kw : 0u);
            cp_async16(slot + 512, kw ? wp1 : W, w1full ? (uint32_t)kw : 0u);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int q = 0; q < XL; ++q) {
                    const int kx = (int)min(16LL, max(0LL, (K - (kq + 8 * q)) * 2));
                    cp_async16_l1(slot + (2 + nt * XL + q) * 512, (kx && xfull[nt]) ? xp[nt] + 16 * q : X,
                                  xfull[nt] ? (uint32_t)kx : 0u);
                }
        }
        if (++is == S) is = 0;
        if (++ij == per) {
            ij = 0;
            ++ib;
            if (ib < nblk) start_block();
        } else {
            wp0 += WADV;
            wp1 += WADV;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) xp[nt] += XADV;
            kq += GV_WARPS * SLAB;
        }
    };

    int issued = 0;
#pragma unroll
    for (int q = 0; q < S - 1; ++q) {
        if (issued < items) {
            issue();
            ++issued;
        }
        cp_async_commit();
    }
    int rs = 0;                                       // ring slot of the item being multiplied
    for (int blk = 0; blk < nblk; ++blk) {
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;
        for (int j = 0; j < per; ++j) {
            if (issued < items) {
                issue();
                ++issued;
            }
            cp_async_commit();
            cp_async_wait<S - 1>();                   // this lane's copies of the current item have landed
            const uint32_t slot = ring + (uint32_t)(rs * SLOT);
            if (++rs == S) rs = 0;
            uint4 w0, w1;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w0.x), "=r"(w0.y), "=r"(w0.z), "=r"(w0.w) : "r"(slot));
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w1.x), "=r"(w1.y), "=r"(w1.z), "=r"(w1.w) : "r"(slot + 512));
            uint4 xv[NT][XL];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int q = 0; q < XL; ++q)
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(xv[nt][q].x), "=r"(xv[nt][q].y), "=r"(xv[nt][q].z), "=r"(xv[nt][q].w)
                                 : "r"(slot + (2 + nt * XL + q) * 512));
            slab_mma<BF16, W8, NT>(acc, w0, w1, xv);
        }
        // D fragment: acc[nt][e] is (W row g, X row nt*8 + 2t + e), acc[nt][2 + e]
        // is (W row g + 8, same X row)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            red[warp][g][nt * 8 + 2 * t] = acc[nt][0];
            red[warp][g][nt * 8 + 2 * t + 1] = acc[nt][1];
            red[warp][g + 8][nt * 8 + 2 * t] = acc[nt][2];
            red[warp][g + 8][nt * 8 + 2 * t + 1] = acc[nt][3];
        }
        __syncthreads();
        const int r = threadIdx.x & 15, c = threadIdx.x >> 4;       // W row r, X row c
        const long long n = r_lo + 16LL * blk + r;
        if (c < COLS && c < a.rows_x && n < r_hi) {
            float v = 0.0f;
#pragma unroll
            for (int w = 0; w < GV_WARPS; ++w) v += red[w][r][c];
            gemv_out(a, n, c, v);
        }
        __syncthreads();
    }
    cp_async_wait<0>();
}

template <bool BF16, bool W8, int NT>
cudaError_t launch_rr(const GemvArgs &a, cudaStream_t st)
{
    constexpr auto kern = gemv_rr_kernel<BF16, W8, NT>;
    constexpr int smem = GV_WARPS * GV_RR_RING;
    static std::atomic<bool> configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev].load(std::memory_order_acquire)) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured[dev].store(true, std::memory_order_release);
    }
    if (a.grid < 1 || a.grid > a.rows_w) return cudaErrorInvalidValue;
    return launch_dependent(kern, dim3((unsigned)a.grid), dim3(GV_WARPS * 32), smem, st, 1u, a);
}

template <bool BF16, bool W8, int NT>
cudaError_t launch_one(const GemvArgs &a, cudaStream_t st)
{
    constexpr auto kern = gemv_kernel<BF16, W8, NT>;
    const long long blocks = ((long long)a.rows_w + 15) / 16 * a.ksplit;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    // an ordinary launch (one small CTA per block and slice: as a dependent,
    // its CTAs would be placed early, crowding the SMs that are idle then)
    if (a.ksplit == 1) {
        kern<<<(unsigned)blocks, GV_WARPS * 32, 0, st>>>(a);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(GV_WARPS * 32, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)a.ksplit;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

cudaError_t launch_gemv(const GemvArgs &a, cudaStream_t st)
{
    if (a.rows_x < 1 || a.rows_x > GEMV_MAX_ROWS || a.rows_w < 1 || a.K < 1) return cudaErrorInvalidValue;
    const int key = (a.x_bf16 ? 4 : 0) | (a.w_i8 ? 2 : 0) | (a.rows_x > 8 ? 1 : 0);
    if (a.rowrange) {
        // 16-byte copies need 16-byte aligned rows of X and W
        if (!a.x_vec || !a.w_vec) return cudaErrorInvalidValue;
        switch (key) {
        case 0: return launch_rr<false, false, 1>(a, st);
        case 1: return launch_rr<false, false, 2>(a, st);
        case 2: return launch_rr<false, true, 1>(a, st);
        case 3: return launch_rr<false, true, 2>(a, st);
        case 4: return launch_rr<true, false, 1>(a, st);
        case 5: return launch_rr<true, false, 2>(a, st);
        case 6: return launch_rr<true, true, 1>(a, st);
        default: return launch_rr<true, true, 2>(a, st);
        }
    }
    if (a.ksplit != 1 && a.ksplit != 2 && a.ksplit != 4 && a.ksplit != 8) return cudaErrorInvalidValue;
    switch (key) {
    case 0: return launch_one<false, false, 1>(a, st);
    case 1: return launch_one<false, false, 2>(a, st);
    case 2: return launch_one<false, true, 1>(a, st);
    case 3: return launch_one<false, true, 2>(a, st);
    case 4: return launch_one<true, false, 1>(a, st);
    case 5: return launch_one<true, false, 2>(a, st);
    case 6: return launch_one<true, true, 1>(a, st);
    default: return launch_one<true, true, 2>(a, st);
    }
}

}  // namespace tc
