// Tensor-core GEMM for sm_103a: C = alpha * op(A) @ op(B) + beta * C with
// f16/bf16 operands and an fp32 accumulator held in TMEM for the whole K
// loop.
//
// Prior art on the pages and what became of it here:
//   * tessl architecture.md, "Cooperative Destination Accumulation": keep
//     the accumulator on chip across the whole K reduction and write C once.
//     Here the accumulator lives in TMEM (tcgen05.mma writes it directly),
//     so C traffic does not grow with K.
//   * tessl architecture.md, "Column-Panel Grid Swizzling": bands of tile
//     rows so that B panels are re-read from L2 rather than HBM.  Here a
//     persistent CTA walks a linear tile index that is mapped through bands
//     of `group_m` tile rows.
//   * tessl architecture.md, "Round 2 Evolutions" (accumulate path):
//     C_old is read once in the epilogue, only when beta != 0.
//   * tessl architecture.md, "Round 2 Evolutions" (split-K dW): tall-K,
//     small-MN shapes split K into slices; here the slices are reduced in a
//     fixed order so the result is deterministic.
//   * tensorcore gemm.md, "The 64x64 tile": cooperative loads into on-chip
//     memory per K block.  Here TMA copies 128-byte-swizzled tiles into a
//     multistage shared-memory ring guarded by mbarriers.
//
// CTA layout (192 threads, one CTA per SM, persistent over output tiles):
//   warps 0-3  epilogue: TMEM -> registers -> alpha/beta -> C (warp w owns
//              TMEM lanes 32w..32w+31, i.e. tile rows 32w..32w+31)
//   warp 4     TMA producer (one elected lane)
//   warp 5     MMA issuer (one elected lane)
// Two accumulator buffers in TMEM let the epilogue of tile i overlap the
// main loop of tile i+1.
//
// Every wait is bounded: on expiry the kernel records a status word, raises
// a CTA-wide abort flag, lets in-flight copies and MMAs land, frees TMEM and
// returns.  It never traps.
#include "elem.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "../../include/tcgemm.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <mutex>
#include <type_traits>

namespace tc {
namespace {

struct Watch {
    volatile uint32_t *abort_flag;
    unsigned *status;
    unsigned long long timeout_ns;
};

// status codes written on a timeout: 0x100 | where
enum : unsigned { W_EMPTY = 1, W_FULL = 2, W_TMEM_EMPTY = 3, W_TMEM_FULL = 4 };

__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, const Watch &w, unsigned where)
{
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 15u) == 0) {
            if (*w.abort_flag) return false;
            if (globaltimer_ns() - t0 > w.timeout_ns) {
                *w.abort_flag = 1u;
                if (w.status) {
                    *(volatile unsigned *)w.status = 0x100u | where;
                    __threadfence_system();
                }
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Watch &w, unsigned where)
{
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, w, where);
}

// Abort path only: wait a short, fixed time for an async arrival (a TMA copy
// or an MMA commit) so that nothing lands in shared memory or TMEM after
// the CTA has released them.
__device__ __noinline__ void drain_wait(uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > 200000000ull) return;
    }
}

struct Unit {
    int b, tm, tn;       // batch entry and tile coordinates
    int tile;            // linear tile id over every batch entry
    int s, S;            // K slice of this unit and the tile's slice count
    int kb0, kb1;        // K-block range [kb0, kb1)
    int ufirst;          // unit of slice 0 of this tile
    int p;               // problem of a grouped launch (0 otherwise)
};

// Kernel parameter holding the problem table of a grouped launch; a
// single-problem launch carries an empty stand-in.
struct NoTable {
    int count;
};
template <bool GROUPED>
using TableOf = std::conditional_t<GROUPED, GroupTable, NoTable>;

// Linear tile id -> (batch entry, tile row, tile column): bands of group_m
// tile rows, column-major inside a band.
__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int tiles_per_batch, int group_m,
                                            int &b, int &tm, int &tn)
{
    b = tile / tiles_per_batch;
    const int t = tile - b * tiles_per_batch;
    const int band = group_m * tiles_n;
    const int g = t / band;
    const int first_m = g * group_m;
    const int rows_in_band = min(tiles_m - first_m, group_m);
    const int in_band = t - g * band;
    tm = first_m + in_band % rows_in_band;
    tn = in_band / rows_in_band;
}

// First K block of slice s of S over num_kb blocks: floor(s * num_kb / S),
// in 32-bit arithmetic whenever the product cannot overflow it.
__device__ __forceinline__ int kb_split(int num_kb, int s, int S)
{
    if (num_kb < 65536) return (int)(((unsigned)s * (unsigned)num_kb) / (unsigned)S);
    return (int)(((long long)s * num_kb) / S);
}

__device__ __forceinline__ Unit decode_unit(const MmaArgs &a, int u)
{
    Unit r;
    const int seg0_units = a.seg0_tiles * a.seg0_split;
    if (u < seg0_units) {
        r.tile = u / a.seg0_split;
        r.s = u - r.tile * a.seg0_split;
        r.S = a.seg0_split;
    } else {
        const int v = u - seg0_units;
        const int q = v / a.seg1_split;
        r.tile = a.seg0_tiles + q;
        r.s = v - q * a.seg1_split;
        r.S = a.seg1_split;
    }
    r.ufirst = u - r.s;
    tile_coords(r.tile, a.tiles_m, a.tiles_n, a.tiles_per_batch, a.group_m, r.b, r.tm, r.tn);
    r.kb0 = kb_split(a.num_kb, r.s, r.S);
    r.kb1 = kb_split(a.num_kb, r.s + 1, r.S);
    r.p = 0;
    return r;
}

// Grouped launch: unit u is one whole-K tile of problem p, found by a
// forward scan from `hint` (each warp visits units in increasing order).
__device__ __forceinline__ Unit decode_grouped(const GroupTable &g, int group_m, int u, int &hint)
{
    int p = hint;
    while (p + 1 < g.count && g.info[p + 1].unit_begin <= u) ++p;
    hint = p;
    const GroupInfo &q = g.info[p];
    Unit r;
    r.p = p;
    r.tile = u - q.unit_begin;
    r.s = 0;
    r.S = 1;
    r.ufirst = u;
    tile_coords(r.tile, q.tiles_m, q.tiles_n, q.tiles_m * q.tiles_n, group_m, r.b, r.tm, r.tn);
    r.kb0 = 0;
    r.kb1 = q.num_kb;
    return r;
}

template <bool GROUPED>
__device__ __forceinline__ Unit decode(const MmaArgs &a, const TableOf<GROUPED> &g, int u, int &hint)
{
    if constexpr (GROUPED)
        return decode_grouped(g, a.group_m, u, hint);
    else
        return decode_unit(a, u);
}

// What the MMA thread needs of unit u: its K-block count and (grouped) its
// problem -- no tile coordinates, and no division for a whole-K unit.  The
// thread's time between two tiles is time the tensor core stands idle.
struct MmaUnit {
    int nkb, p;
};
template <bool GROUPED>
__device__ __forceinline__ MmaUnit mma_unit(const MmaArgs &a, const TableOf<GROUPED> &g, int u, int &hint)
{
    if constexpr (GROUPED) {
        int p = hint;
        while (p + 1 < g.count && g.info[p + 1].unit_begin <= u) ++p;
        hint = p;
        return MmaUnit{g.info[p].num_kb, p};
    } else {
        const int seg0_units = a.seg0_tiles * a.seg0_split;
        const bool seg0 = u < seg0_units;
        const int S = seg0 ? a.seg0_split : a.seg1_split;
        if (S == 1) return MmaUnit{a.num_kb, 0};
        const int s = (seg0 ? u : u - seg0_units) % S;
        return MmaUnit{kb_split(a.num_kb, s + 1, S) - kb_split(a.num_kb, s, S), 0};
    }
}

__device__ __forceinline__ void tma_load(const void *tmap, bool is3d, uint32_t dst, uint32_t bar, int c0,
                                         int c1, int c2)
{
    if (is3d)
        tma_load_3d(dst, tmap, bar, c0, c1, c2);
    else
        tma_load_2d(dst, tmap, bar, c0, c1);
}

// ---------------------------------------------------------------- epilogue

// v <- alpha * v + beta * C_old[row, col0 .. col0+31]; C_old is read only
// when beta != 0 (masked to M, N)
__device__ __forceinline__ void apply_alpha_beta(const MmaArgs &a, int b, long long row, long long col0,
                                                 float (&v)[32])
{
    if (a.beta == 0.0f || row >= a.M) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = a.alpha * v[j];
        return;
    }
    const long long base = (long long)b * a.stride_c + row * a.ldc + col0;
    const bool vec = (col0 + 32 <= a.N) && a.c_vec_ok;
    if (vec && a.c_dtype == TC_F32) {
        const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(a.C) + base);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 c = src[q];
            v[4 * q + 0] = fmaf(a.beta, c.x, a.alpha * v[4 * q + 0]);
            v[4 * q + 1] = fmaf(a.beta, c.y, a.alpha * v[4 * q + 1]);
            v[4 * q + 2] = fmaf(a.beta, c.z, a.alpha * v[4 * q + 2]);
            v[4 * q + 3] = fmaf(a.beta, c.w, a.alpha * v[4 * q + 3]);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float c = (col0 + j < a.N) ? load_c(a.C, base + j, a.c_dtype) : 0.0f;
            v[j] = fmaf(a.beta, c, a.alpha * v[j]);
        }
    }
}

// Column col0 + lane's bias (0 past N or without a bias), which the lane
// loads for bias_act.
__device__ __forceinline__ float bias_of(const MmaArgs &a, int lane, long long col0)
{
    const long long col = col0 + lane;
    return (a.bias && col < a.N) ? load_c(a.bias, col, a.c_dtype) : 0.0f;
}

// x[i] for a run-time i < N, from registers (the unrolled selects keep the
// array out of local memory).
template <int N>
__device__ __forceinline__ float pick(const float (&x)[N], int i)
{
    float r = x[0];
#pragma unroll
    for (int k = 1; k < N; ++k) r = (i == k) ? x[k] : r;
    return r;
}

// The warp's chunk, lane = row, v[j] = column col0 + j: add the column's
// bias (bl: lane j holds column col0 + j's value, from bias_of, shared by
// shuffles) and apply the activation.  Every lane of the warp calls it.
__device__ __forceinline__ void bias_act(const MmaArgs &a, float bl, float (&v)[32])
{
    if (a.bias) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += __shfl_sync(0xffffffffu, bl, j);
    }
    if (a.act == TC_ACT_GELU_TANH) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = gelu_tanh(v[j]);
    }
}

// The int8 path's dequantisation: the warp's chunk (lane = row, v[j] =
// column col0 + j) times the column's scale, before alpha/beta.
__device__ __forceinline__ void col_scale_apply(const MmaArgs &a, int lane, long long col0, float (&v)[32])
{
    const long long col = col0 + lane;
    const float sl = (col < a.N) ? a.col_scale[col] : 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] *= __shfl_sync(0xffffffffu, sl, j);
}

// C[row, col0 .. col0+31] = v with plain stores (C not readable by TMA)
__device__ __forceinline__ void store_direct(const MmaArgs &a, int b, long long row, long long col0,
                                             const float (&v)[32])
{
    if (row >= a.M) return;
    const long long base = (long long)b * a.stride_c + row * a.ldc + col0;
    if ((col0 + 32 <= a.N) && a.c_vec_ok) {
        if (a.c_dtype == TC_F32) {
            float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(a.C) + base);
#pragma unroll
            for (int q = 0; q < 8; ++q)
                dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else {
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.C) + base);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 w;
                w.x = pack2(v[8 * q + 0], v[8 * q + 1], a.c_dtype);
                w.y = pack2(v[8 * q + 2], v[8 * q + 3], a.c_dtype);
                w.z = pack2(v[8 * q + 4], v[8 * q + 5], a.c_dtype);
                w.w = pack2(v[8 * q + 6], v[8 * q + 7], a.c_dtype);
                dst[q] = w;
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (col0 + j < a.N) store_c1(a.C, base + j, v[j], a.c_dtype);
    }
}

// C layouts TMA cannot address (rows not 16-byte multiples): the warp's
// 32 x 32 chunk is transposed through shared memory and every global access
// touches one contiguous 32-element row segment per instruction instead of
// 32 separate rows.  Element (r, c) sits at r * 32 + (c ^ r): for a fixed r
// the 32 columns, and for a fixed c the 32 rows, fall in 32 distinct banks,
// and the buffer is exactly one 4 KB staging buffer.
__device__ __forceinline__ int xp(int r, int c) { return r * 32 + (c ^ r); }

// Row r of the chunk in column `lane`: C + ((b * stride_c + (row0 + r) * ldc + col) elements.
// Every access of the two functions below is unrolled and predicated (no
// early exit), so the 32 row accesses of a lane are independent and in
// flight together.

// v <- alpha * v + beta * C_old, C_old read row-coalesced through `buf`
__device__ __forceinline__ void apply_alpha_beta_staged(const MmaArgs &a, float *buf, int lane, int b,
                                                        long long row0, long long col0, float (&v)[32])
{
    if (a.beta == 0.0f) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = a.alpha * v[j];
        return;
    }
    const long long col = col0 + lane;
    const long long nrows = (col < a.N) ? min(32LL, a.M - row0) : 0LL;
    const long long first = (long long)b * a.stride_c + row0 * a.ldc + col;
    float c[32];
    if (a.c_dtype == TC_F32) {
        const float *src = static_cast<const float *>(a.C) + first;
#pragma unroll
        for (int r = 0; r < 32; ++r) c[r] = (r < nrows) ? src[r * a.ldc] : 0.0f;
    } else {
        const uint16_t *src = static_cast<const uint16_t *>(a.C) + first;
        uint16_t h[32];
#pragma unroll
        for (int r = 0; r < 32; ++r) h[r] = (r < nrows) ? src[r * a.ldc] : (uint16_t)0;
        if (a.c_dtype == TC_BF16) {
#pragma unroll
            for (int r = 0; r < 32; ++r) c[r] = __bfloat162float(__ushort_as_bfloat16(h[r]));
        } else {
#pragma unroll
            for (int r = 0; r < 32; ++r) c[r] = __half2float(__ushort_as_half(h[r]));
        }
    }
#pragma unroll
    for (int r = 0; r < 32; ++r) buf[xp(r, lane)] = c[r];
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = fmaf(a.beta, buf[xp(lane, j)], a.alpha * v[j]);
    __syncwarp();
}

// C[row0 .. row0+31, col0 .. col0+31] = the warp's chunk, row-coalesced through `buf`
__device__ __forceinline__ void store_staged(const MmaArgs &a, float *buf, int lane, int b, long long row0,
                                             long long col0, const float (&v)[32])
{
#pragma unroll
    for (int j = 0; j < 32; ++j) buf[xp(lane, j)] = v[j];
    __syncwarp();
    const long long col = col0 + lane;
    const long long nrows = (col < a.N) ? min(32LL, a.M - row0) : 0LL;
    const long long first = (long long)b * a.stride_c + row0 * a.ldc + col;
    float w[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) w[r] = buf[xp(r, lane)];
    if (a.c_dtype == TC_F32) {
        float *dst = static_cast<float *>(a.C) + first;
#pragma unroll
        for (int r = 0; r < 32; ++r)
            if (r < nrows) dst[r * a.ldc] = w[r];
    } else if (a.c_dtype == TC_BF16) {
        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.C) + first;
#pragma unroll
        for (int r = 0; r < 32; ++r)
            if (r < nrows) dst[r * a.ldc] = __float2bfloat16_rn(w[r]);
    } else {
        __half *dst = static_cast<__half *>(a.C) + first;
#pragma unroll
        for (int r = 0; r < 32; ++r)
            if (r < nrows) dst[r * a.ldc] = __float2half_rn(w[r]);
    }
    __syncwarp();
}

// The warp's 32 x 32 chunk (lane = row) goes through a swizzled shared
// buffer and one TMA store, which also clips rows and columns beyond the
// tensor.  fp32 rows are 128 bytes (128-byte swizzle: 16-byte unit q of row
// r sits at q ^ (r % 8)); 16-bit rows are 64 bytes (64-byte swizzle:
// q ^ ((r / 2) % 4)).  Either way each group of 8 lanes covers all 32 banks.
// BUFS: the warp's staging buffers (the stores that may still be reading
// one of the others: BUFS - 1).
template <int BUFS>
__device__ __forceinline__ void store_tma(const CUtensorMap *map, bool is3d, int dtype, uint8_t *buf, int lane,
                                          int b, long long row0, long long col0, const float (&v)[32])
{
    if (lane == 0) bulk_wait_read<BUFS - 1>();      // this buffer's previous store has read it
    __syncwarp();
    if (dtype == TC_F32) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4 *>(buf + lane * 128 + ((q ^ (lane & 7)) << 4)) =
                make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack2(v[8 * q + 0], v[8 * q + 1], dtype);
            w.y = pack2(v[8 * q + 2], v[8 * q + 3], dtype);
            w.z = pack2(v[8 * q + 4], v[8 * q + 5], dtype);
            w.w = pack2(v[8 * q + 6], v[8 * q + 7], dtype);
            *reinterpret_cast<uint4 *>(buf + lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4)) = w;
        }
    }
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (is3d)
            tma_store_3d(map, smem_u32(buf), (int)col0, (int)row0, b);
        else
            tma_store_2d(map, smem_u32(buf), (int)col0, (int)row0);
        bulk_commit();
    }
}

// ---------------------------------------------------------------- cluster split-K

// Rows of BN + 4 floats: with 16-byte stores by 32 lanes that each own one
// row, every group of 8 lanes covers all 32 banks (row r starts at 16-byte
// unit 33r, i.e. r mod 8 within a 128-byte line).
template <int BN>
__host__ __device__ constexpr int csplit_ld() { return BN + 4; }

// The per-column scale (when present), alpha/beta (C_old read only when
// beta != 0), then the fused bias and activation, then one rounding: four
// consecutive columns of one row of C.
template <bool EPI>
__device__ __forceinline__ void finish4(const MmaArgs &a, int b, long long grow, long long gcol, float (&v)[4])
{
    const long long base = (long long)b * a.stride_c + grow * a.ldc + gcol;
    const bool whole = a.c_vec_ok && gcol + 4 <= a.N;
    if constexpr (EPI) {
        if (a.col_scale) {
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] *= (gcol + j < a.N) ? a.col_scale[gcol + j] : 0.0f;
        }
    }
    if (a.beta != 0.0f) {
        float c[4];
        if (whole && a.c_dtype == TC_F32) {
            const float4 x = *reinterpret_cast<const float4 *>(static_cast<const float *>(a.C) + base);
            c[0] = x.x, c[1] = x.y, c[2] = x.z, c[3] = x.w;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) c[j] = (gcol + j < a.N) ? load_c(a.C, base + j, a.c_dtype) : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = fmaf(a.beta, c[j], a.alpha * v[j]);
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = a.alpha * v[j];
    }
    if constexpr (EPI) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (a.bias && gcol + j < a.N) v[j] += load_c(a.bias, gcol + j, a.c_dtype);
            if (a.act == TC_ACT_GELU_TANH) v[j] = gelu_tanh(v[j]);
        }
    }
    if (whole) {
        if (a.c_dtype == TC_F32) {
            *reinterpret_cast<float4 *>(static_cast<float *>(a.C) + base) = make_float4(v[0], v[1], v[2], v[3]);
        } else {
            uint2 w;
            w.x = pack2(v[0], v[1], a.c_dtype);
            w.y = pack2(v[2], v[3], a.c_dtype);
            *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(a.C) + base) = w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (gcol + j < a.N) store_c1(a.C, base + j, v[j], a.c_dtype);
    }
}

// The K slices of one output tile run as one cluster of S CTAs (slice s on
// the CTA of cluster rank s).  Each CTA has left its slice's fp32 partial
// tile in its own shared memory (rows of csplit_ld<BN>() floats); here the
// CTA of rank r sums rows [r * ceil(BM/S), ...) of all S partial tiles,
// reading its peers' shared memory in slice order (deterministic), and
// writes those rows of C.  Every thread of the CTA takes part.
template <int BN, bool EPI>
__device__ __forceinline__ void csplit_reduce(const MmaArgs &a, const uint8_t *partial)
{
    constexpr int LD = csplit_ld<BN>();
    constexpr int G = BN / 4;                       // 16-byte groups per row
    constexpr int SMAX = 16;
    const int S = a.seg0_split;
    const uint32_t rank = cluster_ctarank();
    const int rows = (BM + S - 1) / S;
    const int r0 = min(BM, (int)rank * rows), r1 = min(BM, r0 + rows);
    const Unit w = decode_unit(a, (int)blockIdx.x);
    const uint32_t base = smem_u32(partial);
    for (int g = threadIdx.x; g < (r1 - r0) * G; g += blockDim.x) {
        const int row = r0 + g / G, c4 = (g % G) * 4;
        const long long grow = (long long)w.tm * BM + row, gcol = (long long)w.tn * BN + c4;
        if (grow >= a.M || gcol >= a.N) continue;
        const uint32_t off = base + (uint32_t)((row * LD + c4) * 4);
        float4 p[SMAX];
#pragma unroll
        for (int q = 0; q < SMAX; ++q)
            if (q < S) p[q] = ld_shared_cluster_f4(mapa_shared(off, (uint32_t)q));
        float v[4] = {p[0].x, p[0].y, p[0].z, p[0].w};
#pragma unroll
        for (int q = 1; q < SMAX; ++q) {
            if (q < S) {
                v[0] += p[q].x;
                v[1] += p[q].y;
                v[2] += p[q].z;
                v[3] += p[q].w;
            }
        }
        finish4<EPI>(a, w.b, grow, gcol, v);
    }
}

// ---------------------------------------------------------------- kernel

// CG = 1: one CTA computes a 128 x BN tile with tcgen05.mma.cta_group::1.
// CG = 2: a cluster of two CTAs computes a 256 x BN tile with
//   tcgen05.mma.cta_group::2 issued by the even CTA; each CTA loads its own
//   128 rows of A and its own BN/2 columns of B, and each CTA's TMEM holds
//   its 128 rows of the accumulator.  Both CTAs' copies complete on the even
//   CTA's "full" barriers; its MMA commits arrive on both CTAs' "empty" and
//   "tmem full" barriers; both CTAs' epilogues release the accumulator on
//   the even CTA's "tmem empty" barrier.
//
// GROUPED: the units are the tiles of several problems (a GroupTable); each
// warp switches descriptors and epilogue fields when its next unit belongs
// to another problem.
//
// EPI: the fused bias/activation epilogue is compiled in (the plain GEMM
// kernels carry none of its code).
//
// I8ACC: the int8 path's exact accumulation on chip.  A unit is a whole
// tile; its K range is cut into slices of args.slice_kb blocks (at most 1024
// products of int8 values, so each slice's fp32 accumulator holds exact
// integers), each slice accumulated from zero in one of the two TMEM
// buffers, and the epilogue adds every slice as int32 to running sums kept
// in a third TMEM region.  The split-K path writes each slice to memory and
// adds them in a second kernel instead; the integer sums, their one rounding
// and everything after are the same.
//
// CSPLIT: split-K inside one launch.  The grid holds one unit per CTA and
// the S K slices of a tile form one cluster (slice = cluster rank); each
// slice's partial tile stays in its CTA's shared memory and csplit_reduce
// adds them across the cluster, so no partial tile goes through global
// memory and no second kernel runs.
template <int BN, int CG, bool GROUPED, bool EPI, bool I8ACC = false, bool CSPLIT = false>
__global__ void __launch_bounds__(mma_threads(BN, CG, EPI || GROUPED), 1)
    mma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmW,
               const MmaArgs args, const __grid_constant__ TableOf<GROUPED> gt)
{
    constexpr int BNL = BN / CG;                   // B columns loaded by this CTA
    constexpr int STAGE = stage_bytes(BN, CG);
    constexpr int A_BYTES = BM * BK * 2;
    // eight epilogue warps where the epilogue has CUDA-core work to hide:
    // the fused bias/activation, and grouped launches (whose ragged problems
    // often store C by plain stores, row-coalesced through shared memory)
    constexpr bool WIDE = EPI || GROUPED;
    constexpr int S = mma_stages(BN, CG, WIDE);
    constexpr int EW = epi_warps(BN, CG, WIDE);    // epilogue warps 0..EW-1, then the TMA and MMA warps
    constexpr int TMA_WARP = EW, MMA_WARP = EW + 1;
    constexpr int CSTEP = EW / 4;                  // chunks between two chunks of one epilogue warp
    constexpr int TCOLS = I8ACC ? 512 : tmem_cols(BN);
    constexpr int ACC_STRIDE = I8ACC ? BN : TCOLS / 2;   // TMEM columns between the two accumulators
    constexpr uint32_t RUN_COL = 2 * BN;           // I8ACC: the running int32 sums
    static_assert(!I8ACC || (EPI && !GROUPED && 3 * BN <= 512), "on-chip slices: two accumulators and the sums");
    static_assert(!CSPLIT || (CG == 1 && !GROUPED && !I8ACC), "cluster split-K: one CTA per slice");
    static_assert(!CSPLIT || BM * csplit_ld<BN>() * 4 <= S * STAGE, "the partial tile fits in the idle ring");
    constexpr int CHUNKS = BN / 32;
    static_assert(CG == 1 || CG == 2, "one CTA or a CTA pair");
    constexpr int CL = CG;                        // CTAs per cluster
    static_assert(BNL % 32 == 0 && BN <= 256, "each CTA's B share must be whole 32-column boxes");
    // An MN-major B share that is not a multiple of 64 columns (the 96 of
    // each CTA of a 256 x 192 pair) is held as 32-column chunks with the
    // 64-byte swizzle (64 K rows x 64 bytes = 4 KB each), copied by boxes
    // of 32 columns (or one 3-D copy of 32-element chunks); the host
    // encodes B's descriptor to match.  A K-major share keeps the 128-byte
    // swizzle: BNL rows of 128 bytes.
    constexpr bool B_SW64 = (BNL % 64) != 0;
    static_assert(!B_SW64 || (!GROUPED && !CSPLIT), "32-column B chunks: plain launches only");
    static_assert(STAGE % 1024 == 0, "stages must keep 1024-byte alignment for the 128B swizzle");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *cstage = smem + S * STAGE;            // epilogue staging
    uint64_t *bars = reinterpret_cast<uint64_t *>(cstage + epi_smem(BN, CG, WIDE));
    uint64_t *full_bar = bars;
    uint64_t *empty_bar = bars + S;
    uint64_t *tfull_bar = bars + 2 * S;
    uint64_t *tempty_bar = bars + 2 * S + 2;
    uint64_t *drain_bar = bars + 2 * S + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * S + 5);
    volatile uint32_t *abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = (CL == 2) ? cluster_ctarank() : 0u;
    const int cluster = blockIdx.x / CL;
    const int nclusters = gridDim.x / CL;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_u32(&full_bar[i]), 1);
            mbar_init(smem_u32(&empty_bar[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&tfull_bar[i]), 1);
            mbar_init(smem_u32(&tempty_bar[i]), EW * CG);   // one arrival per epilogue warp
        }
        mbar_init(smem_u32(drain_bar), 1);
        *abort_flag = 0u;
        fence_barrier_init();
    }
    if (warp == TMA_WARP && lane == 0) {
        if constexpr (!GROUPED) {
            prefetch_tmap(&tmA);
            prefetch_tmap(&tmB);
            if (args.c_tma) prefetch_tmap(&tmC);
            if (args.ws) prefetch_tmap(&tmW);
        }
        // let the next kernel in the stream (the split-K reduction, or the
        // next GEMM) launch early; it waits for this grid to finish before
        // it touches global memory
        griddep_launch_dependents();
    }
    __syncwarp();
    if (warp == 0) {
        if (CG == 1)
            tmem_alloc(smem_u32(tmem_slot), TCOLS);
        else
            tmem_alloc_pair(smem_u32(tmem_slot), TCOLS);
    }
    tc_fence_before();
    __syncthreads();
    if (CL == 2) cluster_sync();     // the peer's barriers exist before anyone signals them
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // launched as a programmatic dependent: everything above (barriers,
    // TMEM, descriptor prefetch) overlapped the previous kernel; the
    // operands, C and the status word are touched only once it has finished
    griddep_wait();

    const Watch watch{abort_flag, args.status, args.timeout_ns};

    if (warp == TMA_WARP) {
        // ------------------------------------------------ TMA producer
        // Its loop per K block is short too (the copies it issues per K block
        // pace it): barrier and stage addresses come from bases computed once.
        if (lane == 0) {
            uint32_t stage = 0, ph = 0, issued = 0;
            bool ok = true;
            int hint = 0;
            const uint32_t s0 = smem_u32(smem);
            const uint32_t full0 = smem_u32(&full_bar[0]), empty0 = smem_u32(&empty_bar[0]);
            // the even CTA's barriers count both CTAs' bytes
            const uint32_t full0_lead = CG == 2 ? mapa_shared(full0, 0) : full0;
            for (int u = cluster; ok && u < args.total_units; u += nclusters) {
                const Unit w = decode<GROUPED>(args, gt, u, hint);
                const CUtensorMap *mapA = &tmA, *mapB = &tmB;
                int a_kmajor = args.a_kmajor, b_kmajor = args.b_kmajor;
                bool a_3d = args.a_3d, b_3d = args.b_3d;
                bool a_chunked = args.a_chunked, b_chunked = args.b_chunked;
                if constexpr (GROUPED) {
                    mapA = &gt.tmA[w.p];
                    mapB = &gt.tmB[w.p];
                    a_kmajor = gt.info[w.p].a_kmajor;
                    b_kmajor = gt.info[w.p].b_kmajor;
                    a_3d = b_3d = false;
                    a_chunked = b_chunked = false;
                }
                const int m0 = w.tm * (BM * CL) + (int)rank * BM;
                const int n0 = w.tn * BN + (CG == 2 ? (int)rank * BNL : 0);
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!wait_bar(empty0 + 8 * stage, ph ^ 1u, watch, W_EMPTY)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full0_lead + 8 * stage;
                    if (CG == 1)
                        mbar_arrive_expect_tx(full0 + 8 * stage, STAGE - args.a_short_bytes);
                    else if (rank == 0)
                        mbar_arrive_expect_tx(full0 + 8 * stage, 2 * STAGE);
                    const uint32_t sa = s0 + stage * STAGE;
                    const uint32_t sb = sa + A_BYTES;
                    const int k0 = kb * BK;
                    auto load = [&](const CUtensorMap *tm, bool is3d, uint32_t dst, int c0, int c1) {
                        if (CG == 1) {
                            tma_load(tm, is3d, dst, fb, c0, c1, w.b);
                        } else if (is3d) {
                            tma_load_3d_pair(dst, tm, fb, c0, c1, w.b);
                        } else {
                            tma_load_2d_pair(dst, tm, fb, c0, c1);
                        }
                    };
                    // one 3-D copy of a chunked descriptor: (element, K row, chunk)
                    auto load_chunks = [&](const CUtensorMap *tm, uint32_t dst, int mn0) {
                        if (CG == 1)
                            tma_load_3d(dst, tm, fb, 0, k0, mn0 / 64);
                        else
                            tma_load_3d_pair(dst, tm, fb, 0, k0, mn0 / 64);
                    };
                    if (a_kmajor) {
                        load(mapA, a_3d, sa, k0, m0);
                    } else if (a_chunked) {
                        load_chunks(mapA, sa, m0);
                    } else {
                        load(mapA, a_3d, sa, m0, k0);
                        load(mapA, a_3d, sa + 8192, m0 + 64, k0);
                    }
                    if (b_kmajor) {
                        load(mapB, b_3d, sb, k0, n0);
                    } else if (B_SW64) {
                        if (b_chunked) {
                            if (CG == 1)
                                tma_load_3d(sb, mapB, fb, 0, k0, n0 / 32);
                            else
                                tma_load_3d_pair(sb, mapB, fb, 0, k0, n0 / 32);
                        } else {
#pragma unroll
                            for (int j = 0; j < BNL / 32; ++j) load(mapB, b_3d, sb + j * 4096, n0 + 32 * j, k0);
                        }
                    } else if (b_chunked) {
                        load_chunks(mapB, sb, n0);
                    } else {
#pragma unroll
                        for (int j = 0; j < BNL / 64; ++j) load(mapB, b_3d, sb + j * 8192, n0 + 64 * j, k0);
                    }
                    ++issued;
                    if (++stage == (uint32_t)S) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok && (CG == 1 || rank == 0)) {
                // let the copies already issued land before shared memory is released
                for (uint32_t i = (issued > (uint32_t)S ? issued - S : 0u); i < issued; ++i)
                    drain_wait(smem_u32(&full_bar[i % S]), (i / S) & 1u);
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------ MMA issuer (even CTA of a pair)
        // One thread feeds the tensor core, and its work between two MMAs
        // paces the K loop: rebuilding both shared-memory descriptors per
        // MMA cost ~3 % of the square bf16 GEMM's time on GB300.  Each
        // descriptor is built once per unit and then advanced by additions,
        // and the ring position is stepped rather than divided out.
        if (lane == 0 && (CG == 1 || rank == 0)) {
            uint32_t stage = 0, ph = 0, local = 0;
            bool ok = true;
            int hint = 0;
            for (int u = cluster; ok && u < args.total_units; u += nclusters) {
                const MmaUnit w = mma_unit<GROUPED>(args, gt, u, hint);
                int a_kmajor = args.a_kmajor, b_kmajor = args.b_kmajor;
                uint32_t idesc = args.idesc;
                if constexpr (GROUPED) {
                    a_kmajor = gt.info[w.p].a_kmajor;
                    b_kmajor = gt.info[w.p].b_kmajor;
                    idesc = gt.info[w.p].idesc;
                }
                // descriptors of stage 0, K step 0.  A stage adds STAGE bytes
                // to the start address; a K step of 16 adds 32 bytes along the
                // swizzled row (K-major) or 16 rows of 128 bytes (MN-major).
                // Shared addresses stay below 2^18 bytes, so the additions
                // never carry out of the descriptor's 14-bit address field.
                const uint32_t s0 = smem_u32(smem);
                const uint64_t ad0 = a_kmajor ? smem_desc_sw128(s0, 16, 1024) : smem_desc_sw128(s0, 8192, 1024);
                // (32-column B chunks: 4 KB apart, 8 K rows of 64 bytes = 512
                // bytes per swizzle atom, a K step of 16 rows = 1024 bytes)
                const uint64_t bd0 = b_kmajor ? smem_desc_sw128(s0 + A_BYTES, 16, 1024)
                                     : B_SW64 ? smem_desc(s0 + A_BYTES, 4096, 512, SMEM_SW64)
                                              : smem_desc_sw128(s0 + A_BYTES, 8192, 1024);
                const uint64_t astep = a_kmajor ? 2u : 128u, bstep = b_kmajor ? 2u : B_SW64 ? 64u : 128u;
                // Segments of the unit, each accumulated in its own TMEM buffer
                // from zero: the whole K range, or (I8ACC) K slices of
                // args.slice_kb blocks that the epilogue adds up on chip.
                const int seg_kb = I8ACC ? args.slice_kb : w.nkb;
                for (int k0 = 0; ok && k0 < w.nkb; k0 += seg_kb, ++local) {
                    const int k1 = min(k0 + seg_kb, w.nkb);
                    const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
                    if (!wait_bar(smem_u32(&tempty_bar[acc]), aph ^ 1u, watch, W_TMEM_EMPTY)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + acc * ACC_STRIDE;
                    for (int kb = k0; kb < k1; ++kb) {
                        if (!wait_bar(smem_u32(&full_bar[stage]), ph, watch, W_FULL)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t soff = (uint64_t)(stage * (STAGE >> 4));
#pragma unroll
                        for (int k = 0; k < BK / MMA_K; ++k) {
                            const uint64_t ad = ad0 + soff + k * astep, bd = bd0 + soff + k * bstep;
                            const uint32_t accum = (kb > k0 || k > 0) ? 1u : 0u;
                            if (CG == 1)
                                mma_f16_ss(d_tmem, ad, bd, idesc, accum);
                            else
                                mma_f16_ss_pair(d_tmem, ad, bd, idesc, accum);
                        }
                        if (CG == 1)
                            mma_commit(smem_u32(&empty_bar[stage]));
                        else
                            mma_commit_pair(smem_u32(&empty_bar[stage]), (uint16_t)0x3);
                        if (++stage == (uint32_t)S) {
                            stage = 0;
                            ph ^= 1u;
                        }
                    }
                    if (!ok) break;
                    // test hook: withhold the "accumulator ready" signal of
                    // this CTA's first segment, so that the epilogue's bounded
                    // wait expires
                    if (args.debug_drop_tfull && local == 0) continue;
                    if (CG == 1)
                        mma_commit(smem_u32(&tfull_bar[acc]));
                    else
                        mma_commit_pair(smem_u32(&tfull_bar[acc]), (uint16_t)0x3);
                }
            }
            if (!ok) {
                if (CG == 1)
                    mma_commit(smem_u32(drain_bar));
                else
                    mma_commit_pair(smem_u32(drain_bar), (uint16_t)0x1);
                drain_wait(smem_u32(drain_bar), 0);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue warps 0..EW-1
        // warp w reads TMEM lane quarter w % 4 (tile rows 32 (w % 4) ..) and,
        // with eight warps, chunks w / 4, w / 4 + 2, ...
        uint32_t local = 0, ebuf = 0;
        const int quarter = warp & 3, chunk0 = warp >> 2;
        const int row_in_tile = (int)rank * BM + quarter * 32 + lane;
        constexpr int EBUFS = epi_bufs(BN, CG, WIDE);
        constexpr int LAST_C0 = CHUNKS - CSTEP;        // this warp's last chunk: LAST_C0 + chunk0
        static_assert(CHUNKS % CSTEP == 0, "chunks split evenly between the warps of a lane quarter");
        uint8_t *my_stage = cstage + warp * epi_warp_bytes(BN, CG, WIDE);
        // The warp's staging is either its TMA chunk buffers (two that
        // alternate over the stores actually issued, a buffer refilled only
        // after one newer store was committed; or one, refilled after its
        // store has read it) or, on the plain-store path, one transpose
        // buffer.  A grouped launch's problems may switch between
        // the two: the switch first lets every earlier store finish reading.
        enum { STG_TMA = 0, STG_XPOSE = 1 };
        int emode = STG_TMA;
        auto staging = [&](int mode) -> uint8_t * {
            if (mode != emode) {
                if (lane == 0) bulk_wait_read<0>();
                __syncwarp();
                emode = mode;
            }
            if (mode == STG_XPOSE) return my_stage;
            uint8_t *buf = my_stage + ebuf * EPI_STAGE_BYTES;
            if (EBUFS == 2) ebuf ^= 1u;
            return buf;
        };
        // grouped: the launch-wide arguments with the current problem's
        // epilogue fields (M, N, C, ldc, dtype, alpha, beta) swapped in
        MmaArgs ga = args;
        const CUtensorMap *mapC = &tmC;
        int cur_p = -1, hint = 0;
        const MmaArgs &ea = GROUPED ? ga : args;
        // alpha/beta, then the chunk to C (TMA store when C allows it); bl:
        // the chunk's bias, lane j holding column col0 + j's
        auto emit = [&](int b, long long row, long long col0, float (&v)[32], float bl) {
            if (!ea.c_tma) {
                float *xbuf = reinterpret_cast<float *>(staging(STG_XPOSE));
                if constexpr (EPI)
                    if (ea.col_scale) col_scale_apply(ea, lane, col0, v);
                apply_alpha_beta_staged(ea, xbuf, lane, b, row - lane, col0, v);
                if constexpr (EPI) bias_act(ea, bl, v);
                store_staged(ea, xbuf, lane, b, row - lane, col0, v);
                return;
            }
            if constexpr (EPI)
                if (ea.col_scale) col_scale_apply(ea, lane, col0, v);
            apply_alpha_beta(ea, b, row, col0, v);
            if constexpr (EPI) bias_act(ea, bl, v);
            if (ea.c_tma) {
                // buffers rotate over the stores actually issued
                const long long row0 = row - lane;
                if (row0 < ea.M && col0 < ea.N)
                    store_tma<EBUFS>(mapC, ea.c_3d, ea.c_dtype, staging(STG_TMA), lane, b, row0, col0, v);
            } else {
                store_direct(ea, b, row, col0, v);
            }
        };
        const uint32_t tempty_leader0 = CG == 2 ? mapa_shared(smem_u32(&tempty_bar[0]), 0) : 0u;
        const uint32_t tempty_leader1 = CG == 2 ? mapa_shared(smem_u32(&tempty_bar[1]), 0) : 0u;
        for (int u = cluster; u < args.total_units; u += nclusters) {
            const Unit w = decode<GROUPED>(args, gt, u, hint);
            if constexpr (GROUPED) {
                if (w.p != cur_p) {
                    const GroupInfo &q = gt.info[w.p];
                    ga.M = q.M;
                    ga.N = q.N;
                    ga.C = q.C;
                    ga.ldc = q.ldc;
                    ga.stride_c = 0;
                    ga.c_dtype = q.c_dtype;
                    ga.c_vec_ok = q.c_vec_ok;
                    ga.c_tma = q.c_tma;
                    ga.c_3d = 0;
                    ga.alpha = q.alpha;
                    ga.beta = q.beta;
                    mapC = &gt.tmC[w.p];
                    cur_p = w.p;
                }
            }
            // the bias of this warp's chunks of the tile, loaded before the
            // wait for the accumulator so that its latency hides behind the MMAs
            constexpr int NCH = CHUNKS / CSTEP;
            float bpre[NCH];
#pragma unroll
            for (int i = 0; i < NCH; ++i)
                bpre[i] = EPI ? bias_of(ea, lane, (long long)w.tn * BN + (chunk0 + i * CSTEP) * 32) : 0.0f;
            // segments of the unit (see the MMA warp): one, or the K slices
            // that I8ACC adds up in TMEM
            const int nseg = I8ACC ? (w.kb1 - w.kb0 + args.slice_kb - 1) / args.slice_kb : 1;
            bool ok = true;
            for (int sg = 0; sg < nseg; ++sg, ++local) {
                const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
                ok = wait_bar(smem_u32(&tfull_bar[acc]), aph, watch, W_TMEM_FULL);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * ACC_STRIDE;
                const long long row = (long long)w.tm * (BM * CL) + row_in_tile;
                // accumulator fully read: hand it back to the MMA warp (not after
                // this CTA's last segment: nothing waits for it then, and the
                // arrival would sit on the kernel's final critical path)
                const bool more = sg + 1 < nseg || u + nclusters < args.total_units;
                auto release = [&]() {
                    if (!more) return;
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (CG == 1)
                            mbar_arrive(smem_u32(&tempty_bar[acc]));
                        else
                            mbar_arrive_cluster(acc ? tempty_leader1 : tempty_leader0);
                    }
                };

                if constexpr (I8ACC) {
                    // This segment's fp32 accumulator holds exact integers (a
                    // K slice of at most 1024 int8 products); they are added as
                    // int32 to the running sums in TMEM columns RUN_COL.. of the
                    // same lanes, and after the last slice the exact sum is
                    // rounded once to fp32 and goes through the epilogue.
                    const uint32_t raddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + RUN_COL;
                    const bool first = sg == 0, last = sg + 1 == nseg;
#pragma unroll 1
                    for (int c = chunk0; c < CHUNKS; c += CSTEP) {
                        uint32_t r[32], q[32];
                        __syncwarp();
                        tmem_ld_32x32b_x32(taddr + c * 32, r);
                        if (!first) tmem_ld_32x32b_x32(raddr + c * 32, q);
                        tmem_ld_wait();
                        if (c == LAST_C0 + chunk0) release();
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const int x = __float2int_rn(__uint_as_float(r[j]));
                            q[j] = (uint32_t)(first ? x : (int)q[j] + x);
                        }
                        if (!last) {
                            tmem_st_32x32b_x32(raddr + c * 32, q);
                        } else {
                            float v[32];
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] = __int2float_rn((int)q[j]);
                            emit(w.b, row, (long long)w.tn * BN + c * 32, v, pick(bpre, (c - chunk0) / CSTEP));
                        }
                    }
                    if (!last) tmem_st_wait();
                } else if (w.S == 1) {
#pragma unroll 1
                    for (int c = chunk0; c < CHUNKS; c += CSTEP) {
                        uint32_t r[32];
                        __syncwarp();
                        tmem_ld_32x32b_x32(taddr + c * 32, r);
                        tmem_ld_wait();
                        if (c == LAST_C0 + chunk0) release();
                        float v[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                        emit(w.b, row, (long long)w.tn * BN + c * 32, v, pick(bpre, (c - chunk0) / CSTEP));
                    }
                } else if constexpr (CSPLIT) {
                    // K slice of a cluster split: the partial tile goes to this
                    // CTA's shared memory.  The ring is idle: every copy into it
                    // was consumed by an MMA, and every MMA has completed (this
                    // accumulator's commit).  csplit_reduce adds the slices.
                    float *red = reinterpret_cast<float *>(smem) + (quarter * 32 + lane) * csplit_ld<BN>();
#pragma unroll 1
                    for (int c = chunk0; c < CHUNKS; c += CSTEP) {
                        uint32_t r[32];
                        __syncwarp();
                        tmem_ld_32x32b_x32(taddr + c * 32, r);
                        tmem_ld_wait();
                        if (c == LAST_C0 + chunk0) release();
                        float4 *dst = reinterpret_cast<float4 *>(red + c * 32);
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            dst[q] = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                                 __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
                    }
                } else {
                    // K slice: the raw fp32 partial tile goes to its workspace
                    // slot (row-major, (BM * CG) x BN per unit); the reduction
                    // kernel sums the slices in slice order afterwards
                    const long long wrow0 =
                        (long long)(w.ufirst + w.s - args.split_base) * (BM * CG) + (int)rank * BM + quarter * 32;
#pragma unroll 1
                    for (int c = chunk0; c < CHUNKS; c += CSTEP) {
                        uint32_t r[32];
                        __syncwarp();
                        tmem_ld_32x32b_x32(taddr + c * 32, r);
                        tmem_ld_wait();
                        if (c == LAST_C0 + chunk0) release();
                        float v[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                        store_tma<EBUFS>(&tmW, false, TC_F32, staging(STG_TMA), lane, 0, wrow0, c * 32, v);
                    }
                }
            }
            if (!ok) break;
        }
        // every TMA store has read its shared-memory source before the CTA
        // releases it (the global writes complete with the kernel)
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if constexpr (CSPLIT) {
        cluster_sync();              // every slice's partial tile is in its CTA's shared memory
        csplit_reduce<BN, EPI>(args, smem);
        cluster_sync();              // no CTA releases its shared memory while a peer may read it
    } else if (CL == 2) {
        cluster_sync();              // no CTA leaves while its peer may still signal it or copy into it
    }
    tc_fence_after();
    if (warp == 0) {
        if (CG == 1)
            tmem_dealloc(tmem_base, TCOLS);
        else
            tmem_dealloc_pair(tmem_base, TCOLS);
    }
}

template <int BN, int CG, bool GROUPED = false, bool EPI = false, bool I8ACC = false, bool CSPLIT = false>
cudaError_t launch_kernel(const MmaLaunch &L, cudaStream_t st, const TableOf<GROUPED> &gt = TableOf<GROUPED>{})
{
    constexpr auto kern = mma_kernel<BN, CG, GROUPED, EPI, I8ACC, CSPLIT>;
    constexpr int smem = mma_smem_bytes(BN, CG, EPI || GROUPED);
    constexpr int threads = mma_threads(BN, CG, EPI || GROUPED);
    // per device: the kernel's shared-memory limit is raised once (callers
    // of the context-free entry point may race here from several threads;
    // setting the attribute twice is harmless)
    static std::atomic<bool> configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        if (CG == 2 || CSPLIT) {
            // cluster splits of up to 16 CTAs go beyond the portable 8
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, CSPLIT ? 1 : 0);
            if (e != cudaSuccess) return e;
        }
        configured[dev].store(true, std::memory_order_release);
    }
    const int cluster = CSPLIT ? L.args.seg0_split : CG;
    if (CSPLIT && (cluster < 2 || cluster > 16 || L.grid != L.args.total_units || L.grid % cluster != 0))
        return cudaErrorInvalidValue;
    return launch_dependent(kern, dim3(L.grid), dim3(threads), smem, st, (unsigned)cluster, L.tmA, L.tmB, L.tmC,
                            L.tmW, L.args, gt);
}

// Clusters of S CTAs of the BN-wide cluster-split kernel that can be
// resident at once on the current device (0 when such a cluster cannot run).
template <int BN>
int csplit_clusters_for(int S)
{
    constexpr auto kern = mma_kernel<BN, 1, false, false, false, true>;
    constexpr int smem = mma_smem_bytes(BN, 1);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)S, 1, 1);
    cfg.blockDim = dim3(MMA_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

template <int BN>
int pairs_for()
{
    constexpr int smem = mma_smem_bytes(BN, 2);
    if (cudaFuncSetAttribute(mma_kernel<BN, 2, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(MMA_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, mma_kernel<BN, 2, false, false>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

// ---------------------------------------------------------------- split-K reduction
// C tile = alpha * (p_0 + p_1 + ... + p_{S-1}) + beta * C_old, the slices
// summed in slice order (deterministic).  One CTA of bn threads owns COLS
// rows of one tile (its coordinates are decoded once per CTA); each thread
// owns COLS consecutive columns of one row, so every slice is read with
// 16-byte loads and C written with 16-byte (COLS = 8) or 8/16-byte stores,
// contiguous across a warp.  COLS = 8 unless that leaves few threads (a
// long split of few tiles), where COLS = 4 doubles them.  Launched as a
// programmatic dependent of the GEMM kernel: griddepcontrol.wait returns
// once that grid has finished and its partial tiles are visible.
// INT: the int8 path -- the slices hold exact integers, summed in 64 bits,
// then scaled per column (a template flag, so the fp32 reduction carries
// none of it).
template <bool INT, int COLS>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const ReduceArgs r)
{
    static_assert(COLS == 4 || COLS == 8, "whole 16-byte loads");
    griddep_wait();
    griddep_launch_dependents();     // the next GEMM may start its set-up
    // a GEMM wait that expired left partial tiles unwritten: do not sum them
    if (r.status && *reinterpret_cast<const volatile unsigned *>(r.status) != 0u) return;
    const int groups = r.bn / COLS;                    // threads per row
    const int ctas_per_tile = r.rows_per_tile / COLS;  // COLS rows per CTA
    const int t = blockIdx.x / ctas_per_tile;
    const int row = (blockIdx.x - t * ctas_per_tile) * COLS + (int)threadIdx.x / groups;
    const int cc = (int)threadIdx.x % groups;
    int b, tm, tn;
    tile_coords(r.first_tile + t, r.tiles_m, r.tiles_n, r.tiles_per_batch, r.group_m, b, tm, tn);
    const long long grow = (long long)tm * r.rows_per_tile + row;
    const long long gcol = (long long)tn * r.bn + cc * COLS;
    if (grow >= r.M || gcol >= r.N) return;
    const size_t slice = (size_t)r.rows_per_tile * r.bn;      // floats per partial tile
    const float *src = r.ws + (size_t)t * r.S * slice + (size_t)row * r.bn + cc * COLS;
    // the thread's COLS columns of slice s
    auto load = [&](int s, float (&p)[COLS]) {
#pragma unroll
        for (int q = 0; q < COLS / 4; ++q) {
            const float4 x = __ldcg(reinterpret_cast<const float4 *>(src + s * slice) + q);
            p[4 * q + 0] = x.x;
            p[4 * q + 1] = x.y;
            p[4 * q + 2] = x.z;
            p[4 * q + 3] = x.w;
        }
    };
    // Slices are added one after another in slice order; up to four
    // slices' loads are issued before their additions, so that a long
    // split (few threads, many slices) keeps several loads in flight.
    using Acc = std::conditional_t<INT, long long, float>;
    Acc acc[COLS] = {};
    auto add = [&](const float (&p)[COLS]) {
#pragma unroll
        for (int j = 0; j < COLS; ++j) {
            if constexpr (INT)
                acc[j] += __float2ll_rn(p[j]);     // exact integers: an exact 64-bit sum
            else
                acc[j] += p[j];
        }
    };
    int s = 0;
    for (; s + 4 <= r.S; s += 4) {
        float p[4][COLS];
#pragma unroll
        for (int i = 0; i < 4; ++i) load(s + i, p[i]);
#pragma unroll
        for (int i = 0; i < 4; ++i) add(p[i]);
    }
    for (; s < r.S; ++s) {
        float p[COLS];
        load(s, p);
        add(p);
    }
    float v[COLS];
    if constexpr (INT) {
        // one rounding of the exact sum to fp32, then the column's scale
#pragma unroll
        for (int j = 0; j < COLS; ++j) v[j] = __ll2float_rn(acc[j]);
#pragma unroll
        for (int j = 0; j < COLS; ++j)
            if (gcol + j < r.N) v[j] *= r.col_scale[gcol + j];
    } else {
#pragma unroll
        for (int j = 0; j < COLS; ++j) v[j] = acc[j];
        if (r.col_scale) {
            // a per-column scale on float slices (the int8-weight product)
#pragma unroll
            for (int j = 0; j < COLS; ++j)
                if (gcol + j < r.N) v[j] *= r.col_scale[gcol + j];
        }
    }
    const long long base = (long long)b * r.stride_c + grow * r.ldc + gcol;
#pragma unroll
    for (int j = 0; j < COLS; ++j) {
        const float c = (r.beta != 0.0f && gcol + j < r.N) ? load_c(r.C, base + j, r.c_dtype) : 0.0f;
        v[j] = (r.beta != 0.0f) ? fmaf(r.beta, c, r.alpha * v[j]) : r.alpha * v[j];
        if (r.bias && gcol + j < r.N) v[j] += load_c(r.bias, gcol + j, r.c_dtype);
        if (r.act == TC_ACT_GELU_TANH) v[j] = gelu_tanh(v[j]);
    }
    if (r.c_vec_ok && gcol + COLS <= r.N) {
        if (r.c_dtype == TC_F32) {
            float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(r.C) + base);
#pragma unroll
            for (int q = 0; q < COLS / 4; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else if constexpr (COLS == 8) {
            uint4 w;
            w.x = pack2(v[0], v[1], r.c_dtype);
            w.y = pack2(v[2], v[3], r.c_dtype);
            w.z = pack2(v[4], v[5], r.c_dtype);
            w.w = pack2(v[6], v[7], r.c_dtype);
            *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(r.C) + base) = w;
        } else {
            uint2 w;
            w.x = pack2(v[0], v[1], r.c_dtype);
            w.y = pack2(v[2], v[3], r.c_dtype);
            *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(r.C) + base) = w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < COLS; ++j)
            if (gcol + j < r.N) store_c1(r.C, base + j, v[j], r.c_dtype);
    }
}

}  // namespace

cudaError_t launch_reduce(const ReduceArgs &r, cudaStream_t st)
{
    if (r.bn % 8 != 0 || r.bn > 256 || r.rows_per_tile % 8 != 0 || r.ntiles < 1) return cudaErrorInvalidValue;
    // 8 columns per thread unless that leaves fewer threads than about one
    // 256-thread CTA per SM of a GB300
    const long long threads8 = (long long)r.ntiles * r.rows_per_tile * (r.bn / 8);
    const int cols = threads8 < 152LL * 256 ? 4 : 8;
    const dim3 grid((unsigned)r.ntiles * (unsigned)(r.rows_per_tile / cols)), block((unsigned)r.bn);
    if (r.int_sum)
        return cols == 4 ? launch_dependent(splitk_reduce_kernel<true, 4>, grid, block, 0, st, 1u, r)
                         : launch_dependent(splitk_reduce_kernel<true, 8>, grid, block, 0, st, 1u, r);
    return cols == 4 ? launch_dependent(splitk_reduce_kernel<false, 4>, grid, block, 0, st, 1u, r)
                     : launch_dependent(splitk_reduce_kernel<false, 8>, grid, block, 0, st, 1u, r);
}

cudaError_t launch_mma(const MmaLaunch &L, cudaStream_t st)
{
    const bool epi = L.args.bias != nullptr || L.args.act != TC_ACT_NONE || L.args.col_scale != nullptr;
    if (L.csplit) {
        if (L.cg != 1 || L.i8acc) return cudaErrorInvalidValue;
        switch (L.bn) {
        case 64: return epi ? launch_kernel<64, 1, false, true, false, true>(L, st)
                            : launch_kernel<64, 1, false, false, false, true>(L, st);
        case 128: return epi ? launch_kernel<128, 1, false, true, false, true>(L, st)
                             : launch_kernel<128, 1, false, false, false, true>(L, st);
        default: return cudaErrorInvalidValue;
        }
    }
    if (L.i8acc) {
        if (L.bn != 128 || L.args.slice_kb < 1 || L.args.col_scale == nullptr) return cudaErrorInvalidValue;
        return L.cg == 2 ? launch_kernel<128, 2, false, true, true>(L, st) : launch_kernel<128, 1, false, true, true>(L, st);
    }
    if (L.cg == 2) {
        switch (L.bn) {
        case 128: return epi ? launch_kernel<128, 2, false, true>(L, st) : launch_kernel<128, 2>(L, st);
        case 192: return epi ? launch_kernel<192, 2, false, true>(L, st) : launch_kernel<192, 2>(L, st);
        case 256: return epi ? launch_kernel<256, 2, false, true>(L, st) : launch_kernel<256, 2>(L, st);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (L.bn) {
    case 64: return epi ? launch_kernel<64, 1, false, true>(L, st) : launch_kernel<64, 1>(L, st);
    case 128: return epi ? launch_kernel<128, 1, false, true>(L, st) : launch_kernel<128, 1>(L, st);
    case 192: return epi ? launch_kernel<192, 1, false, true>(L, st) : launch_kernel<192, 1>(L, st);
    case 256: return epi ? launch_kernel<256, 1, false, true>(L, st) : launch_kernel<256, 1>(L, st);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_mma_grouped(const MmaLaunch &L, const GroupTable &g, cudaStream_t st)
{
    if (g.count < 1 || g.count > GROUP_MAX) return cudaErrorInvalidValue;
    if (L.cg == 2 && L.bn == 256) return launch_kernel<256, 2, true>(L, st, g);
    if (L.cg == 2 && L.bn == 128) return launch_kernel<128, 2, true>(L, st, g);
    if (L.cg == 1 && L.bn == 256) return launch_kernel<256, 1, true>(L, st, g);
    if (L.cg == 1 && L.bn == 128) return launch_kernel<128, 1, true>(L, st, g);
    return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------- static scratch
// Scratch of the entry point that allocates nothing (tc_gemm_splitk_noalloc):
// a file-scope device array, zero at load, held by every GPU that loads this
// library until the process exits.  Layout: split-K partial tiles, then a
// status word.
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

cudaError_t noalloc_scratch(NoallocScratch *out)
{
    // The array's name is only a host-side stand-in: its device address is
    // looked up once per device, with that device current.
    static std::mutex mu;
    static void *addr[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(mu);
    if (!addr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        if (!ptr) return cudaErrorInvalidSymbol;
        addr[dev] = ptr;
    }
    unsigned char *base = static_cast<unsigned char *>(addr[dev]);
    out->partials = reinterpret_cast<float *>(base);
    out->status = reinterpret_cast<unsigned *>(base + NOALLOC_PARTIAL_BYTES);
    return cudaSuccess;
}

int max_active_csplit_clusters(int bn, int S)
{
    if (S < 2 || S > 16) return 0;
    switch (bn) {
    case 64: return csplit_clusters_for<64>(S);
    case 128: return csplit_clusters_for<128>(S);
    default: return 0;
    }
}

int max_active_pairs(int bn)
{
    switch (bn) {
    case 128: return pairs_for<128>();
    case 192: return pairs_for<192>();
    case 256: return pairs_for<256>();
    default: return 0;
    }
}

}  // namespace tc
