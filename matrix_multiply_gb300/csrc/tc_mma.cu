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
#include "internal.h"
#include "ptx.cuh"
#include "../../include/tcgemm.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

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
    int b, tm, tn, s, kb0, kb1, tile;
};

__device__ __forceinline__ Unit decode_unit(const MmaArgs &a, int u)
{
    Unit r;
    r.s = u % a.split_k;
    const int rest = u / a.split_k;
    r.b = rest / a.tiles_per_batch;
    const int t = rest - r.b * a.tiles_per_batch;
    r.tile = t;
    // bands of group_m tile rows, column-major inside a band
    const int band = a.group_m * a.tiles_n;
    const int g = t / band;
    const int first_m = g * a.group_m;
    const int rows_in_band = min(a.tiles_m - first_m, a.group_m);
    const int in_band = t - g * band;
    r.tm = first_m + in_band % rows_in_band;
    r.tn = in_band / rows_in_band;
    r.kb0 = (int)(((long long)r.s * a.num_kb) / a.split_k);
    r.kb1 = (int)(((long long)(r.s + 1) * a.num_kb) / a.split_k);
    return r;
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

// out[row, col0 .. col0+31] = alpha * v + beta * C_old  (masked to M, N)
__device__ __forceinline__ void store_row_chunk(const MmaArgs &a, int b, long long row, long long col0,
                                                float (&v)[32])
{
    if (row >= a.M) return;
    const long long base = (long long)b * a.stride_c + row * a.ldc + col0;
    const bool full = (col0 + 32 <= a.N);
    const bool vec = full && a.c_vec_ok;
    if (a.beta != 0.0f) {
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
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = a.alpha * v[j];
    }

    if (vec) {
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

// ---------------------------------------------------------------- kernel

template <int BN>
__global__ void __launch_bounds__(MMA_THREADS, 1)
    mma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const MmaArgs args)
{
    constexpr int STAGE = stage_bytes(BN);
    constexpr int A_BYTES = BM * BK * 2;
    constexpr int S = mma_stages(BN);
    constexpr int TCOLS = tmem_cols(BN);
    constexpr int ACC_STRIDE = TCOLS / 2;      // TMEM columns between the two accumulators
    constexpr int CHUNKS = BN / 32;
    static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN must be 64, 128, 192 or 256");
    static_assert(STAGE % 1024 == 0, "stages must keep 1024-byte alignment for the 128B swizzle");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S * STAGE);
    uint64_t *full_bar = bars;
    uint64_t *empty_bar = bars + S;
    uint64_t *tfull_bar = bars + 2 * S;
    uint64_t *tempty_bar = bars + 2 * S + 2;
    uint64_t *drain_bar = bars + 2 * S + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * S + 5);
    volatile uint32_t *abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_u32(&full_bar[i]), 1);
            mbar_init(smem_u32(&empty_bar[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&tfull_bar[i]), 1);
            mbar_init(smem_u32(&tempty_bar[i]), 128);
        }
        mbar_init(smem_u32(drain_bar), 1);
        *abort_flag = 0u;
        fence_barrier_init();
    }
    if (warp == 4 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    __syncwarp();
    if (warp == 0) tmem_alloc(smem_u32(tmem_slot), TCOLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const Watch watch{abort_flag, args.status, args.timeout_ns};

    if (warp == 4) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < args.total_units; u += gridDim.x) {
                const Unit w = decode_unit(args, u);
                const int m0 = w.tm * BM, n0 = w.tn * BN;
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    const uint32_t stage = it % S, ph = (it / S) & 1u;
                    if (!wait_bar(smem_u32(&empty_bar[stage]), ph ^ 1u, watch, W_EMPTY)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&full_bar[stage]);
                    mbar_arrive_expect_tx(fb, STAGE);
                    const uint32_t sa = smem_u32(smem + stage * STAGE);
                    const uint32_t sb = sa + A_BYTES;
                    const int k0 = kb * BK;
                    if (args.a_kmajor) {
                        tma_load(&tmA, args.a_3d, sa, fb, k0, m0, w.b);
                    } else {
                        tma_load(&tmA, args.a_3d, sa, fb, m0, k0, w.b);
                        tma_load(&tmA, args.a_3d, sa + 8192, fb, m0 + 64, k0, w.b);
                    }
                    if (args.b_kmajor) {
                        tma_load(&tmB, args.b_3d, sb, fb, k0, n0, w.b);
                    } else {
#pragma unroll
                        for (int j = 0; j < BN / 64; ++j)
                            tma_load(&tmB, args.b_3d, sb + j * 8192, fb, n0 + 64 * j, k0, w.b);
                    }
                    ++it;
                }
            }
            if (!ok) {
                // let the copies already issued land before shared memory is released
                for (uint32_t i = (it > (uint32_t)S ? it - S : 0u); i < it; ++i)
                    drain_wait(smem_u32(&full_bar[i % S]), (i / S) & 1u);
            }
        }
        __syncwarp();
    } else if (warp == 5) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t it = 0, local = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < args.total_units; u += gridDim.x, ++local) {
                const Unit w = decode_unit(args, u);
                const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
                if (!wait_bar(smem_u32(&tempty_bar[acc]), aph ^ 1u, watch, W_TMEM_EMPTY)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * ACC_STRIDE;
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    const uint32_t stage = it % S, ph = (it / S) & 1u;
                    if (!wait_bar(smem_u32(&full_bar[stage]), ph, watch, W_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * STAGE);
                    const uint32_t sb = sa + A_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / MMA_K; ++k) {
                        // K-major: advance 32 bytes along the swizzled row;
                        // MN-major: advance 16 rows of 128 bytes.
                        const uint64_t ad = args.a_kmajor ? smem_desc_sw128(sa + 32 * k, 16, 1024)
                                                          : smem_desc_sw128(sa + 2048 * k, 8192, 1024);
                        const uint64_t bd = args.b_kmajor ? smem_desc_sw128(sb + 32 * k, 16, 1024)
                                                          : smem_desc_sw128(sb + 2048 * k, 8192, 1024);
                        mma_f16_ss(d_tmem, ad, bd, args.idesc, (kb > w.kb0 || k > 0) ? 1u : 0u);
                    }
                    mma_commit(smem_u32(&empty_bar[stage]));
                    ++it;
                }
                if (!ok) break;
                mma_commit(smem_u32(&tfull_bar[acc]));
            }
            if (!ok) {
                mma_commit(smem_u32(drain_bar));
                drain_wait(smem_u32(drain_bar), 0);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue warps 0-3
        uint32_t local = 0;
        const int row_in_tile = warp * 32 + lane;
        for (int u = blockIdx.x; u < args.total_units; u += gridDim.x, ++local) {
            const Unit w = decode_unit(args, u);
            const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
            bool ok = wait_bar(smem_u32(&tfull_bar[acc]), aph, watch, W_TMEM_FULL);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(warp * 32) << 16) + acc * ACC_STRIDE;
            const long long row = (long long)w.tm * BM + row_in_tile;

            if (args.split_k == 1) {
#pragma unroll 1
                for (int c = 0; c < CHUNKS; ++c) {
                    uint32_t r[32];
                    __syncwarp();
                    tmem_ld_32x32b_x32(taddr + c * 32, r);
                    tmem_ld_wait();
                    if (c == CHUNKS - 1) {
                        // accumulator fully read: hand it back to the MMA warp
                        tc_fence_before();
                        mbar_arrive(smem_u32(&tempty_bar[acc]));
                    }
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                    store_row_chunk(args, w.b, row, (long long)w.tn * BN + c * 32, v);
                }
            } else {
                // split-K: park this slice's partial tile (this warp's 32 rows),
                // column-interleaved so each store instruction is coalesced
                const long long tile_id = (long long)w.b * args.tiles_per_batch + w.tile;
                const size_t slab = (size_t)BN * 32;          // floats per warp quarter
                float *mine = args.ws + ((size_t)(tile_id * args.split_k + w.s) * 4 + warp) * slab;
#pragma unroll 1
                for (int c = 0; c < CHUNKS; ++c) {
                    uint32_t r[32];
                    __syncwarp();
                    tmem_ld_32x32b_x32(taddr + c * 32, r);
                    tmem_ld_wait();
                    if (c == CHUNKS - 1) {
                        tc_fence_before();
                        mbar_arrive(smem_u32(&tempty_bar[acc]));
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) __stcg(mine + (size_t)(c * 32 + j) * 32 + lane, __uint_as_float(r[j]));
                }
                __threadfence();
                __syncwarp();
                unsigned old = 0;
                unsigned *ticket = args.tickets + tile_id * 4 + warp;
                if (lane == 0) old = atomicAdd(ticket, 1u);
                old = __shfl_sync(0xffffffffu, old, 0);
                if (old == (unsigned)(args.split_k - 1)) {
                    // last slice to arrive: sum the slices in the fixed order 0..S-1
                    __threadfence();
                    const float *first = args.ws + ((size_t)(tile_id * args.split_k) * 4 + warp) * slab;
                    const size_t sstride = (size_t)4 * slab;
#pragma unroll 1
                    for (int c = 0; c < CHUNKS; ++c) {
                        float v[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = 0.0f;
                        for (int s = 0; s < args.split_k; ++s) {
                            const float *p = first + s * sstride + (size_t)(c * 32) * 32 + lane;
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] += __ldcg(p + j * 32);
                        }
                        store_row_chunk(args, w.b, row, (long long)w.tn * BN + c * 32, v);
                    }
                    if (lane == 0) *ticket = 0u;       // ready for the next launch
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem_base, TCOLS);
}

template <int BN>
cudaError_t launch_bn(const MmaLaunch &L, cudaStream_t st)
{
    constexpr int smem = mma_smem_bytes(BN);
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(mma_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    mma_kernel<BN><<<L.grid, MMA_THREADS, smem, st>>>(L.tmA, L.tmB, L.args);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mma(const MmaLaunch &L, cudaStream_t st)
{
    switch (L.bn) {
    case 64: return launch_bn<64>(L, st);
    case 128: return launch_bn<128>(L, st);
    case 192: return launch_bn<192>(L, st);
    case 256: return launch_bn<256>(L, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace tc
