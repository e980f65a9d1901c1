// Launch descriptions shared by the host API (api.cpp) and the kernels.
// Plain structs; no PyTorch types anywhere in the library.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace tc {

// Tile geometry of the tensor-core kernel.  Every output tile is BM rows by
// BN columns; the K loop steps BK elements (one 128-byte swizzle row of a
// 16-bit type) per pipeline stage.
constexpr int BM = 128;
constexpr int BK = 64;
constexpr int MMA_K = 16;                       // K of one kind::f16 tcgen05.mma
constexpr int MMA_THREADS = 192;                // 4 epilogue warps, TMA warp, MMA warp
constexpr int SMEM_LIMIT = 232448;              // max dynamic shared memory per block
constexpr int SMEM_RESERVE = 1024 + 256;        // alignment slack + barriers

__host__ __device__ constexpr int stage_bytes(int bn) { return (BM + bn) * BK * 2; }
__host__ __device__ constexpr int tmem_cols(int bn)
{
    return (2 * bn <= 128) ? 128 : (2 * bn <= 256) ? 256 : 512;
}
__host__ __device__ constexpr int mma_stages(int bn)
{
    return ((SMEM_LIMIT - SMEM_RESERVE) / stage_bytes(bn)) > 8
               ? 8
               : ((SMEM_LIMIT - SMEM_RESERVE) / stage_bytes(bn));
}
__host__ __device__ constexpr int mma_smem_bytes(int bn)
{
    return mma_stages(bn) * stage_bytes(bn) + SMEM_RESERVE;
}

// Device-side arguments of the tensor-core kernel (the two TMA descriptors
// travel as separate __grid_constant__ parameters).
struct MmaArgs {
    int M, N, K;
    int num_kb;            // ceil(K / BK)
    int tiles_m, tiles_n;  // per batch entry
    int tiles_per_batch;
    int batch;
    int split_k;           // K slices per output tile (1 = no split)
    int total_units;       // batch * tiles_per_batch * split_k
    int group_m;           // rasterisation band height, in tile rows
    int a_kmajor, b_kmajor;
    int a_3d, b_3d;        // 3-D descriptors: the batch index is the third coordinate
    uint32_t idesc;        // tcgen05 instruction descriptor
    float alpha, beta;
    void *C;
    long long ldc, stride_c;
    int c_dtype;           // TC_F16 / TC_BF16 / TC_F32
    int c_vec_ok;          // 16-byte vector stores allowed on C
    float *ws;             // split-K partial tiles
    unsigned *tickets;     // split-K arrival counters (zero between launches)
    unsigned *status;      // device status word (0 = fine)
    unsigned long long timeout_ns;
};

struct MmaLaunch {
    int bn;
    int grid;
    CUtensorMap tmA, tmB;
    MmaArgs args;
};

cudaError_t launch_mma(const MmaLaunch &L, cudaStream_t st);

// fp32 FFMA kernel (exact fp32, ascending-k fused multiply-add chain)
struct FfmaArgs {
    int M, N, K;
    int batch;
    int ta, tb;
    const float *A, *B;
    float *C;
    long long lda, ldb, ldc;
    long long stride_a, stride_b, stride_c;
    float alpha, beta;
};
enum FfmaTile { FFMA_SMALL = 0, FFMA_LARGE = 1 };
cudaError_t launch_ffma(const FfmaArgs &a, int tile, cudaStream_t st);

// Copy a strided batch of 16-bit matrices (rows x cols, leading dimension
// ld_src) into a buffer with leading dimension ld_dst (a multiple of 8) and a
// 16-byte aligned base, so that TMA can read it.
struct PackArgs {
    const uint16_t *src;
    uint16_t *dst;
    long long rows, cols, ld_src, ld_dst, stride_src, stride_dst;
    int batch;
};
cudaError_t launch_pack(const PackArgs &p, cudaStream_t st);

}  // namespace tc
