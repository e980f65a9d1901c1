// Launch descriptions shared by the host API (api.cpp) and the kernels.
// Plain structs; no PyTorch types anywhere in the library.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <utility>

namespace tc {

// Launch `kern` as a programmatic dependent of the stream's previous kernel
// (clusters of `cluster` CTAs when above 1).  Its CTAs may be scheduled as
// soon as every CTA of that kernel has executed
// griddepcontrol.launch_dependents or exited, so the launch and the
// kernel's set-up overlap the previous kernel's last CTAs; every kernel
// launched this way runs griddepcontrol.wait -- which returns once the
// previous grid has completed and its memory operations are visible --
// before its first global memory access.  Behind anything but a kernel
// (a copy, an event, another stream's work) the launch is ordered as usual.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             unsigned cluster, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cluster > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Tile geometry of the tensor-core kernel.  Every output tile is BM rows by
// BN columns; the K loop steps BK elements (one 128-byte swizzle row of a
// 16-bit type) per pipeline stage.
constexpr int BM = 128;
constexpr int BK = 64;
constexpr int MMA_K = 16;                       // K of one kind::f16 tcgen05.mma
constexpr int MMA_THREADS = 192;                // 4 epilogue warps, TMA warp, MMA warp (plain GEMM kernels)
constexpr int SMEM_LIMIT = 232448;              // max dynamic shared memory per block
constexpr int EPI_STAGE_BYTES = 4096;           // one 32 x 32 output chunk (fp32 worst case)

// Epilogue warps: four (warp w reads TMEM lanes 32w..32w+31), or, for the
// fused bias/activation epilogue and for grouped launches (`epi` true),
// eight -- two per TMEM lane quarter, each taking every other 32-column
// chunk -- so that CUDA-core epilogue work takes half as long: the tail
// tile's, which no next tile hides, and the plain-store epilogue of ragged
// problems, which otherwise holds the accumulator longer than the next
// tile's K loop runs.  The one-CTA 192-wide tile keeps four (its fifth
// pipeline stage needs the space).
__host__ __device__ constexpr int epi_warps(int bn, int cg, bool epi) { return (epi && !(bn == 192 && cg == 1)) ? 8 : 4; }
__host__ __device__ constexpr int mma_threads(int bn, int cg, bool epi) { return (epi_warps(bn, cg, epi) + 2) * 32; }
// Epilogue staging per warp: with four warps two chunk buffers (one TMA
// store may still be reading the other), except for the 192-wide tiles,
// which keep one buffer so that one more pipeline stage fits (the one-CTA
// tile's 40 KB stages: a fifth; the pair's 28 KB: a seventh; their K loops
// are bound by the latency the ring covers and their shapes run a single
// wave, which drains once); with eight warps one buffer each.  The plain-store
// path's 32 x 32-float transpose buffer is one such buffer, so a warp's
// staging never overlaps another warp's (a launch may use both paths: C by
// plain stores, split-K partial tiles by TMA stores).  Buffers start at
// multiples of 1024 bytes, the alignment the swizzled TMA layouts assume
// (the swizzle uses the absolute shared address).
__host__ __device__ constexpr int epi_bufs(int bn, int cg, bool epi)
{
    return (epi_warps(bn, cg, epi) == 8 || bn == 192) ? 1 : 2;
}
__host__ __device__ constexpr int epi_warp_bytes(int bn, int cg, bool epi)
{
    return epi_warps(bn, cg, epi) == 8 ? EPI_STAGE_BYTES : epi_bufs(bn, cg, epi) == 1 ? 5120 : 8192;
}
__host__ __device__ constexpr int epi_smem(int bn, int cg, bool epi) { return epi_warps(bn, cg, epi) * epi_warp_bytes(bn, cg, epi); }

__host__ __device__ constexpr int smem_reserve(int bn, int cg, bool epi)   // alignment slack + barriers + epilogue staging
{
    return 1024 + 256 + epi_smem(bn, cg, epi);
}

// One pipeline stage of a CTA: its 128 rows of A and its share of B (all BN
// columns for a single CTA; BN/2 for each CTA of a pair running
// tcgen05.mma.cta_group::2 on a 256 x BN tile).
__host__ __device__ constexpr int stage_bytes(int bn, int cg) { return (BM + bn / cg) * BK * 2; }
__host__ __device__ constexpr int tmem_cols(int bn)
{
    return (2 * bn <= 128) ? 128 : (2 * bn <= 256) ? 256 : 512;
}
__host__ __device__ constexpr int mma_stages(int bn, int cg, bool epi = false)
{
    return ((SMEM_LIMIT - smem_reserve(bn, cg, epi)) / stage_bytes(bn, cg)) > 8
               ? 8
               : ((SMEM_LIMIT - smem_reserve(bn, cg, epi)) / stage_bytes(bn, cg));
}
__host__ __device__ constexpr int mma_smem_bytes(int bn, int cg, bool epi = false)
{
    return mma_stages(bn, cg, epi) * stage_bytes(bn, cg) + smem_reserve(bn, cg, epi);
}

// Device-side arguments of the tensor-core kernel (the two TMA descriptors
// travel as separate __grid_constant__ parameters).
struct MmaArgs {
    int M, N, K;
    int num_kb;            // ceil(K / BK)
    int tiles_m, tiles_n;  // per batch entry
    int tiles_per_batch;
    int batch;
    // Work units: output tiles in the linear (band-swizzled) order, each cut
    // into K slices.  Tiles [0, seg0_tiles) have seg0_split slices each, the
    // remaining tiles seg1_split slices each; unit u enumerates (tile, slice)
    // pairs in that order.  A tile with more than one slice parks its
    // partial sums in ws slot (u - split_base) and the last slice to finish
    // reduces them in slice order.
    int seg0_tiles, seg0_split, seg1_split;
    int split_base;
    int total_units;
    int group_m;           // rasterisation band height, in tile rows
    int a_kmajor, b_kmajor;
    int a_3d, b_3d;        // 3-D descriptors: the batch index is the third coordinate
    // MN-major operand read through a chunked 3-D descriptor (64 elements,
    // K rows, 64-element chunks): one copy brings a CTA's whole share of
    // the operand for a K block instead of one copy per 64-wide chunk
    int a_chunked, b_chunked;
    uint32_t idesc;        // tcgen05 instruction descriptor
    float alpha, beta;
    void *C;
    long long ldc, stride_c;
    int c_dtype;           // TC_F16 / TC_BF16 / TC_F32
    int c_vec_ok;          // 16-byte vector loads/stores allowed on C
    int c_tma;             // C is written by TMA stores through the third descriptor
    int c_3d;              // that descriptor is 3-D (batch index third)
    float *ws;             // split-K partial tiles (written through the fourth descriptor)
    unsigned *status;      // device status word (0 = fine)
    unsigned long long timeout_ns;
    int debug_drop_tfull;  // test hook: never signal the first tile's accumulator
    // fused epilogue: bias (N values of c_dtype, or null) and activation
    // (TC_ACT_*) applied after alpha/beta, before the one rounding; a
    // per-column scale (N floats, or null) applied to the accumulator before
    // alpha/beta (the int8 path's dequantisation)
    const void *bias;
    int act;
    const float *col_scale;
    int slice_kb;          // on-chip int8 accumulation: K blocks per exact slice
    // one-CTA tiles over fewer than BM rows of a K-major A: its copies carry
    // only the rows that exist (rounded up to 8) and a stage this many fewer
    // bytes; the tile's other rows hold stale data, which reaches only
    // output rows beyond M (never stored)
    int a_short_bytes;
};

struct MmaLaunch {
    int bn;
    int cg;      // CTAs per tile: 1, or 2 for a CTA pair (cluster of two)
    int i8acc;   // int8 slices summed in TMEM (BN = 128 only; args.slice_kb, col_scale)
    // split-K inside one launch: the args.seg0_split K slices of a tile form
    // one cluster and add their partial tiles through distributed shared
    // memory (BN 64 or 128, one CTA per unit: grid == args.total_units)
    int csplit;
    int grid;    // CTAs (a multiple of cg)
    CUtensorMap tmA, tmB, tmC, tmW;   // A, B, C and the split-K workspace
    MmaArgs args;
};

cudaError_t launch_mma(const MmaLaunch &L, cudaStream_t st);

// A group of independent problems in one persistent launch.  Every problem
// has its own TMA descriptors and epilogue fields; all share the kernel
// shape (BN, CTAs per tile) and take one K slice per tile.  Unit u (one
// output tile) belongs to the problem p with unit_begin[p] <= u <
// unit_begin[p + 1]; the table travels as a kernel parameter.
constexpr int GROUP_MAX = 64;
struct GroupInfo {
    int M, N, num_kb;
    int tiles_m, tiles_n;
    int unit_begin;
    int a_kmajor, b_kmajor;
    uint32_t idesc;
    int c_dtype, c_vec_ok, c_tma;
    float alpha, beta;
    void *C;
    long long ldc;
};
struct GroupTable {
    CUtensorMap tmA[GROUP_MAX], tmB[GROUP_MAX], tmC[GROUP_MAX];
    GroupInfo info[GROUP_MAX];
    int count;
};
// L.args carries the launch-wide fields (total_units, group_m, status,
// timeout); the per-problem ones come from the table.
cudaError_t launch_mma_grouped(const MmaLaunch &L, const GroupTable &g, cudaStream_t st);
// Largest number of CTA pairs of the BN-wide pair kernel that can be
// resident at once on the current device (0 if the pair kernel cannot run).
int max_active_pairs(int bn);
// Largest number of S-CTA clusters of the BN-wide cluster-split kernel
// resident at once on the current device (0 if such a cluster cannot run).
int max_active_csplit_clusters(int bn, int S);

// Split-K reduction: tiles [first_tile, first_tile + ntiles) each have S
// fp32 partial tiles (rows_per_tile x bn, row-major) at
// ws + ((tile - first_tile) * S + s) * rows_per_tile * bn.
struct ReduceArgs {
    const float *ws;
    int rows_per_tile, bn;
    int first_tile, ntiles, S;
    int tiles_m, tiles_n, tiles_per_batch, group_m;
    int M, N;
    float alpha, beta;
    void *C;
    long long ldc, stride_c;
    int c_dtype, c_vec_ok;
    const void *bias;      // fused epilogue, as in MmaArgs
    int act;
    const float *col_scale;
    int int_sum;           // the slices are integers: add them as 64-bit integers
    // a status word in device memory (or null): nonzero when one of the
    // GEMM's bounded waits expired, so some partial tiles were never
    // written; the reduction then leaves C alone
    const unsigned *status;
};
// One CTA of bn threads per 8 (or, for small reductions, 4) rows of a tile,
// 8 (4) columns per thread; c_vec_ok allows 16-byte accesses to C.
cudaError_t launch_reduce(const ReduceArgs &r, cudaStream_t st);

// Static scratch of the entry point that allocates nothing: split-K partial
// tiles (at most NOALLOC_PARTIAL_BYTES) and one status word.
constexpr size_t NOALLOC_PARTIAL_BYTES = size_t(16) << 20;
constexpr size_t NOALLOC_SCRATCH_BYTES = NOALLOC_PARTIAL_BYTES + 256;
struct NoallocScratch {
    float *partials;
    unsigned *status;
};
// Device addresses of the static scratch on the current device (looked up
// once per device).
cudaError_t noalloc_scratch(NoallocScratch *out);

// Skinny products (gemv.cu): Out = alpha * (X W^T) (* scale[w row]) +
// beta * Out_old for X with at most GEMV_MAX_ROWS rows.  X is [rows_x, K]
// (f16 or bf16, row stride ldx elements), W is [rows_w, K] (X's type, or
// int8 when w_i8; row stride ldw elements); the output element of (X row
// i, W row j) is at C + i * c_sx + j * c_sw (elements of c_dtype).  The
// cluster kernel splits K across a cluster of ksplit CTAs (1, 2, 4 or 8)
// whose sums are added in rank order.
constexpr int GEMV_MAX_ROWS = 16;
struct GemvArgs {
    const void *X, *W;
    void *C;
    const float *scale;    // per W row, or null
    int rows_x, rows_w;
    long long K, ldx, ldw;
    long long c_sx, c_sw;
    int c_dtype;
    float alpha, beta;
    int x_vec, w_vec;      // 16-byte loads allowed: 16-byte aligned base and row stride
    int w_i8, x_bf16;
    int ksplit;
    // row-range kernel (16-byte aligned rows of X and W): `grid` persistent
    // CTAs (at most rows_w), CTA c owning W rows [c rows_w / grid,
    // (c + 1) rows_w / grid) -- or, with block_rows, whole 16-row blocks
    // [16 (c nb / grid), 16 ((c + 1) nb / grid)) of the nb = ceil(rows_w / 16)
    // blocks; ksplit is then unused
    int rowrange, grid, block_rows;
};
cudaError_t launch_gemv(const GemvArgs &a, cudaStream_t st);
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
enum FfmaTile { FFMA_SMALL = 0, FFMA_LARGE = 1, FFMA_PANEL = 2 };
cudaError_t launch_ffma(const FfmaArgs &a, int tile, cudaStream_t st);

// Relaxed fp32: a stored fp32 matrix (rows x cols, leading dimension ld_src)
// becomes three bf16 copies placed side by side along its K dimension (the
// columns when k_along_cols, else the rows), part j = hi or lo per
// parts[j] (0 = hi = bf16(x), 1 = lo = bf16(x - hi)), in a buffer with
// leading dimension ld_dst (a multiple of 64) and a 256-byte aligned base.
struct SplitArgs {
    const float *src;
    uint16_t *dst;
    long long rows, cols, ld_src, ld_dst;
    int k_along_cols;
    int parts[3];
};
cudaError_t launch_split(const SplitArgs &a, cudaStream_t st);

// int8 matrix (rows x cols, leading dimension ld_src) -> bf16, or f16 when
// to_f16 (both exact for int8), with leading dimension ld_dst (a multiple
// of 64) and a 256-byte aligned base.
struct WidenArgs {
    const int8_t *src;
    uint16_t *dst;
    long long rows, cols, ld_src, ld_dst;
    int to_f16;
};
cudaError_t launch_widen(const WidenArgs &a, cudaStream_t st);

// Copy a strided batch of 16-bit matrices (rows x cols, leading dimension
// ld_src) into a buffer with leading dimension ld_dst (a multiple of 64) and
// a 256-byte aligned base, so that TMA can read it.
struct PackArgs {
    const uint16_t *src;
    uint16_t *dst;
    long long rows, cols, ld_src, ld_dst, stride_src, stride_dst;
    int batch;
};
// Up to PACK_MAX such copies in one launch (block_begin is filled in by
// launch_pack: the first CTA of each copy, then the total).
constexpr int PACK_MAX = 128;
struct PackBatch {
    int count;
    long long block_begin[PACK_MAX + 1];
    PackArgs seg[PACK_MAX];
};
cudaError_t launch_pack(PackBatch &pb, cudaStream_t st);

}  // namespace tc
