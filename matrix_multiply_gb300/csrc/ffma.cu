// fp32-exact GEMM on the FFMA CUDA cores (no TF32, no tensor cores).
//
// The tessl architecture.md "GEMM Pipeline & Kernel Selection" chart routes
// "f32 exact" NN work to its own small-tile kernel, and the phobos matmul
// page's "sgemm" kernel is the fp32 loop with the alpha/beta epilogue.  Here
// every output element is one fused multiply-add chain over k in ascending
// order, acc = fma(a_ik, b_kj, acc), followed by alpha*acc + beta*C_old:
// deterministic and never reassociated.
//
// Tiles are staged through shared memory (A transposed to [k][m], B as
// [k][n]) with register double buffering of the next K block; each thread
// owns a TM x TN register block with a strided row/column assignment so
// shared-memory reads are conflict-free.  Every layout (NN/TN/NT/TT), any
// leading dimension and ragged edges go through bounds-checked loads.
#include "internal.h"
#include "ptx.cuh"

#include <atomic>

namespace tc {
namespace {

template <int BM, int BN, int BK, int TM, int TN>
__global__ void __launch_bounds__(256) ffma_kernel(const FfmaArgs a)
{
    griddep_launch_dependents();     // launched as a programmatic dependent (see launch_dependent)
    griddep_wait();
    static_assert((BM / TM) * (BN / TN) == 256, "256 threads");
    static_assert((BM * BK) % 256 == 0 && (BN * BK) % 256 == 0, "tile loads");
    constexpr int LA = BM * BK / 256;   // A elements loaded per thread per K block
    constexpr int LB = BN * BK / 256;
    __shared__ float As[2][BK][BM + 4];
    __shared__ float Bs[2][BK][BN + 4];

    const int tid = threadIdx.x;
    const int tx = tid % (BN / TN);     // column group
    const int ty = tid / (BN / TN);     // row group
    const long long n0 = (long long)blockIdx.x * BN;
    const long long tiles_m = ((long long)a.M + BM - 1) / BM;

    for (int b = blockIdx.z; b < a.batch; b += gridDim.z)
    for (long long mt = blockIdx.y; mt < tiles_m; mt += gridDim.y) {
        const long long m0 = mt * BM;
        const float *A = a.A + (long long)b * a.stride_a;
        const float *B = a.B + (long long)b * a.stride_b;
        float *C = a.C + (long long)b * a.stride_c;

        // element e of the A tile: (m, k).  Consecutive threads walk the
        // stored-contiguous dimension so global loads coalesce.
        auto a_coord = [&](int e, int &m, int &k) {
            if (a.ta) { m = e % BM; k = e / BM; }      // stored [K,M]: m contiguous
            else      { k = e % BK; m = e / BK; }      // stored [M,K]: k contiguous
        };
        auto b_coord = [&](int e, int &k, int &n) {
            if (a.tb) { k = e % BK; n = e / BK; }      // stored [N,K]: k contiguous
            else      { n = e % BN; k = e / BN; }      // stored [K,N]: n contiguous
        };
        auto load_a = [&](long long kb, float (&ra)[LA]) {
#pragma unroll
            for (int i = 0; i < LA; ++i) {
                int m, k;
                a_coord(tid + i * 256, m, k);
                const long long gm = m0 + m, gk = kb + k;
                ra[i] = (gm < a.M && gk < a.K)
                            ? (a.ta ? A[gk * a.lda + gm] : A[gm * a.lda + gk])
                            : 0.0f;
            }
        };
        auto load_b = [&](long long kb, float (&rb)[LB]) {
#pragma unroll
            for (int i = 0; i < LB; ++i) {
                int k, n;
                b_coord(tid + i * 256, k, n);
                const long long gk = kb + k, gn = n0 + n;
                rb[i] = (gk < a.K && gn < a.N)
                            ? (a.tb ? B[gn * a.ldb + gk] : B[gk * a.ldb + gn])
                            : 0.0f;
            }
        };
        auto store_tiles = [&](int buf, const float (&ra)[LA], const float (&rb)[LB]) {
#pragma unroll
            for (int i = 0; i < LA; ++i) {
                int m, k;
                a_coord(tid + i * 256, m, k);
                As[buf][k][m] = ra[i];
            }
#pragma unroll
            for (int i = 0; i < LB; ++i) {
                int k, n;
                b_coord(tid + i * 256, k, n);
                Bs[buf][k][n] = rb[i];
            }
        };

        float acc[TM][TN];
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;

        float ra[LA], rb[LB];
        load_a(0, ra);
        load_b(0, rb);
        store_tiles(0, ra, rb);
        __syncthreads();

        int buf = 0;
        for (long long kb = 0; kb < a.K; kb += BK) {
            const bool more = kb + BK < a.K;
            if (more) {
                load_a(kb + BK, ra);
                load_b(kb + BK, rb);
            }
            const int kend = (int)min((long long)BK, a.K - kb);   // zero-padded beyond K, but stop the chain at K
            for (int kk = 0; kk < kend; ++kk) {
                float av[TM], bv[TN];
#pragma unroll
                for (int i = 0; i < TM; ++i) av[i] = As[buf][kk][ty + i * (BM / TM)];
#pragma unroll
                for (int j = 0; j < TN; ++j) bv[j] = Bs[buf][kk][tx + j * (BN / TN)];
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
            }
            if (more) {
                store_tiles(buf ^ 1, ra, rb);
                __syncthreads();
                buf ^= 1;
            }
        }

#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const long long gm = m0 + ty + i * (BM / TM);
            if (gm >= a.M) continue;
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                const long long gn = n0 + tx + j * (BN / TN);
                if (gn >= a.N) continue;
                float *c = C + gm * a.ldc + gn;
                const float r = a.alpha * acc[i][j];
                *c = (a.beta != 0.0f) ? fmaf(a.beta, *c, r) : r;
            }
        }
        __syncthreads();   // shared tiles are reused by the next tile
    }
}

// Large problems: 128 x 128 tiles, 256 threads, 8 x 8 outputs per thread as
// a 2 x 2 grid of 4 x 4 blocks (rows 4ty.. and 64 + 4ty.., columns 4tx..
// and 64 + 4tx..), so that every shared-memory read is one 16-byte load
// that 16 lanes share (A) or that covers 256 contiguous bytes (B).  The
// layouts are template parameters (no per-element branches); K steps of 16
// are fully unrolled; the next K block is loaded into registers (16-byte
// loads when VEC: aligned bases and leading dimensions that are multiples
// of 4) while the current one is multiplied.  Per output it is still one
// fmaf chain in ascending k (zero-filled operands past K add exact zeros).
template <bool TA, bool TB, bool VEC>
__global__ void __launch_bounds__(256, 2) ffma128_kernel(const FfmaArgs a)
{
    griddep_launch_dependents();     // launched as a programmatic dependent (see launch_dependent)
    griddep_wait();
    constexpr int BM = 128, BN = 128, BK = 16, LDS = 132;    // 528-byte rows keep 16-byte alignment
    __shared__ __align__(16) float As[2][BK][LDS];
    __shared__ __align__(16) float Bs[2][BK][LDS];
    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const long long n0 = (long long)blockIdx.x * BN;
    const long long tiles_m = ((long long)a.M + BM - 1) / BM;

    for (int b = blockIdx.z; b < a.batch; b += gridDim.z)
    for (long long mt = blockIdx.y; mt < tiles_m; mt += gridDim.y) {
        const long long m0 = mt * BM;
        const float *A = a.A + (long long)b * a.stride_a;
        const float *B = a.B + (long long)b * a.stride_b;
        float *C = a.C + (long long)b * a.stride_c;

        // four consecutive elements of a stored row starting at (r, c),
        // zero past the matrix (rows >= nr, columns >= nc)
        auto load4 = [&](const float *P, long long ld, long long r, long long c, long long nr, long long nc) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r >= nr) return v;
            const float *q = P + r * ld + c;
            if (VEC && c + 4 <= nc) return __ldg(reinterpret_cast<const float4 *>(q));
            if (c + 0 < nc) v.x = __ldg(q + 0);
            if (c + 1 < nc) v.y = __ldg(q + 1);
            if (c + 2 < nc) v.z = __ldg(q + 2);
            if (c + 3 < nc) v.w = __ldg(q + 3);
            return v;
        };
        // A tile (128 m x 16 k) and B tile (16 k x 128 n): 512 float4 each,
        // two per thread, along the stored-contiguous dimension
        float4 ra[2], rb[2];
        auto load_tiles = [&](long long k0) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int e = tid + 256 * i;
                if (TA) ra[i] = load4(A, a.lda, k0 + e / 32, m0 + (e % 32) * 4, a.K, a.M);   // [K][M]
                else    ra[i] = load4(A, a.lda, m0 + e / 4, k0 + (e % 4) * 4, a.M, a.K);    // [M][K]
                if (TB) rb[i] = load4(B, a.ldb, n0 + e / 4, k0 + (e % 4) * 4, a.N, a.K);    // [N][K]
                else    rb[i] = load4(B, a.ldb, k0 + e / 32, n0 + (e % 32) * 4, a.K, a.N);  // [K][N]
            }
        };
        auto store_tiles = [&](int buf) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int e = tid + 256 * i;
                if (TA) {
                    *reinterpret_cast<float4 *>(&As[buf][e / 32][(e % 32) * 4]) = ra[i];
                } else {
                    const int m = e / 4, k = (e % 4) * 4;
                    As[buf][k + 0][m] = ra[i].x;
                    As[buf][k + 1][m] = ra[i].y;
                    As[buf][k + 2][m] = ra[i].z;
                    As[buf][k + 3][m] = ra[i].w;
                }
                if (TB) {
                    const int n = e / 4, k = (e % 4) * 4;
                    Bs[buf][k + 0][n] = rb[i].x;
                    Bs[buf][k + 1][n] = rb[i].y;
                    Bs[buf][k + 2][n] = rb[i].z;
                    Bs[buf][k + 3][n] = rb[i].w;
                } else {
                    *reinterpret_cast<float4 *>(&Bs[buf][e / 32][(e % 32) * 4]) = rb[i];
                }
            }
        };

        float acc[8][8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

        load_tiles(0);
        store_tiles(0);
        __syncthreads();
        int buf = 0;
        for (long long k0 = 0; k0 < a.K; k0 += BK) {
            const bool more = k0 + BK < a.K;
            if (more) load_tiles(k0 + BK);
#pragma unroll
            for (int kk = 0; kk < BK; ++kk) {
                const float4 a0 = *reinterpret_cast<const float4 *>(&As[buf][kk][ty * 4]);
                const float4 a1 = *reinterpret_cast<const float4 *>(&As[buf][kk][64 + ty * 4]);
                const float4 b0 = *reinterpret_cast<const float4 *>(&Bs[buf][kk][tx * 4]);
                const float4 b1 = *reinterpret_cast<const float4 *>(&Bs[buf][kk][64 + tx * 4]);
                const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
            }
            if (more) {
                store_tiles(buf ^ 1);
                __syncthreads();
                buf ^= 1;
            }
        }

        // alpha/beta; 16-byte accesses of C where aligned and inside N
        const bool cvec = VEC && (a.ldc % 4 == 0) && ((reinterpret_cast<uintptr_t>(C) & 15u) == 0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const long long gm = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
            if (gm >= a.M) continue;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const long long gn = n0 + h * 64 + tx * 4;
                float *c = C + gm * a.ldc + gn;
                float v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] = a.alpha * acc[i][h * 4 + j];
                if (cvec && gn + 4 <= a.N) {
                    if (a.beta != 0.0f) {
                        const float4 o = *reinterpret_cast<const float4 *>(c);
                        v[0] = fmaf(a.beta, o.x, v[0]);
                        v[1] = fmaf(a.beta, o.y, v[1]);
                        v[2] = fmaf(a.beta, o.z, v[2]);
                        v[3] = fmaf(a.beta, o.w, v[3]);
                    }
                    *reinterpret_cast<float4 *>(c) = make_float4(v[0], v[1], v[2], v[3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (gn + j < a.N) c[j] = (a.beta != 0.0f) ? fmaf(a.beta, c[j], v[j]) : v[j];
                }
            }
        }
        __syncthreads();   // the shared tiles are refilled by the next tile
    }
}

// Small NN problems with 16-byte aligned rows (the pages' fp32 256^3 shape):
// 16 x 32 tiles, 128 threads, one row and four columns per thread.  A and B
// arrive in K chunks of 64 through a cp.async ring of SNBUF buffers (bytes
// past M, N or K read as zeros): SNBUF - 1 chunks are in flight before the
// first multiply-add, so a short K pays the load latency about once, and the
// first multiply-adds start after one chunk rather than after the whole K
// panel; every shared read is 16 bytes (four k of the thread's A row, four
// columns of a B row).  Per output one fmaf chain in ascending k.
constexpr int SBM = 16, SBN = 32, SKC = 64, SLDA = SKC + 4, SNBUF = 3;

__device__ __forceinline__ void cp_async16_f(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__global__ void __launch_bounds__(128) ffma_small_nn_kernel(const FfmaArgs a)
{
    griddep_launch_dependents();     // a dependent launched next may start its set-up
    griddep_wait();                  // (no-op: this kernel is launched in the ordinary way)
    __shared__ __align__(16) float As[SNBUF][SBM][SLDA];
    __shared__ __align__(16) float Bs[SNBUF][SKC][SBN];
    const int tid = threadIdx.x;
    const int tx = tid & 7, ty = tid >> 3;
    const long long n0 = (long long)blockIdx.x * SBN;
    const long long tiles_m = ((long long)a.M + SBM - 1) / SBM;
    const long long nchunk = ((long long)a.K + SKC - 1) / SKC;
    for (int b = blockIdx.z; b < a.batch; b += gridDim.z)
    for (long long mt = blockIdx.y; mt < tiles_m; mt += gridDim.y) {
        const long long m0 = mt * SBM;
        const float *A = a.A + (long long)b * a.stride_a;
        const float *B = a.B + (long long)b * a.stride_b;
        float *C = a.C + (long long)b * a.stride_c;
        // chunk c into buffer c % SNBUF: A 16 x 64 (2 pieces of 16 bytes a
        // thread), B 64 x 32 (4 pieces a thread)
        auto issue = [&](long long c) {
            const long long k0 = c * SKC;
            const int buf = (int)(c % SNBUF);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int e = tid + 128 * i;
                const int r = e >> 4, q = (e & 15) * 4;
                const long long gm = m0 + r, gk = k0 + q;
                const long long left = (gm < a.M) ? (a.K - gk) : 0;
                const uint32_t bytes = left >= 4 ? 16u : left > 0 ? (uint32_t)left * 4u : 0u;
                cp_async16_f((uint32_t)__cvta_generic_to_shared(&As[buf][r][q]), bytes ? A + gm * a.lda + gk : A,
                             bytes);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int e = tid + 128 * i;
                const int r = e >> 3, q = (e & 7) * 4;
                const long long gk = k0 + r, gn = n0 + q;
                const long long left = (gk < a.K) ? (a.N - gn) : 0;
                const uint32_t bytes = left >= 4 ? 16u : left > 0 ? (uint32_t)left * 4u : 0u;
                cp_async16_f((uint32_t)__cvta_generic_to_shared(&Bs[buf][r][q]), bytes ? B + gk * a.ldb + gn : B,
                             bytes);
            }
        };
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int i = 0; i < SNBUF - 1; ++i) {
            if (i < nchunk) issue(i);
            asm volatile("cp.async.commit_group;" ::: "memory");
        }
        for (long long c = 0; c < nchunk; ++c) {
            // chunk c + SNBUF - 1 into the buffer chunk c - 1 used (free since
            // the previous iteration's closing barrier), then wait for chunk c
            if (c + SNBUF - 1 < nchunk) issue(c + SNBUF - 1);
            asm volatile("cp.async.commit_group;" ::: "memory");
            asm volatile("cp.async.wait_group %0;" ::"n"(SNBUF - 1) : "memory");   // chunk c has landed
            __syncthreads();
            const int buf = (int)(c % SNBUF);
#pragma unroll
            for (int kk = 0; kk < SKC; kk += 4) {
                const float4 a4 = *reinterpret_cast<const float4 *>(&As[buf][ty][kk]);
                const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4 b4 = *reinterpret_cast<const float4 *>(&Bs[buf][kk + u][tx * 4]);
                    acc[0] = fmaf(av[u], b4.x, acc[0]);
                    acc[1] = fmaf(av[u], b4.y, acc[1]);
                    acc[2] = fmaf(av[u], b4.z, acc[2]);
                    acc[3] = fmaf(av[u], b4.w, acc[3]);
                }
            }
            __syncthreads();                                           // buffer free again
        }
        const long long gm = m0 + ty, gn = n0 + tx * 4;
        if (gm < a.M) {
            float *cp = C + gm * a.ldc + gn;
            float v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = a.alpha * acc[j];
            const bool vec = gn + 4 <= a.N && (a.ldc % 4) == 0 && ((reinterpret_cast<uintptr_t>(cp) & 15u) == 0);
            if (vec) {
                if (a.beta != 0.0f) {
                    const float4 o = *reinterpret_cast<const float4 *>(cp);
                    v[0] = fmaf(a.beta, o.x, v[0]);
                    v[1] = fmaf(a.beta, o.y, v[1]);
                    v[2] = fmaf(a.beta, o.z, v[2]);
                    v[3] = fmaf(a.beta, o.w, v[3]);
                }
                *reinterpret_cast<float4 *>(cp) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (gn + j < a.N) cp[j] = (a.beta != 0.0f) ? fmaf(a.beta, cp[j], v[j]) : v[j];
            }
        }
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();
    }
}

// Small problems: each CTA stages whole K panels (up to KC columns of A's
// 16 rows and KC rows of B's 32 columns) into shared memory with every load
// issued back to back, then runs the chains; one global-load latency per
// panel instead of one per 32-wide K block.  16 x 32 tiles, 256 threads, two
// outputs per thread.
constexpr int PBM = 16, PBN = 32;
constexpr int PANEL_SMEM = 96 * 1024;
constexpr int PANEL_KC = PANEL_SMEM / ((PBM + PBN) * 4);    // 512

__global__ void __launch_bounds__(256) ffma_panel_kernel(const FfmaArgs a)
{
    griddep_launch_dependents();     // launched as a programmatic dependent (see launch_dependent)
    griddep_wait();
    extern __shared__ float panel[];
    float *As = panel;                    // [KC][PBM]
    float *Bs = panel + PANEL_KC * PBM;   // [KC][PBN]
    const int tid = threadIdx.x;
    const int tx = tid % 16;              // columns tx and tx + 16
    const int ty = tid / 16;              // row ty
    const long long n0 = (long long)blockIdx.x * PBN;
    const long long tiles_m = ((long long)a.M + PBM - 1) / PBM;
    for (int b = blockIdx.z; b < a.batch; b += gridDim.z)
    for (long long mt = blockIdx.y; mt < tiles_m; mt += gridDim.y) {
        const long long m0 = mt * PBM;
        const float *A = a.A + (long long)b * a.stride_a;
        const float *B = a.B + (long long)b * a.stride_b;
        float *C = a.C + (long long)b * a.stride_c;
        float acc0 = 0.0f, acc1 = 0.0f;
        for (long long k0 = 0; k0 < a.K; k0 += PANEL_KC) {
            const int kc = (int)min((long long)PANEL_KC, a.K - k0);
            // A panel: PBM x kc; consecutive threads walk the stored-contiguous
            // dimension.  Loads go to registers 32 at a time before any
            // shared-memory store, so 32 loads are in flight per thread.
            const int na = PBM * kc, nb = PBN * kc;
            for (int e0 = tid; e0 < na; e0 += 32 * 256) {
                float r[32];
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    const int e = e0 + q * 256;
                    int m, k;
                    if (a.ta) { m = e % PBM; k = e / PBM; } else { k = e % kc; m = e / kc; }
                    const long long gm = m0 + m, gk = k0 + k;
                    r[q] = (e < na && gm < a.M) ? (a.ta ? A[gk * a.lda + gm] : A[gm * a.lda + gk]) : 0.0f;
                }
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    const int e = e0 + q * 256;
                    if (e >= na) break;
                    int m, k;
                    if (a.ta) { m = e % PBM; k = e / PBM; } else { k = e % kc; m = e / kc; }
                    As[k * PBM + m] = r[q];
                }
            }
            for (int e0 = tid; e0 < nb; e0 += 32 * 256) {
                float r[32];
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    const int e = e0 + q * 256;
                    int k, n;
                    if (a.tb) { k = e % kc; n = e / kc; } else { n = e % PBN; k = e / PBN; }
                    const long long gk = k0 + k, gn = n0 + n;
                    r[q] = (e < nb && gn < a.N) ? (a.tb ? B[gn * a.ldb + gk] : B[gk * a.ldb + gn]) : 0.0f;
                }
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    const int e = e0 + q * 256;
                    if (e >= nb) break;
                    int k, n;
                    if (a.tb) { k = e % kc; n = e / kc; } else { n = e % PBN; k = e / PBN; }
                    Bs[k * PBN + n] = r[q];
                }
            }
            __syncthreads();
            for (int k = 0; k < kc; ++k) {
                const float av = As[k * PBM + ty];
                acc0 = fmaf(av, Bs[k * PBN + tx], acc0);
                acc1 = fmaf(av, Bs[k * PBN + tx + 16], acc1);
            }
            __syncthreads();
        }
        const long long gm = m0 + ty;
        if (gm < a.M) {
            const float accs[2] = {acc0, acc1};
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const long long gn = n0 + tx + 16 * j;
                if (gn >= a.N) continue;
                float *c = C + gm * a.ldc + gn;
                const float r = a.alpha * accs[j];
                *c = (a.beta != 0.0f) ? fmaf(a.beta, *c, r) : r;
            }
        }
    }
}

}  // namespace

cudaError_t launch_ffma(const FfmaArgs &a, int tile, cudaStream_t st)
{
    if (tile == FFMA_PANEL && !a.ta && !a.tb &&
        ((reinterpret_cast<uintptr_t>(a.A) | reinterpret_cast<uintptr_t>(a.B)) & 15u) == 0 && a.lda % 4 == 0 &&
        a.ldb % 4 == 0 && a.stride_a % 4 == 0 && a.stride_b % 4 == 0) {
        const int zb = a.batch < 65535 ? a.batch : 65535;
        const long long ty = ((long long)a.M + SBM - 1) / SBM;
        dim3 grid((unsigned)(((long long)a.N + SBN - 1) / SBN), (unsigned)(ty < 65535 ? ty : 65535), zb);
        // an ordinary launch: as a dependent, the next grid's many small
        // CTAs would be placed early, crowding the few idle SMs (256^3:
        // 7.7 us a step against 6.7)
        ffma_small_nn_kernel<<<grid, 128, 0, st>>>(a);
        return cudaGetLastError();
    }
    if (tile == FFMA_PANEL) {
        static std::atomic<bool> configured[64] = {};
        int dev = 0;
        cudaGetDevice(&dev);
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (!configured[dev].load(std::memory_order_acquire)) {
            cudaError_t e =
                cudaFuncSetAttribute(ffma_panel_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PANEL_SMEM);
            if (e != cudaSuccess) return e;
            configured[dev].store(true, std::memory_order_release);
        }
        const int zb = a.batch < 65535 ? a.batch : 65535;
        const long long ty = ((long long)a.M + PBM - 1) / PBM;
        dim3 grid((unsigned)(((long long)a.N + PBN - 1) / PBN), (unsigned)(ty < 65535 ? ty : 65535), zb);
        return launch_dependent(ffma_panel_kernel, grid, dim3(256), PANEL_SMEM, st, 1u, a);
    }
    const int zb = a.batch < 65535 ? a.batch : 65535;
    if (tile == FFMA_LARGE) {
        const long long ty = ((long long)a.M + 127) / 128;
        dim3 grid((unsigned)(((long long)a.N + 127) / 128), (unsigned)(ty < 65535 ? ty : 65535), zb);
        // 16-byte loads need 16-byte aligned bases and row / batch strides
        const bool vec = ((reinterpret_cast<uintptr_t>(a.A) | reinterpret_cast<uintptr_t>(a.B)) & 15u) == 0 &&
                         a.lda % 4 == 0 && a.ldb % 4 == 0 && a.stride_a % 4 == 0 && a.stride_b % 4 == 0 &&
                         a.stride_c % 4 == 0;
        const int key = (a.ta ? 4 : 0) | (a.tb ? 2 : 0) | (vec ? 1 : 0);
        switch (key) {
        case 0: return launch_dependent(ffma128_kernel<false, false, false>, grid, dim3(256), 0, st, 1u, a);
        case 1: return launch_dependent(ffma128_kernel<false, false, true>, grid, dim3(256), 0, st, 1u, a);
        case 2: return launch_dependent(ffma128_kernel<false, true, false>, grid, dim3(256), 0, st, 1u, a);
        case 3: return launch_dependent(ffma128_kernel<false, true, true>, grid, dim3(256), 0, st, 1u, a);
        case 4: return launch_dependent(ffma128_kernel<true, false, false>, grid, dim3(256), 0, st, 1u, a);
        case 5: return launch_dependent(ffma128_kernel<true, false, true>, grid, dim3(256), 0, st, 1u, a);
        case 6: return launch_dependent(ffma128_kernel<true, true, false>, grid, dim3(256), 0, st, 1u, a);
        default: return launch_dependent(ffma128_kernel<true, true, true>, grid, dim3(256), 0, st, 1u, a);
        }
    } else {
        const long long ty = ((long long)a.M + 31) / 32;
        dim3 grid((unsigned)(((long long)a.N + 31) / 32), (unsigned)(ty < 65535 ? ty : 65535), zb);
        return launch_dependent(ffma_kernel<32, 32, 32, 2, 2>, grid, dim3(256), 0, st, 1u, a);
    }
}

}  // namespace tc
