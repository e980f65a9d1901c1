/*
 * tcgemm -- GEMM for GB300 (sm_103a): C = alpha * op(A) @ op(B) + beta * C.
 *
 * The operation is the one defined on the tensorcore gemm.md page, section
 * "Surface": BLAS row-major layout, C[M,N] = alpha * A[M,K] @ B[K,N] +
 * beta * C[M,N], with optional transposes and leading dimensions that
 * default to row-major contiguous when 0.  The descriptor below keeps that
 * page's field list.  The async/stream and batched calls follow the same
 * page's section "Async, batched, and streams"; the validation order (checked
 * sizes, non-zero dims, finite scalars, no overlap, nothing launched on
 * error) follows the tessl architecture.md sections "GEMM Pipeline & Kernel
 * Selection" and "The Kernel Library and the nn Boundary".
 *
 * Conventions shared by every call:
 *   - Matrices are row-major.  op(A) is A stored [M,K] (lda >= K), or, with
 *     transpose_a, A stored [K,M] (lda >= M).  op(B) is B stored [K,N]
 *     (ldb >= N), or, with transpose_b, B stored [N,K] (ldb >= K) -- the
 *     layout of a linear layer's weight (phobos matmul page, "matmul_t").
 *     C is stored [M,N] (ldc >= N).  Leading dimensions count ELEMENTS;
 *     0 means contiguous.
 *   - A, B and C are DEVICE pointers (except tc_gemm_host) owned by the
 *     caller; they must stay valid until the work completes (tc_stream_sync
 *     for the async calls).  The library never frees caller memory.
 *   - Types: a_dtype == b_dtype in {TC_F16, TC_BF16, TC_F32};
 *     accum_dtype == TC_F32; c_dtype == a_dtype or TC_F32.  f16/bf16 inputs
 *     run on the tcgen05 tensor cores; f32 inputs run on FFMA CUDA cores in
 *     exact fp32 (never TF32).
 *   - beta == 0 means C is not read (NaN/Inf in C do not propagate).
 *     alpha == 0 is not special-cased.  The output is rounded once,
 *     round-to-nearest-even, from the fp32 value alpha*acc + beta*C_old.
 *   - Results are bitwise deterministic run to run for every variant,
 *     including split-K.
 *   - Errors: every call returns a tc_status_t and never aborts or traps.
 *     On any error detected before launch, nothing is enqueued and C is
 *     untouched.  A raw-pointer ABI cannot check buffer capacity; the
 *     Python binding checks capacity in elements.  Failures on the device
 *     surface at tc_stream_sync / the synchronous call.
 */
#ifndef TCGEMM_H
#define TCGEMM_H

#include <stdbool.h>
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* TC_I8 / TC_I32: operands and accumulator of tc_gemm_i8_dequant; TC_I8
 * also the weight type of tc_gemm_q8_weight. */
typedef enum { TC_F16 = 1, TC_BF16 = 2, TC_F32 = 3, TC_I8 = 4, TC_I32 = 5 } tc_dtype_t;

typedef enum {
    TC_OK = 0,
    TC_ERR_NULL = 1,               /* a required pointer is NULL */
    TC_ERR_DIM = 2,                /* M, N or K outside [1, 2^31-1]; batch < 1 */
    TC_ERR_LD = 3,                 /* a leading dimension below its minimum, or negative */
    TC_ERR_DTYPE = 4,              /* unsupported dtype combination */
    TC_ERR_SCALAR = 5,             /* alpha or beta not finite */
    TC_ERR_OVERLAP = 6,            /* C's byte range overlaps A's or B's */
    TC_ERR_OVERFLOW = 7,           /* an element or byte count overflows int64 */
    TC_ERR_ALIGN_UNSUPPORTED = 8,  /* only from tc_gemm_splitk_noalloc: operands TMA cannot read in place */
    TC_ERR_CUDA = 9,               /* a CUDA runtime error (launch, copy, no device) */
    TC_ERR_DEVICE_TIMEOUT = 10,    /* a kernel's bounded wait expired; it stopped early */
    TC_ERR_STRIDE = 11,            /* batched: negative stride */
    TC_ERR_VARIANT = 12,           /* a forced variant cannot serve this problem */
    TC_ERR_SCRATCH = 13,           /* tc_gemm_splitk_noalloc: more scratch than its static buffer holds */
    TC_ERR_EPILOGUE = 14,          /* fused epilogue: unknown activation, or f32 operands (see tc_gemm_epilogue) */
    TC_ERR_LAYOUT = 15             /* transpose flags the call does not support (tc_gemm_q8_weight) */
} tc_status_t;

/* tensorcore gemm.md, "Surface": the GEMM descriptor, field for field. */
typedef struct {
    int32_t M, N, K;
    tc_dtype_t a_dtype, b_dtype, c_dtype, accum_dtype;
    bool transpose_a, transpose_b;
    float alpha, beta;
    int32_t lda, ldb, ldc;
} tc_gemm_desc;

/* tensorcore gemm.md, "Async, batched, and streams": same-shape batch with
 * element strides between consecutive matrices (stride 0 = the same matrix
 * for every batch entry, allowed for A and B only). */
typedef struct {
    tc_gemm_desc base;
    int32_t batch;
    int64_t stride_a, stride_b, stride_c;
} tc_gemm_batched_desc;

/* tessl architecture.md, "Fused Epilogue": the operation
 *   C = activation(alpha * op(A) @ op(B) + beta * C_prev + bias)
 * computed in fp32 while the accumulator is on chip, with one rounding to
 * c_dtype at the end.  `bias` is a DEVICE pointer to N values of c_dtype,
 * one per output column (the page's row-stride-0 view: the same value for
 * every row), or NULL for no bias; it must not overlap C.  GeluTanh is
 * 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))). */
typedef enum { TC_ACT_NONE = 0, TC_ACT_GELU_TANH = 1 } tc_activation_t;
typedef struct {
    const void *bias;
    tc_activation_t activation;
} tc_epilogue;

typedef struct tc_ctx tc_ctx;
typedef struct tc_stream tc_stream;

/* tensorcore gemm.md, "Async, batched, and streams": every call there takes
 * a `ctx` as its first argument; the page does not print how one is made,
 * so the constructor and destructor are this library's own.
 * Create a context on CUDA device `device` (it becomes current for the
 * calling thread).  The context owns the TMA descriptor encoder, a default
 * stream and a device status word.  Returns TC_ERR_CUDA when no usable
 * device exists.  *out is NULL on error. */
tc_status_t tc_ctx_create(tc_ctx **out, int device);
/* Waits for the default stream, then frees everything the context owns
 * (never caller memory).  NULL is a no-op. */
void tc_ctx_destroy(tc_ctx *ctx);

/* tensorcore gemm.md, "Async, batched, and streams": a stream on which
 * tc_gemm_async enqueues work; only tc_stream_sync waits for it.  Each
 * stream owns its own workspace (split-K partials, repacked operands), so
 * work on different streams never shares scratch memory.  Stream order is
 * kept: most of the library's kernels are launched as programmatic
 * dependents of the kernel before them on the stream, so their set-up may
 * overlap its last blocks, but each waits for that kernel to complete
 * before it reads or writes any operand.  They also signal
 * griddepcontrol.launch_dependents early, so a caller's own kernel launched
 * after them with programmatic stream serialisation must wait
 * (cudaGridDependencySynchronize) before it reads their results; ordinary
 * launches, copies and events are ordered as usual (build addition: the
 * pages do not describe launches). */
tc_status_t tc_stream_create(tc_ctx *ctx, tc_stream **out);
/* Wrap an existing cudaStream_t (e.g. PyTorch's current stream); the
 * library does not destroy the wrapped stream. */
tc_status_t tc_stream_wrap(tc_ctx *ctx, void *cuda_stream, tc_stream **out);
/* Wait for the stream's work; returns TC_ERR_DEVICE_TIMEOUT if a kernel
 * reported an expired wait, TC_ERR_CUDA on a CUDA error.  After
 * TC_ERR_DEVICE_TIMEOUT the contents of every C the stream's work wrote
 * since the previous sync are undefined (a kernel that stopped early may
 * have written part of a tile, or a sum of incomplete partials); the
 * stream and the context stay usable. */
tc_status_t tc_stream_sync(tc_stream *s);
/* The cudaStream_t behind the stream (for event timing by the caller). */
void *tc_stream_handle(tc_stream *s);
void tc_stream_destroy(tc_stream *s);

/* tensorcore gemm.md, "Surface": the synchronous GEMM, on the context's
 * default stream (returns when C is written). */
tc_status_t tc_gemm(tc_ctx *ctx, const tc_gemm_desc *d, const void *A, const void *B, void *C);
/* tensorcore gemm.md, "Async, batched, and streams": enqueue the GEMM on
 * stream s and return; the work is complete only after tc_stream_sync(s). */
tc_status_t tc_gemm_async(tc_ctx *ctx, const tc_gemm_desc *d, const void *A, const void *B,
                          void *C, tc_stream *s);
/* Same-shape batch: matrix i is at A + i*stride_a (elements), etc.  One
 * launch covers every batch entry. */
tc_status_t tc_gemm_batched(tc_ctx *ctx, const tc_gemm_batched_desc *bd, const void *A,
                            const void *B, void *C);
tc_status_t tc_gemm_batched_async(tc_ctx *ctx, const tc_gemm_batched_desc *bd, const void *A,
                                  const void *B, void *C, tc_stream *s);
/* This library's addition for the ragged batch (no page prints a grouped
 * call; the tessl architecture.md "GEMM Pipeline & Kernel Selection" chart
 * routes ragged edges to bounds-checked slices): n independent problems,
 * each with its own descriptor and device pointers, enqueued on s.  All
 * descriptors are validated before anything is enqueued; f16/bf16 problems
 * share one persistent tensor-core launch per 64 problems, f32 problems run
 * one by one on the exact path. */
tc_status_t tc_gemm_grouped_async(tc_ctx *ctx, int n, const tc_gemm_desc *d,
                                  const void *const *A, const void *const *B, void *const *C,
                                  tc_stream *s);
/* GEMM with the fused bias + activation epilogue (tc_epilogue above); the
 * same kernels, tiles, split-K and determinism as tc_gemm.  Refused with
 * TC_ERR_EPILOGUE, nothing enqueued, for an unknown activation and for f32
 * operands: the exact-fp32 kernel accumulates in registers per output with
 * no separate epilogue to fuse into, and the page refuses that path rather
 * than falling back to separate passes.  TC_ERR_NULL when epi is NULL,
 * TC_ERR_OVERLAP when the bias overlaps C. */
tc_status_t tc_gemm_epilogue(tc_ctx *ctx, const tc_gemm_desc *d, const tc_epilogue *epi, const void *A,
                             const void *B, void *C);
tc_status_t tc_gemm_epilogue_async(tc_ctx *ctx, const tc_gemm_desc *d, const tc_epilogue *epi,
                                   const void *A, const void *B, void *C, tc_stream *s);

/* Relaxed fp32 (tessl architecture.md, "GEMM Pipeline & Kernel Selection":
 * a relaxed precision mode beside f32-exact): fp32 A and B (a_dtype ==
 * b_dtype == TC_F32, so c_dtype == TC_F32) on the bf16 tensor cores.  Each
 * value is split into two bf16 parts, x = hi + lo (+ less than 2^-16 |x|),
 * and the three products hi*hi + hi*lo + lo*hi are summed by one tensor-core
 * GEMM over 3K: every product is exact in fp32, so the result meets the
 * 1e-4 * sum_k |a b| bound of the non-exact paths, at the bf16 rate divided
 * by three (plus one pass that writes the split operands into a per-stream
 * buffer the library owns).  Not bit-compatible with the exact path;
 * deterministic run to run.  epi (may be NULL) adds the fused epilogue,
 * which the exact path refuses.  TC_ERR_DTYPE for non-f32 operands. */
tc_status_t tc_gemm_f32_relaxed(tc_ctx *ctx, const tc_gemm_desc *d, const tc_epilogue *epi, const void *A,
                                const void *B, void *C);
tc_status_t tc_gemm_f32_relaxed_async(tc_ctx *ctx, const tc_gemm_desc *d, const tc_epilogue *epi,
                                      const void *A, const void *B, void *C, tc_stream *s);

/* Integer GEMM with per-column dequantisation (tessl architecture.md,
 * "Integer GEMM"):
 *   acc[m, n] = sum_k op(A)[m, k] * op(B)[k, n]   (int8 x int8, exact)
 *   C[m, n]   = alpha * (acc[m, n] * col_scale[n]) + beta * C_old[m, n]
 * The descriptor has a_dtype == b_dtype == TC_I8, accum_dtype == TC_I32,
 * c_dtype == TC_F32 (TC_ERR_DTYPE otherwise); col_scale is a DEVICE pointer
 * to N floats (TC_ERR_NULL if NULL; it must not overlap C).  K > 131072 is
 * refused (TC_ERR_DIM): past it a full-range sum can leave int32.  The
 * accumulation is exact: operands are widened to bf16 (exact for int8) in
 * a per-stream buffer the library owns, the tensor cores sum at most 1024
 * products per K slice in fp32 (below 2^24, exact), and the slices are
 * added as 64-bit integers; the result is rounded once to fp32 and once by
 * the scale (and alpha, beta).  Deterministic run to run. */
tc_status_t tc_gemm_i8_dequant(tc_ctx *ctx, const tc_gemm_desc *d, const float *col_scale, const void *A,
                               const void *B, void *C);
tc_status_t tc_gemm_i8_dequant_async(tc_ctx *ctx, const tc_gemm_desc *d, const float *col_scale,
                                     const void *A, const void *B, void *C, tc_stream *s);

/* int8-weight product (Foundry metal.md, "Custom Compute Kernels":
 * fm_sgemm_q8(X[M,K], W_q8[N,K], scales[N]) and its M = 1 form
 * fm_matvec_q8; tensorcore gemm.md "Kernel variants": the M <= 4 GEMV over
 * Q8 weights with fp16 output):
 *   acc[m, n] = sum_k X[m, k] * W[n, k]          (fp32 accumulation)
 *   C[m, n]   = alpha * (acc[m, n] * scale[n]) + beta * C_old[m, n]
 * i.e. X times the transpose of the dequantised weight W[n, k] * scale[n],
 * one scale per weight row (per output column).  The descriptor has
 * a_dtype = X's type (TC_F16 or TC_BF16), b_dtype = TC_I8, accum_dtype =
 * TC_F32, c_dtype = a_dtype or TC_F32 (TC_ERR_DTYPE otherwise), and
 * transpose_a = false, transpose_b = true: X stored [M,K] (lda >= K), W
 * stored [N,K] (ldb >= K), the pages' layout (TC_ERR_LAYOUT otherwise).
 * X, W, C and scale (N floats, TC_ERR_NULL if NULL, must not overlap C)
 * are DEVICE pointers owned by the caller.  Up to 16 rows of X the int8
 * weights are streamed once and widened in registers (one launch, no
 * scratch); beyond, they are first widened exactly to X's type in a
 * per-stream buffer the library owns, then the tensor-core GEMM applies the
 * scales in its epilogue.  Any alignment and leading dimension; the same
 * validation, error and determinism rules as tc_gemm.  The Q4_0 / Q4_K
 * block formats and the Q8_0 block layout are not printed on the pages and
 * have no entry point. */
tc_status_t tc_gemm_q8_weight(tc_ctx *ctx, const tc_gemm_desc *d, const float *scale, const void *X,
                              const void *W, void *C);
tc_status_t tc_gemm_q8_weight_async(tc_ctx *ctx, const tc_gemm_desc *d, const float *scale, const void *X,
                                    const void *W, void *C, tc_stream *s);
/* Host-only: the validation tc_gemm_q8_weight runs first (no device needed). */
tc_status_t tc_gemm_q8_weight_validate(const tc_gemm_desc *d, const float *scale, const void *X, const void *W,
                                       const void *C);

/* Same GEMM with HOST operands: copies A and B (and C when beta != 0) to the
 * device, runs, copies C back and waits.  Device buffers are cached in the
 * context, so concurrent calls on one context run one after the other.
 * Pinned host memory gives full copy bandwidth. */
tc_status_t tc_gemm_host(tc_ctx *ctx, const tc_gemm_desc *d, const void *A_host,
                         const void *B_host, void *C_host);

/* Split-K GEMM that allocates nothing.  The paper has no counterpart to
 * this call; it exists for callers that cannot allocate device memory: code
 * in a process whose device memory is owned by another allocator with a
 * fixed budget (a framework's caching allocator, a plugin handed only its
 * inputs and outputs), and latency-critical paths that cannot afford the
 * device-wide synchronisation cudaMalloc and cudaFree imply.  It needs no
 * context either (creating one allocates).
 *
 * It runs the tensor-core kernel in its split-K form (128 x 128 output tiles,
 * K cut into `split` slices) followed by the reduction kernel that sums the
 * slices' fp32 partial tiles in slice order, so results are deterministic
 * and equal to tc_gemm's split-K variant with the same slice count.  The
 * partial tiles live in one file-scope device array of 16 MiB + 256 B that
 * every GPU which loads this library holds until the process exits.  Limit:
 * split * ceil(M/128) * ceil(N/128) * 64 KiB <= 16 MiB whenever split > 1,
 * else TC_ERR_SCRATCH (nothing is launched).  split = 0 picks the slice
 * count from the SM count (always within the limit on GB300).
 *
 * Arguments: d, A, B, C as for tc_gemm_async (device pointers, caller
 * owned); cuda_stream is a cudaStream_t (NULL = legacy default stream).
 * Only f16/bf16 operands (TC_ERR_DTYPE for f32), with 16-byte aligned bases
 * and leading dimensions that are multiples of 8 elements
 * (TC_ERR_ALIGN_UNSUPPORTED otherwise: repacking would need scratch sized
 * by the operands).  The call is asynchronous: it clears the array's status
 * word with cudaMemsetAsync and launches on cuda_stream; a device-side wait
 * timeout is not reported by this call, and when one happens the contents of
 * C are undefined (the reduction kernel then skips C: it may be partly
 * written by the slices of a single-slice call, or keep its old values).
 *
 * Every call, on any stream, shares the one array and it keeps the last
 * call's contents: calls whose kernels overlap on the GPU race and corrupt
 * each other's results; serialise them (one stream, or events).  The first
 * call on each device performs set-up (it looks up the array's device
 * address and the TMA encoder and sets the kernel's shared-memory limit);
 * make that first call before any stream capture.  That set-up is kept for
 * the life of the process: after cudaDeviceReset on a device, this entry
 * point must not be called again on that device. */
tc_status_t tc_gemm_splitk_noalloc(const tc_gemm_desc *d, const void *A, const void *B, void *C, int split,
                                   void *cuda_stream);

/* Host-only checks, no device needed: the same validation every call runs
 * first.  A, B, C are only compared as addresses (overlap), never read. */
tc_status_t tc_gemm_validate(const tc_gemm_desc *d, const void *A, const void *B, const void *C);
tc_status_t tc_gemm_batched_validate(const tc_gemm_batched_desc *bd, const void *A,
                                     const void *B, const void *C);
tc_status_t tc_gemm_epilogue_validate(const tc_gemm_desc *d, const tc_epilogue *epi, const void *A,
                                      const void *B, const void *C);
/* Host-only: the kernel variant the dispatcher would pick for this problem
 * on a GPU with num_sms SMs, written into buf (NUL-terminated, truncated to
 * len).  A, B, C are inspected for 16-byte alignment only. */
tc_status_t tc_gemm_plan(const tc_gemm_desc *d, const void *A, const void *B, const void *C,
                         int num_sms, char *buf, size_t len);

/* The variant and configuration of the last kernel this context launched
 * (tensorcore gemm.md "Fallback ladder": which path served the call). */
const char *tc_last_kernel(tc_ctx *ctx);
/* This library's test hook for the tessl architecture.md rule "nothing is
 * launched on error" (section "The Kernel Library and the nn Boundary"):
 * the number of kernels this context has launched; a refused call leaves it
 * unchanged. */
uint64_t tc_launch_count(tc_ctx *ctx);
const char *tc_status_string(tc_status_t st);

#ifdef __cplusplus
}
#endif
#endif /* TCGEMM_H */
