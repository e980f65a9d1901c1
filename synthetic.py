"""Seeded synthetic inputs for the GEMM workloads.

This module only draws random numbers and lays them out as stored operands.
It holds none of the GEMM arithmetic: both the CUDA path (through the tests
and the benchmark) and the CPU oracle consume the tensors it returns, so the
two sides always see identical bits.

Recipe (the same for every workload):
  * a fresh ``torch.Generator('cpu').manual_seed(seed)`` per workload (and,
    for the square sweep, per size);
  * operands are drawn in the order A, then B, then C (when C is pre-filled),
    each directly in its *stored* shape: A is [M,K], or [K,M] when
    ``transpose_a``; B is [K,N], or [N,K] when ``transpose_b``; C is [M,N];
  * values are drawn as fp32 -- ``uniform[-1,1]`` as ``2*rand-1`` and
    ``normal(0,s)`` as ``s*randn`` -- then converted to the storage dtype with
    PyTorch's round-to-nearest-even cast.

The workloads follow the tensorcore gemm.md "Measured perf" shapes and the
tessl architecture.md "Round 2 Evolutions" table (square NN, TN/NT weight
gradient shapes, split-K and narrow-N).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32, "i8": torch.int8}


@dataclass
class Problem:
    """One GEMM problem: C[M,N] = alpha*op(A)@op(B) + beta*C (row-major)."""

    M: int
    N: int
    K: int
    ab_dtype: str           # "f16" | "bf16" | "f32" (A and B share it)
    c_dtype: str            # "f16" | "bf16" | "f32"
    transpose_a: bool = False
    transpose_b: bool = False
    alpha: float = 1.0
    beta: float = 0.0
    A: torch.Tensor | None = field(default=None, repr=False)
    B: torch.Tensor | None = field(default=None, repr=False)
    C: torch.Tensor | None = field(default=None, repr=False)   # C_old (input)

    @property
    def layout(self) -> str:
        return ("T" if self.transpose_a else "N") + ("T" if self.transpose_b else "N")

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


def _draw(gen: torch.Generator, shape, dist: str, scale: float) -> torch.Tensor:
    if dist == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    if dist == "normal":
        return torch.randn(shape, generator=gen, dtype=torch.float32) * scale
    if dist == "int":
        # integer-valued entries in [-scale, scale]
        s = int(scale)
        return torch.randint(-s, s + 1, shape, generator=gen).to(torch.float32)
    raise ValueError(dist)


def make_problem(M, N, K, ab_dtype, c_dtype, *, transpose_a=False, transpose_b=False,
                 alpha=1.0, beta=0.0, seed=0, dist="uniform", scale=1.0,
                 c_fill="zero", gen: torch.Generator | None = None,
                 lda=0, ldb=0, ldc=0) -> Problem:
    """Draw one problem's operands.  ``gen`` continues an existing stream
    (used by the ragged batch); otherwise a fresh generator seeded ``seed``.

    A non-zero ``lda/ldb/ldc`` pads the stored rows to that many elements
    (the padding holds random values as well, so a kernel that reads past
    the logical row shows up as a parity failure)."""
    g = gen if gen is not None else torch.Generator("cpu").manual_seed(seed)
    dt_ab, dt_c = DTYPES[ab_dtype], DTYPES[c_dtype]
    a_rows, a_cols = (K, M) if transpose_a else (M, K)
    b_rows, b_cols = (N, K) if transpose_b else (K, N)
    A = _draw(g, (a_rows, max(a_cols, lda)), dist, scale).to(dt_ab)
    B = _draw(g, (b_rows, max(b_cols, ldb)), dist, scale).to(dt_ab)
    if c_fill == "zero":
        C = torch.zeros((M, max(N, ldc)), dtype=dt_c)
    elif c_fill == "uniform":
        C = _draw(g, (M, max(N, ldc)), "uniform", 1.0).to(dt_c)
    elif c_fill == "nan":
        C = torch.full((M, max(N, ldc)), float("nan"), dtype=dt_c)
    elif c_fill == "int":
        C = _draw(g, (M, max(N, ldc)), "int", scale).to(dt_c)
    else:
        raise ValueError(c_fill)
    return Problem(M, N, K, ab_dtype, c_dtype, transpose_a, transpose_b, alpha, beta, A, B, C)


# --------------------------------------------------------------------------
# The named workloads.
# --------------------------------------------------------------------------

def fp32_nn_256() -> Problem:
    """fp32 NN 256^3, uniform[-1,1] from seed 0, C zero, alpha=1 beta=0."""
    return make_problem(256, 256, 256, "f32", "f32", seed=0, dist="uniform")


def bf16_nn_4096() -> Problem:
    """bf16 NN 4096^3, bf16 out, normal(0,1) from seed 1, alpha=1 beta=0."""
    return make_problem(4096, 4096, 4096, "bf16", "bf16", seed=1, dist="normal", scale=1.0)


def bf16_tn_nt_4096x8192(layout: str) -> Problem:
    """bf16 M=N=4096 K=8192, fp32 out, alpha=0.5 beta=1, C uniform[-1,1],
    inputs normal(0,0.02) from seed 2.  ``layout`` is "TN" (A stored [K,M])
    or "NT" (B stored [N,K])."""
    assert layout in ("TN", "NT")
    return make_problem(4096, 4096, 8192, "bf16", "f32", transpose_a=(layout == "TN"),
                        transpose_b=(layout == "NT"), alpha=0.5, beta=1.0, seed=2,
                        dist="normal", scale=0.02, c_fill="uniform")


def bf16_tn_splitk_256x16384() -> Problem:
    """bf16 TN M=N=256 K=16384 (weight-gradient shape), fp32 out, normal(0,1), seed 3."""
    return make_problem(256, 256, 16384, "bf16", "f32", transpose_a=True, seed=3,
                        dist="normal", scale=1.0)


def fp16_nn_narrow_8192x384x4096() -> Problem:
    """fp16 NN M=8192 N=384 K=4096, fp16 out, normal(0,1) from a fresh seed-3 generator."""
    return make_problem(8192, 384, 4096, "f16", "f16", seed=3, dist="normal", scale=1.0)


SQUARE_SIZES = (256, 512, 1024, 2048, 4096, 8192)


def fp16_nn_square(n: int) -> Problem:
    """fp16 NN n^3, fp16 out, uniform[-1,1], fresh seed-4 generator per size."""
    return make_problem(n, n, n, "f16", "f16", seed=4, dist="uniform")


def ragged_shapes(count: int = 64, lo: int = 1, hi: int = 3000, seed: int = 4):
    """The (M,N,K) triples of the ragged batch, drawn first from a fresh generator."""
    g = torch.Generator("cpu").manual_seed(seed)
    mnk = torch.randint(lo, hi + 1, (count, 3), generator=g)
    return g, [tuple(int(v) for v in row) for row in mnk]


def fp16_ragged(count: int = 64, lo: int = 1, hi: int = 3000, seed: int = 4):
    """64 independent fp16 NN problems, M,N,K ~ U[1,3000], contiguous, uniform[-1,1]."""
    g, shapes = ragged_shapes(count, lo, hi, seed)
    return [make_problem(M, N, K, "f16", "f16", gen=g, dist="uniform") for (M, N, K) in shapes]


# The fused bias + GELU epilogue (tessl architecture.md, "Fused Epilogue"):
# the page times 512^3, 1024^3 and 2048x2048x512 with bf16 operands.
EPILOGUE_SHAPES = ((512, 512, 512), (1024, 1024, 1024), (2048, 2048, 512))


def bf16_epilogue(M: int, N: int, K: int, seed: int = 5):
    """bf16 NN, bf16 out, alpha=1 beta=0, A and B normal(0,1) then the bias
    (N values, normal(0,1), bf16) from the same fresh generator.  Returns
    (problem, bias)."""
    g = torch.Generator("cpu").manual_seed(seed)
    p = make_problem(M, N, K, "bf16", "bf16", gen=g, dist="normal", scale=1.0)
    bias = _draw(g, (N,), "normal", 1.0).to(torch.bfloat16)
    return p, bias


# The GEMV / small-M decode shape (tensorcore gemm.md: "M <= 4 GEMV", fp16
# out, "the synthetic 7B decode shape"): activations x[M, K] times a weight
# W stored [N, K] (transpose_b), with the layer sizes of a 7B model (hidden
# 4096, MLP 11008).
DECODE_SHAPES = ((1, 4096, 4096), (4, 11008, 4096), (4, 4096, 11008))


def f16_decode(M: int, N: int, K: int, seed: int = 6) -> Problem:
    """fp16 x[M, K] @ W[N, K]^T, fp16 out, normal(0,1) from a fresh generator."""
    return make_problem(M, N, K, "f16", "f16", transpose_b=True, seed=seed, dist="normal")


def fp32_nn_4096() -> Problem:
    """fp32 NN 4096^3, fp32 out, uniform[-1,1] from a fresh seed-7 generator
    (the exact and the relaxed fp32 paths at the headline size)."""
    return make_problem(4096, 4096, 4096, "f32", "f32", seed=7, dist="uniform")


# The int8 GEMM with per-column dequantisation (tessl architecture.md,
# "Integer GEMM"): full-range int8 operands, fp32 output.

def i8_problem(M, N, K, *, transpose_a=False, transpose_b=False, alpha=1.0, beta=0.0, seed=0,
               c_fill="zero") -> Problem:
    """int8 A and B uniform over [-128, 127] (drawn A then B then C, in their
    stored shapes), fp32 C."""
    g = torch.Generator("cpu").manual_seed(seed)
    A = torch.randint(-128, 128, (K, M) if transpose_a else (M, K), generator=g).to(torch.int8)
    B = torch.randint(-128, 128, (N, K) if transpose_b else (K, N), generator=g).to(torch.int8)
    C = torch.zeros(M, N) if c_fill == "zero" else _draw(g, (M, N), "uniform", 1.0)
    return Problem(M, N, K, "i8", "f32", transpose_a, transpose_b, alpha, beta, A, B, C)


def i8_dequant_4096():
    """int8 NN 4096^3 with per-column scales uniform in [0, 1e-3) drawn after
    A and B (seed 8).  Returns (problem, scale)."""
    p = i8_problem(4096, 4096, 4096, seed=8)
    scale = torch.rand(4096, generator=torch.Generator("cpu").manual_seed(9)) * 1e-3
    return p, scale



# The int8-weight product (Foundry metal.md, "Custom Compute Kernels":
# fm_sgemm_q8(X[M,K], W_q8[N,K], scales[N]); tensorcore gemm.md "Kernel
# variants": the M <= 4 GEMV over Q8 weights with fp16 output), at the
# decode shapes above.  The pages give no distributions: the activations are
# normal(0,1) rounded to the half type, the weights uniform over the full
# int8 range, and the per-row scales uniform in [0.5e-3, 1.5e-3) (the scale
# of a row of normal(0,0.02) weights quantised to 127 levels).

def q8_weight_problem(M, N, K, x_dtype="f16", c_dtype="f16", *, alpha=1.0, beta=0.0, seed=10,
                      c_fill="zero", x_dist="normal", ldx=0, ldw=0):
    """X [M,K] (x_dtype), W int8 stored [N,K] (transpose_b), then the N
    scales, then C when pre-filled, drawn in that order from one fresh
    generator.  Returns (problem, scale); problem.A = X, problem.B = W."""
    g = torch.Generator("cpu").manual_seed(seed)
    X = _draw(g, (M, max(K, ldx)), x_dist, 4.0 if x_dist == "int" else 1.0).to(DTYPES[x_dtype])
    W = torch.randint(-128, 128, (N, max(K, ldw)), generator=g).to(torch.int8)
    scale = torch.rand(N, generator=g) * 1e-3 + 0.5e-3
    if c_fill == "zero":
        C = torch.zeros(M, N, dtype=DTYPES[c_dtype])
    else:
        C = _draw(g, (M, N), "uniform", 1.0).to(DTYPES[c_dtype])
    p = Problem(M, N, K, x_dtype, c_dtype, False, True, alpha, beta, X, W, C)
    return p, scale


def q8_decode(M: int, N: int, K: int, seed: int = 10):
    """fp16 x[M, K] @ (W_q8[N, K] * scale[n])^T, fp16 out (the decode shapes)."""
    return q8_weight_problem(M, N, K, "f16", "f16", seed=seed)


def signed_permutation(n: int, seed: int, dtype=torch.float32):
    """A signed permutation matrix P[n, n] (column j holds s_j = +-1 at row
    perm[j], zeros elsewhere; in ``dtype``) from a fresh generator, with perm
    and s as integer arrays.  X @ P is then a signed permutation of X's columns:
    exact in every dtype, so a chain of such products can be checked value
    for value however long it is."""
    g = torch.Generator("cpu").manual_seed(seed)
    perm = torch.randperm(n, generator=g)
    s = torch.randint(0, 2, (n,), generator=g) * 2 - 1
    P = torch.zeros(n, n, dtype=dtype)
    P[perm, torch.arange(n)] = s.to(dtype)
    return P, perm.numpy(), s.numpy()
