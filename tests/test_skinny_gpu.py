"""Skinny products -- GEMMs with at most 16 rows on one side, the
decode-time GEMV shape of the tensorcore gemm.md page ("M <= 4 GEMV") --
against the CPU oracle on GB300, under the GEMM bound of tests/parity.py
(1e-4 * sum|ab| plus one output ulp), bitwise on integer data, and the fused
epilogue under tests/parity.bound_epilogue.  NT products (both operands
K-contiguous) run on the skinny-product kernel, which streams the larger
operand once; every other layout, the fused epilogue and batches run on the
tensor-core kernel (the short side padded inside a 128-row tile by TMA zero
fill, split-K when the tiles are few), which gemv=0 also forces for NT."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import parity
import synthetic

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import matrix_multiply_gb300 as tg
else:  # collected on CPU only to be deselected
    tg = None

LAYOUTS = [(False, False), (True, False), (False, True), (True, True)]
DT_PAIRS = [("bf16", "bf16"), ("bf16", "f32"), ("f16", "f16"), ("f16", "f32")]


@pytest.fixture(scope="module")
def ctx():
    c = tg.Context(0)
    yield c
    c.close()


@pytest.fixture
def force(monkeypatch):
    def set_(spec):
        if spec:
            monkeypatch.setenv("TC_FORCE_VARIANT", spec)
        else:
            monkeypatch.delenv("TC_FORCE_VARIANT", raising=False)
    return set_


def run(ctx, p, **ld):
    A, B, C = p.A.cuda(), p.B.cuda(), p.C.cuda()
    d = tg.make_desc(p.M, p.N, p.K, p.ab_dtype, p.c_dtype, transpose_a=p.transpose_a,
                     transpose_b=p.transpose_b, alpha=p.alpha, beta=p.beta,
                     lda=A.shape[1], ldb=B.shape[1], ldc=C.shape[1])
    tg.tc_gemm(ctx, d, A, B, C)
    return C.cpu()


def check(ctx, p, what=""):
    out = run(ctx, p)
    R, T = oracle.gemm(p)
    parity.check(oracle.decode(out)[:, : p.N], R, T, p.c_dtype, what=f"{what} {ctx.last_kernel}")


# (M, N, K): small M; small N (the transposed product); both small; K of one
# element, of a ragged 16-byte tail, and long enough to cut across CTAs
SHAPES = [(1, 1000, 77), (3, 4097, 3000), (8, 300, 1), (8, 2050, 9001), (4000, 5, 130), (777, 8, 4100),
          (1, 1, 1), (6, 7, 33)]


@pytest.mark.parametrize("spec", ["", "gemv=0"])
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("ab,c", DT_PAIRS)
@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_skinny_parity(ctx, force, spec, shape, ab, c, ta, tb):
    force(spec)
    M, N, K = shape
    p = synthetic.make_problem(M, N, K, ab, c, transpose_a=ta, transpose_b=tb, alpha=0.75, beta=0.5,
                               seed=M + 7 * N + K, dist="normal", c_fill="uniform")
    check(ctx, p, f"{ab}->{c} {p.layout} {shape}")


@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_skinny_integer_bitwise(ctx, ta, tb):
    """Integer entries: every partial sum is an integer below 2^24, so the
    fp32 sums are exact whatever the split of K."""
    for (M, N, K) in [(4, 3000, 4096), (2500, 3, 4096), (8, 129, 100)]:
        p = synthetic.make_problem(M, N, K, "bf16", "f32", transpose_a=ta, transpose_b=tb, alpha=1.0, beta=1.0,
                                   seed=K + M, dist="int", scale=4.0, c_fill="int")
        out = run(ctx, p)
        R, _ = oracle.gemm(p)
        assert np.array_equal(out.numpy().astype(np.float64), R), (M, N, K, ctx.last_kernel)


def test_skinny_unaligned_operands(ctx):
    """Odd leading dimensions and bases off 16 bytes: element loads instead
    of 16-byte loads."""
    for ta, tb in LAYOUTS:
        p = synthetic.make_problem(5, 1001, 999, "f16", "f16", transpose_a=ta, transpose_b=tb, seed=81,
                                   dist="normal", lda=(5 if ta else 999) + 3, ldb=(999 if tb else 1001) + 1,
                                   ldc=1001 + 5, beta=1.0, c_fill="uniform")
        A = torch.empty(p.A.numel() + 1, dtype=p.A.dtype, device="cuda")
        A[1:] = p.A.reshape(-1).cuda()
        B, C = p.B.cuda(), p.C.cuda()
        d = tg.make_desc(p.M, p.N, p.K, "f16", "f16", transpose_a=ta, transpose_b=tb, beta=1.0,
                         lda=p.A.shape[1], ldb=p.B.shape[1], ldc=p.C.shape[1])
        tg.tc_gemm(ctx, d, A[1:], B, C)
        R, T = oracle.gemm(p)
        parity.check(oracle.decode(C.cpu())[:, : p.N], R, T, "f16", what=f"unaligned {p.layout} {ctx.last_kernel}")


@pytest.mark.parametrize("shape", [(4, 4096, 4096), (4096, 2, 4096), (1, 300, 20000)])
def test_skinny_deterministic(ctx, shape):
    M, N, K = shape
    p = synthetic.make_problem(M, N, K, "bf16", "f32", transpose_b=True, seed=82, dist="normal")
    outs = [run(ctx, p) for _ in range(6)]
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    R, T = oracle.gemm(p)
    parity.check(outs[0].numpy(), R, T, "f32", what=f"{shape} {ctx.last_kernel}")


def test_skinny_batched(ctx):
    M, N, K, batch = 3, 700, 513, 4
    g = torch.Generator().manual_seed(83)
    A = torch.randn(batch, M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(K, N, generator=g).to(torch.bfloat16)          # one B for every entry
    C = torch.zeros(batch, M, N)
    Ad, Bd, Cd = A.cuda(), B.cuda(), C.cuda()
    bd = tg.tc_gemm_batched_desc(tg.make_desc(M, N, K, "bf16", "f32"), batch, M * K, 0, M * N)
    tg.tc_gemm_batched(ctx, bd, Ad, Bd, Cd)
    out = Cd.cpu()
    for i in range(batch):
        R, T = oracle.gemm(synthetic.Problem(M, N, K, "bf16", "f32", A=A[i], B=B, C=C[i]))
        parity.check(out[i].numpy(), R, T, "f32", what=f"batch {i}")


@pytest.mark.parametrize("shape", [(4, 1500, 3000), (1500, 4, 3000)])
def test_skinny_fused_epilogue(ctx, shape):
    """bias + GELU on the skinny path; the bias follows C's columns (p for a
    small M, q for a small N)."""
    M, N, K = shape
    p = synthetic.make_problem(M, N, K, "bf16", "bf16", transpose_b=True, alpha=0.5, beta=1.0, seed=84,
                               dist="normal", c_fill="uniform")
    bias = torch.randn(N, generator=torch.Generator().manual_seed(85)).to(torch.bfloat16)
    A, B, C = p.A.cuda(), p.B.cuda(), p.C.cuda()
    d = tg.make_desc(M, N, K, "bf16", "bf16", transpose_b=True, alpha=0.5, beta=1.0)
    tg.tc_gemm_epilogue(ctx, d, A, B, C, bias=bias.cuda(), activation="gelu_tanh")
    assert ctx.last_kernel.endswith("_bias_gelu")
    R, T, Y = oracle.gemm_epilogue(p, bias, "gelu_tanh")
    parity.check_epilogue(oracle.decode(C.cpu()), R, T, Y, np.abs(oracle.decode(bias))[None, :], "bf16",
                          "gelu_tanh", what=f"{shape}")


@pytest.mark.parametrize("shape", list(synthetic.DECODE_SHAPES))
def test_decode_shapes(ctx, shape):
    p = synthetic.f16_decode(*shape)
    check(ctx, p, f"decode {shape}")
    assert ctx.last_kernel.startswith("gemv_nt_f16_f16_x"), ctx.last_kernel


@pytest.mark.parametrize("M", list(range(1, 18)))
@pytest.mark.parametrize("ab", ["f16", "bf16"])
def test_gemv_every_row_count(ctx, M, ab):
    """1 to 16 rows of X (one or two 8-row MMA column tiles, rows beyond M
    zero), and 17, which goes to the tensor cores; the transposed product
    (few columns) takes the same kernel with the roles swapped."""
    p = synthetic.make_problem(M, 300, 2000, ab, "f32", transpose_b=True, alpha=0.5, beta=1.0, seed=M + 90,
                               dist="normal", c_fill="uniform")
    check(ctx, p, f"M={M}")
    assert ctx.last_kernel.startswith("gemv_" if M <= 16 else "tcgen05_"), ctx.last_kernel
    q = synthetic.make_problem(300, M, 2000, ab, ab, transpose_b=True, seed=M + 91, dist="normal")
    check(ctx, q, f"N={M}")
    if M <= 16:
        assert "_swap" in ctx.last_kernel, ctx.last_kernel


@pytest.mark.parametrize("spec", ["", "gemv_ks=1", "gemv_ks=2", "gemv_ks=4", "gemv_ks=8", "gemv_blocks=0",
                                  "gemv_blocks=1", "gemv_grid=230", "gemv_grid=1000", "gemv_blocks=1 gemv_grid=1000"])
def test_gemv_forms_integer_bitwise(ctx, force, spec):
    """The row-range form (each CTA an equal share of W's rows, the warps'
    sums added in warp order) and the cluster form with K cut over 1 to 8
    CTAs (sums added in rank order): integer data give the exact result
    whatever the cut.  K = 9001 rows are not 16-byte multiples and 5 rows
    are fewer than the SMs, so those take the cluster form whatever is asked.
    5003 rows are 313 16-row blocks, more than two per SM, so by default
    they go out in whole blocks (157 CTAs of 2, the last ragged)."""
    force(spec)
    for (M, N, K) in [(4, 1000, 4096), (16, 33, 9001), (1, 5, 17), (9, 300, 2048), (4, 5003, 1024)]:
        p = synthetic.make_problem(M, N, K, "f16", "f32", transpose_b=True, beta=1.0, seed=K + len(spec),
                                   dist="int", scale=4.0, c_fill="int")
        out = run(ctx, p)
        rr = "gemv_ks" not in spec and K % 8 == 0 and N >= 152
        assert ("_rr" in ctx.last_kernel) == rr, ctx.last_kernel
        if spec == "" and N == 5003:
            assert ctx.last_kernel.endswith("_rr157b"), ctx.last_kernel
        R, _ = oracle.gemm(p)
        assert np.array_equal(out.numpy().astype(np.float64), R), (M, N, K, ctx.last_kernel)


@pytest.mark.parametrize("ab", ["f16", "bf16"])
def test_gemv_both_forms_agree(ctx, force, ab):
    """The row-range and cluster forms on the same problem: both within the
    bound (their K orders differ), each bitwise equal to itself run to run."""
    p = synthetic.make_problem(7, 3000, 5120, ab, "f32", transpose_b=True, alpha=0.5, beta=-1.0, seed=97,
                               dist="normal", c_fill="uniform")
    R, T = oracle.gemm(p)
    for spec in ["", "gemv_rr=0"]:
        force(spec)
        outs = [run(ctx, p) for _ in range(3)]
        for o in outs[1:]:
            assert torch.equal(o, outs[0]), ctx.last_kernel
        parity.check(outs[0].numpy(), R, T, "f32", what=f"{spec} {ctx.last_kernel}")
