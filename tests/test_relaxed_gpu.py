"""Relaxed fp32 (tc_gemm_f32_relaxed): fp32 operands on the bf16 tensor
cores through a two-part bf16 split, against the CPU oracle's fp64 product
of the same fp32 inputs.  The bound is the non-exact paths' 1e-4 * sum|ab|
(tests/parity.py); the split's own error is below 2^-15 |ab| per product,
so the observed error is also checked against 5e-5 * sum|ab| -- a single
bf16 rounding of the operands (about 4e-3) would fail it."""
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


@pytest.fixture(scope="module")
def ctx():
    c = tg.Context(0)
    yield c
    c.close()


def run_relaxed(ctx, p, bias=None, activation=None):
    A, B, C = p.A.cuda(), p.B.cuda(), p.C.cuda()
    d = tg.make_desc(p.M, p.N, p.K, "f32", "f32", transpose_a=p.transpose_a, transpose_b=p.transpose_b,
                     alpha=p.alpha, beta=p.beta, lda=A.shape[1], ldb=B.shape[1], ldc=C.shape[1])
    tg.tc_gemm_f32_relaxed(ctx, d, A, B, C, bias=None if bias is None else bias.cuda(), activation=activation)
    return C.cpu()


@pytest.mark.parametrize("ta,tb", LAYOUTS)
@pytest.mark.parametrize("shape", [(1, 1, 1), (5, 7, 3), (256, 256, 256), (300, 200, 333), (640, 520, 1000)])
def test_relaxed_parity(ctx, ta, tb, shape):
    M, N, K = shape
    p = synthetic.make_problem(M, N, K, "f32", "f32", transpose_a=ta, transpose_b=tb, alpha=-1.25, beta=0.5,
                               seed=11 + K, dist="uniform", c_fill="uniform")
    out = run_relaxed(ctx, p)
    R, T = oracle.gemm(p)
    stats = parity.check(out.numpy()[:, :N], R, T, "f32", what=f"relaxed {p.layout} {shape} {ctx.last_kernel}")
    assert stats["max_err_over_T"] < 5e-5, stats
    assert ctx.last_kernel.startswith("relaxed_f32_3xbf16_tcgen05_"), ctx.last_kernel


def test_relaxed_padded_and_nan_c(ctx):
    p = synthetic.make_problem(130, 70, 90, "f32", "f32", transpose_b=True, seed=12, dist="normal", lda=97, ldb=93,
                               ldc=75, c_fill="nan")
    out = run_relaxed(ctx, p)                       # beta = 0: the NaN-filled C is not read
    R, T = oracle.gemm(p)
    parity.check(out.numpy()[:, :70], R, T, "f32", what=f"relaxed padded {ctx.last_kernel}")


def test_relaxed_fused_epilogue(ctx):
    p = synthetic.make_problem(300, 260, 520, "f32", "f32", alpha=0.5, beta=1.0, seed=13, dist="normal",
                               c_fill="uniform")
    bias = torch.randn(260, generator=torch.Generator().manual_seed(14))
    out = run_relaxed(ctx, p, bias=bias, activation="gelu_tanh")
    R, T, Y = oracle.gemm_epilogue(p, bias, "gelu_tanh")
    parity.check_epilogue(out.numpy(), R, T, Y, np.abs(oracle.decode(bias))[None, :], "f32", "gelu_tanh",
                          what=f"relaxed epilogue {ctx.last_kernel}")
    assert ctx.last_kernel.endswith("_bias_gelu")


def test_relaxed_deterministic_and_distinct_from_exact(ctx):
    p = synthetic.make_problem(512, 384, 2048, "f32", "f32", seed=15, dist="normal")
    outs = [run_relaxed(ctx, p) for _ in range(4)]
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    A, B, C = p.A.cuda(), p.B.cuda(), p.C.cuda()
    tg.tc_gemm(ctx, tg.make_desc(512, 384, 2048, "f32", "f32"), A, B, C)
    assert ctx.last_kernel.startswith("ffma_")      # the exact path is unchanged
    R, T = oracle.gemm(p)
    parity.check(C.cpu().numpy(), R, T, "f32", exact_f32=True, what="exact")
    parity.check(outs[0].numpy(), R, T, "f32", what="relaxed")


def test_relaxed_refusals_launch_nothing(ctx):
    before = ctx.launch_count
    A = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(64, 64, device="cuda")
    with pytest.raises(tg.TcError) as err:
        tg.tc_gemm_f32_relaxed(ctx, tg.make_desc(64, 64, 64, "bf16", "f32"), A, A, C)
    assert err.value.status == tg.TC_ERR_DTYPE
    Af = torch.zeros(64, 64, device="cuda")
    with pytest.raises(tg.TcError) as err:
        tg.tc_gemm_f32_relaxed(ctx, tg.make_desc(64, 64, 64, "f32", "f32"), Af, Af, C, activation=5)
    assert err.value.status == tg.TC_ERR_EPILOGUE
    assert ctx.launch_count == before


def test_relaxed_named_workload(ctx):
    """The fp32 NN 256^3 workload, relaxed, under the standard bound."""
    p = synthetic.fp32_nn_256()
    out = run_relaxed(ctx, p)
    R, T = oracle.gemm(p)
    parity.check(out.numpy(), R, T, "f32", what=f"fp32 256^3 relaxed {ctx.last_kernel}")
