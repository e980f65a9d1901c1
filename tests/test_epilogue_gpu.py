"""Parity of the fused bias + GELU epilogue with the CPU oracle (GB300).

tessl architecture.md, "Fused Epilogue": C = activation(alpha * A@B +
beta * C_prev + bias), bias per column, activation none or GeluTanh,
refused on the exact-fp32 path.  The oracle (oracle.gemm_epilogue) applies
the bias and the activation in fp64 on top of its fp64 GEMM; the bound is
tests/parity.bound_epilogue (the GEMM's 1e-4 * sum|ab|, carried through the
activation's slope, plus the fp32 evaluation of GELU and one output ulp).
"""
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
TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


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


def make_bias(N, c_dtype, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(N, generator=g) * scale).to(TORCH_DT[c_dtype])


def run_epilogue(ctx, p, bias, activation, ldc=0):
    A, B, C = p.A.cuda(), p.B.cuda(), p.C.cuda()
    d = tg.make_desc(p.M, p.N, p.K, p.ab_dtype, p.c_dtype, transpose_a=p.transpose_a,
                     transpose_b=p.transpose_b, alpha=p.alpha, beta=p.beta,
                     lda=A.shape[1], ldb=B.shape[1], ldc=ldc or C.shape[1])
    tg.tc_gemm_epilogue(ctx, d, A, B, C, bias=None if bias is None else bias.cuda(), activation=activation)
    return C.cpu()


def check(ctx, p, bias, activation, what=""):
    out = run_epilogue(ctx, p, bias, activation)
    R, T, Y = oracle.gemm_epilogue(p, bias, activation)
    babs = 0.0 if bias is None else np.abs(oracle.decode(bias))[None, : p.N]
    got = oracle.decode(out)[:, : p.N]
    return parity.check_epilogue(got, R, T, Y, babs, p.c_dtype, activation, what=f"{what} {ctx.last_kernel}")


@pytest.mark.parametrize("activation", ["none", "gelu_tanh"])
@pytest.mark.parametrize("ab,c", DT_PAIRS)
@pytest.mark.parametrize("ta,tb", LAYOUTS)
@pytest.mark.parametrize("shape", [(5, 7, 3), (300, 200, 333), (257, 385, 130)])
def test_epilogue_parity(ctx, activation, ab, c, ta, tb, shape):
    M, N, K = shape
    p = synthetic.make_problem(M, N, K, ab, c, transpose_a=ta, transpose_b=tb, alpha=0.75, beta=0.5,
                               seed=M + 3 * K, dist="normal", c_fill="uniform")
    bias = make_bias(N, c, seed=N)
    check(ctx, p, bias, activation, f"{ab}->{c} {p.layout} {shape} {activation}")
    want = "_bias" + ("_gelu" if activation == "gelu_tanh" else "")
    assert ctx.last_kernel.endswith(want), ctx.last_kernel


@pytest.mark.parametrize("spec", ["", "cg=2", "cg=1 bn=64", "cg=1 bn=192", "bn=128 split=3", "bn=128 split=3 csplit=0",
                                  "bn=64 split=16", "bn=256 split=5",
                                  "sms=5 tail=2", "cg=2 sms=6 tail=2", "store=direct", "pack=1",
                                  "pack=1 split=4", "cg=2 bn=128", "cg=2 bn=192", "cg=2 bn=192 sms=4 tail=2"])
@pytest.mark.parametrize("c", ["bf16", "f32"])
def test_epilogue_every_variant(ctx, force, spec, c):
    """The epilogue in the tensor-core kernel's own store paths (TMA, plain,
    staged), in the on-chip reduction of a cluster split and in the split-K
    reduction kernel."""
    force(spec)
    p = synthetic.make_problem(333, 470, 1100, "bf16", c, transpose_b=True, alpha=-0.5, beta=1.0, seed=41,
                               dist="normal", c_fill="uniform")
    check(ctx, p, make_bias(470, c, seed=42, scale=3.0), "gelu_tanh", spec)


def test_epilogue_unaligned_c_and_bias(ctx):
    """Odd ldc (the staged store path) and a bias at an odd element offset."""
    p = synthetic.make_problem(150, 97, 210, "f16", "f16", seed=43, dist="normal", beta=1.0, c_fill="uniform",
                               ldc=101)
    flat = make_bias(97 + 3, "f16", seed=44)
    bias = flat[3:]
    out = run_epilogue(ctx, p, bias, "gelu_tanh", ldc=101)
    R, T, Y = oracle.gemm_epilogue(p, bias, "gelu_tanh")
    parity.check_epilogue(oracle.decode(out)[:, :97], R, T, Y, np.abs(oracle.decode(bias))[None, :], "f16",
                          "gelu_tanh", what=f"unaligned {ctx.last_kernel}")


def test_bias_only_integer_exact(ctx, force):
    """No activation, integer data and an integer bias: every value is an
    integer below 2^24, so the result is exact in fp32 on every path."""
    for spec in ["", "bn=128 split=4", "bn=128 split=4 csplit=0", "sms=5 tail=3", "store=direct"]:
        force(spec)
        p = synthetic.make_problem(200, 136, 1024, "bf16", "f32", alpha=1.0, beta=1.0, seed=45, dist="int",
                                   scale=4.0, c_fill="int")
        bias = torch.arange(136, dtype=torch.float32) - 60.0
        out = run_epilogue(ctx, p, bias, "none")
        R, _, _ = oracle.gemm_epilogue(p, bias, "none")
        assert np.array_equal(out.numpy().astype(np.float64), R), spec


def test_gelu_without_bias_and_no_op_epilogue(ctx):
    p = synthetic.make_problem(130, 260, 300, "bf16", "bf16", seed=46, dist="normal")
    check(ctx, p, None, "gelu_tanh", "gelu, no bias")
    assert ctx.last_kernel.endswith("_gelu") and "_bias" not in ctx.last_kernel
    # no bias and no activation: the plain GEMM, bit for bit
    A, B = p.A.cuda(), p.B.cuda()
    d = tg.make_desc(p.M, p.N, p.K, "bf16", "bf16")
    C1 = torch.zeros(p.M, p.N, dtype=torch.bfloat16, device="cuda")
    C2 = torch.zeros_like(C1)
    tg.tc_gemm_epilogue(ctx, d, A, B, C1, bias=None, activation="none")
    tg.tc_gemm(ctx, d, A, B, C2)
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))


def test_epilogue_deterministic(ctx, force):
    for spec in ["", "bn=128 split=6", "bn=128 split=6 csplit=0"]:
        force(spec)
        p = synthetic.make_problem(384, 512, 2048, "bf16", "f32", seed=47, dist="normal")
        bias = make_bias(512, "f32", seed=48)
        outs = [run_epilogue(ctx, p, bias, "gelu_tanh") for _ in range(4)]
        for o in outs[1:]:
            assert torch.equal(o, outs[0]), spec


def test_epilogue_refusals_launch_nothing(ctx):
    before = ctx.launch_count
    A = torch.zeros(64, 64, device="cuda")
    B = torch.zeros(64, 64, device="cuda")
    C = torch.zeros(64, 64, device="cuda")
    d = tg.make_desc(64, 64, 64, "f32", "f32")
    with pytest.raises(tg.TcError) as err:
        tg.tc_gemm_epilogue(ctx, d, A, B, C, bias=torch.zeros(64, device="cuda"), activation="gelu_tanh")
    assert err.value.status == tg.TC_ERR_EPILOGUE          # the exact-fp32 path has nothing to fuse into
    Ah = A.to(torch.bfloat16)
    Bh = B.to(torch.bfloat16)
    dh = tg.make_desc(64, 64, 64, "bf16", "f32")
    with pytest.raises(tg.TcError) as err:
        tg.tc_gemm_epilogue(ctx, dh, Ah, Bh, C, bias=None, activation=9)
    assert err.value.status == tg.TC_ERR_EPILOGUE
    with pytest.raises(tg.TcError) as err:
        tg.tc_gemm_epilogue(ctx, dh, Ah, Bh, C, bias=C.view(-1)[10:74], activation="gelu_tanh")
    assert err.value.status == tg.TC_ERR_OVERLAP
    assert ctx.launch_count == before


@pytest.mark.parametrize("shape", list(synthetic.EPILOGUE_SHAPES))
def test_pages_epilogue_shapes(ctx, shape):
    """The fused-epilogue workloads (bf16, bias + GELU) on sampled elements
    plus every ragged edge."""
    p, bias = synthetic.bf16_epilogue(*shape)
    out = run_epilogue(ctx, p, bias, "gelu_tanh")
    rows, cols = parity.sample_points(p.M, p.N, 3000, np.random.default_rng(1))
    R, T, Y = oracle.gemm_epilogue_points(p, bias, "gelu_tanh", rows, cols)
    got = oracle.decode(out)[rows, cols]
    parity.check_epilogue(got, R, T, Y, np.abs(oracle.decode(bias))[cols], "bf16", "gelu_tanh",
                          what=f"{shape} {ctx.last_kernel}")
