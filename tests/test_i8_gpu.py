"""The int8 GEMM with per-column dequantisation (tessl architecture.md,
"Integer GEMM") against the CPU oracle on GB300.  The accumulation is exact,
so with scale 1, alpha 1 and beta 0 the fp32 output equals the oracle's
integer rounded once to fp32, bit for bit; with scales, alpha and beta the
device rounds twice more (scale, then alpha/beta with C), bounded by a few
ulp of the terms."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
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


def run(ctx, p, scale, **kw):
    A, B, C = p.A.cuda(), p.B.cuda(), p.C.cuda()
    d = tg.make_desc(p.M, p.N, p.K, "i8", "f32", transpose_a=p.transpose_a, transpose_b=p.transpose_b,
                     alpha=p.alpha, beta=p.beta, lda=A.shape[1], ldb=B.shape[1], ldc=C.shape[1])
    tg.tc_gemm_i8_dequant(ctx, d, A, B, C, scale.cuda())
    return C.cpu()


@pytest.mark.parametrize("ta,tb", LAYOUTS)
@pytest.mark.parametrize("K", [1, 100, 1024, 1025, 5000])
def test_i8_exact(ctx, ta, tb, K):
    """Full-range int8; K up to 1024 is one slice, beyond it several slices
    summed as integers."""
    p = synthetic.i8_problem(300, 260, K, transpose_a=ta, transpose_b=tb, seed=K + 3)
    out = run(ctx, p, torch.ones(260))
    _, _, ACC = oracle.gemm_i8_dequant(p, torch.ones(260))
    assert np.array_equal(out.numpy(), ACC.astype(np.float32)), ctx.last_kernel
    assert ctx.last_kernel.startswith("i8_dequant_tcgen05_") and ctx.last_kernel.endswith(f"_i8acc_s{(K + 1023) // 1024}")


@pytest.fixture
def force(monkeypatch):
    def set_(spec):
        if spec:
            monkeypatch.setenv("TC_FORCE_VARIANT", spec)
        else:
            monkeypatch.delenv("TC_FORCE_VARIANT", raising=False)
    return set_


@pytest.mark.parametrize("ta,tb", LAYOUTS)
@pytest.mark.parametrize("shape", [(300, 260, 1000), (300, 260, 1024), (700, 390, 1025), (1100, 260, 3000),
                                   (2048, 2048, 2100)])
def test_i8_on_chip_equals_memory_slices(ctx, force, ta, tb, shape):
    """K slices summed as int32 in TMEM give the same bits as slices written
    to memory and added by the reduction kernel: the same exact integer,
    rounded once, then the same scale and alpha/beta.  Shapes span one slice,
    a slice boundary, ragged last slices, both CTA shapes (the small ones run
    128x128 tiles, the 2048^2 one CTA pairs) and ragged M, N."""
    M, N, K = shape
    p = synthetic.i8_problem(M, N, K, transpose_a=ta, transpose_b=tb, seed=M + K)
    p.alpha, p.beta = 0.75, -0.5
    p.C = (torch.randn(M, N, generator=torch.Generator().manual_seed(K))).float()
    scale = torch.rand(N, generator=torch.Generator().manual_seed(N)) + 0.5
    force("i8acc=0")
    ref = run(ctx, p, scale)
    k_mem = ctx.last_kernel
    force("")
    got = run(ctx, p, scale)
    assert "_i8acc_" in ctx.last_kernel and "_i8acc_" not in k_mem, (ctx.last_kernel, k_mem)
    assert torch.equal(got.view(torch.int32), ref.view(torch.int32)), ctx.last_kernel


def test_i8_on_chip_largest_sums(ctx):
    """All -128 at K = 65536, the largest K summed on chip: every int32 sum is
    2^30, exact."""
    K = 65536
    A = torch.full((300, K), -128, dtype=torch.int8)
    B = torch.full((K, 136), -128, dtype=torch.int8)
    p = synthetic.Problem(300, 136, K, "i8", "f32", False, False, 1.0, 0.0, A, B, torch.zeros(300, 136))
    out = run(ctx, p, torch.ones(136))
    assert "_i8acc_" in ctx.last_kernel, ctx.last_kernel
    assert (out == 2.0 ** 30).all()


def test_i8_full_range_at_the_k_limit(ctx):
    """All -128 at K = 131072: the sum is 2^31, one past int32."""
    K = 131072
    A = torch.full((8, K), -128, dtype=torch.int8)
    B = torch.full((K, 16), -128, dtype=torch.int8)
    p = synthetic.Problem(8, 16, K, "i8", "f32", False, False, 1.0, 0.0, A, B, torch.zeros(8, 16))
    out = run(ctx, p, torch.ones(16))
    assert (out == 2.0 ** 31).all()


@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_i8_dequant_alpha_beta(ctx, ta, tb):
    p = synthetic.i8_problem(257, 385, 3000, transpose_a=ta, transpose_b=tb, seed=21, alpha=0.75, beta=-0.5,
                             c_fill="uniform")
    scale = torch.rand(385, generator=torch.Generator().manual_seed(22)) * 1e-3
    out = run(ctx, p, scale).numpy().astype(np.float64)
    R, _, ACC = oracle.gemm_i8_dequant(p, scale)
    Cold = p.C.double().numpy()
    term = np.abs(0.75 * ACC * scale.double().numpy()[None, :]) + np.abs(0.5 * Cold)
    lim = 4 * 2.0 ** -24 * term + 1e-30
    bad = ~(np.abs(out - R) <= lim)
    assert not bad.any(), (np.argwhere(bad)[:5], ctx.last_kernel)


def test_i8_deterministic(ctx):
    p = synthetic.i8_problem(512, 384, 8192, seed=23)
    scale = torch.rand(384, generator=torch.Generator().manual_seed(24))
    outs = [run(ctx, p, scale) for _ in range(4)]
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_i8_refusals_launch_nothing(ctx):
    before = ctx.launch_count
    A = torch.zeros(64, 64, dtype=torch.int8, device="cuda")
    C = torch.zeros(64, 64, device="cuda")
    s = torch.ones(64, device="cuda")
    with pytest.raises(tg.TcError) as err:                       # past the page's K limit
        tg.tc_gemm_i8_dequant(ctx, tg.make_desc(64, 64, 131073, "i8", "f32"), 1 << 20, 2 << 40, C, s)
    assert err.value.status == tg.TC_ERR_DIM
    with pytest.raises(tg.TcError) as err:                       # int8 operands on the plain GEMM
        tg.tc_gemm(ctx, tg.make_desc(64, 64, 64, "i8", "f32"), A, A, C)
    assert err.value.status == tg.TC_ERR_DTYPE
    with pytest.raises(tg.TcError) as err:                       # float operands on the int8 GEMM
        tg.tc_gemm_i8_dequant(ctx, tg.make_desc(64, 64, 64, "bf16", "f32"), 1 << 20, 2 << 40, 3 << 40, s)
    assert err.value.status == tg.TC_ERR_DTYPE
    with pytest.raises(tg.TcError) as err:                       # no scale
        tg.tc_gemm_i8_dequant(ctx, tg.make_desc(64, 64, 64, "i8", "f32"), A, A, C, None)
    assert err.value.status == tg.TC_ERR_NULL
    assert ctx.launch_count == before


def test_i8_named_workload(ctx):
    """The int8 workload at 4096^3: sampled elements and ragged edges, exact
    integers times the column scale (one fp32 rounding each)."""
    p, scale = synthetic.i8_dequant_4096()
    out = run(ctx, p, scale)
    rng = np.random.default_rng(2)
    rows = rng.integers(0, 4096, 400)
    R, _, ACC = oracle.gemm_i8_dequant(p, scale, 0, None)
    got = out.numpy()[rows].astype(np.float64)
    want = (ACC[rows].astype(np.float32).astype(np.float64) * scale.double().numpy()[None, :])
    lim = 2 * 2.0 ** -24 * np.abs(want) + 1e-30
    assert (np.abs(got - want) <= lim).all(), ctx.last_kernel
