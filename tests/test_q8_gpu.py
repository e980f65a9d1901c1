"""The int8-weight product (Foundry metal.md, "Custom Compute Kernels":
fm_sgemm_q8 / fm_matvec_q8; tensorcore gemm.md "Kernel variants": the M <= 4
GEMV over Q8 weights) against the CPU oracle on GB300:

    C[m, n] = alpha * scale[n] * sum_k X[m, k] * W[n, k] + beta * C_old[m, n]

X f16/bf16 stored [M,K], W int8 stored [N,K], one scale per weight row.
The bound is the GEMM's (tests/parity.py) with T the absolute-product sum of
the dequantised weights, |scale[n]| * sum_k |x w|.  Integer activations
with unit scales are compared bitwise.  Up to 16 activation rows the int8
weights are streamed by the skinny-product kernel; beyond, they are widened
once and run through the tensor-core GEMM with the scale in its epilogue."""
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


def run(ctx, p, scale, X=None, W=None, stream=None):
    X = p.A.cuda() if X is None else X
    W = p.B.cuda() if W is None else W
    C = p.C.cuda()
    d = tg.make_desc(p.M, p.N, p.K, p.ab_dtype, p.c_dtype, b_dtype="i8", transpose_b=True, alpha=p.alpha,
                     beta=p.beta, lda=p.A.shape[1], ldb=p.B.shape[1], ldc=C.shape[1])
    if stream is None:
        tg.tc_gemm_q8_weight(ctx, d, X, W, C, scale.cuda())
    else:
        tg.tc_gemm_q8_weight_async(ctx, d, X, W, C, scale.cuda(), stream)
        stream.sync()
    return C.cpu()


def check(ctx, p, scale, what="", **kw):
    out = run(ctx, p, scale, **kw)
    R, T, _ = oracle.gemm_q8_weight(p, scale)
    return parity.check(oracle.decode(out)[:, : p.N], R, T, p.c_dtype, what=f"{what} {ctx.last_kernel}")


SHAPES = [(1, 1, 1), (1, 1000, 77), (2, 17, 4096), (4, 300, 3000), (7, 129, 1000), (8, 1000, 64), (9, 33, 100),
          (16, 513, 2049), (17, 300, 700), (40, 260, 1500)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("x,c", [("f16", "f16"), ("f16", "f32"), ("bf16", "bf16"), ("bf16", "f32")])
def test_q8_parity(ctx, shape, x, c):
    M, N, K = shape
    p, scale = synthetic.q8_weight_problem(M, N, K, x, c, alpha=0.75, beta=-0.5, seed=M + 3 * N + K,
                                           c_fill="uniform")
    check(ctx, p, scale, f"{x}->{c} {shape}")
    want = "gemv_q8w" if M <= 16 else "q8w_widen_tcgen05"
    assert ctx.last_kernel.startswith(want), ctx.last_kernel


@pytest.mark.parametrize("spec", ["", "gemv_ks=1", "gemv_ks=2", "gemv_ks=4", "gemv_ks=8", "gemv_blocks=0",
                                  "gemv_blocks=1"])
@pytest.mark.parametrize("x", ["f16", "bf16"])
def test_q8_integer_bitwise(ctx, force, spec, x):
    """Integer activations in [-4, 4] and unit scales: every partial sum is an
    integer below 2^24, so the fp32 result is exact whatever the K split or
    the share of W's rows (or 16-row blocks, 313 of them for 5003 rows) that
    each CTA of the row-range form takes."""
    force(spec)
    for (M, N, K) in [(4, 1100, 4096), (13, 200, 9000), (1, 64, 33), (4, 5003, 1024)]:
        p, _ = synthetic.q8_weight_problem(M, N, K, x, "f32", seed=K + M, x_dist="int")
        out = run(ctx, p, torch.ones(N))
        _, _, ACC = oracle.gemm_q8_weight(p, torch.ones(N))
        assert np.array_equal(out.numpy().astype(np.float64), ACC), (M, N, K, ctx.last_kernel)


def test_q8_unaligned(ctx):
    """Rows that are not 16-byte multiples and bases off 16 bytes: element
    loads instead of 16-byte loads, for X and for W."""
    for M, N, K in [(3, 301, 999), (16, 77, 1001)]:
        p, scale = synthetic.q8_weight_problem(M, N, K, "f16", "f16", beta=1.0, seed=K, c_fill="uniform",
                                               ldx=K + 3, ldw=K + 5)
        X = torch.empty(p.A.numel() + 1, dtype=p.A.dtype, device="cuda")
        X[1:] = p.A.reshape(-1).cuda()
        W = torch.empty(p.B.numel() + 7, dtype=torch.int8, device="cuda")
        W[7:] = p.B.reshape(-1).cuda()
        check(ctx, p, scale, f"unaligned {M}x{N}x{K}", X=X[1:], W=W[7:])


@pytest.mark.parametrize("shape", list(synthetic.DECODE_SHAPES))
def test_q8_decode_shapes(ctx, shape):
    """The decode shapes at full size, every output element."""
    p, scale = synthetic.q8_decode(*shape)
    check(ctx, p, scale, f"decode {shape}")
    assert ctx.last_kernel.startswith("gemv_q8w_nt_f16_f16"), ctx.last_kernel


def test_q8_deterministic_and_async(ctx):
    p, scale = synthetic.q8_weight_problem(4, 4096, 11008, "bf16", "f32", seed=71)
    outs = [run(ctx, p, scale) for _ in range(4)]
    stream = tg.Stream(ctx)
    outs.append(run(ctx, p, scale, stream=stream))
    stream.close()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_q8_wide_path_matches_bound(ctx, force):
    """More than 16 activation rows: the widened weights through the tensor
    cores, in their split-K and plain forms."""
    for spec in ["", "bn=128 split=4", "bn=128 split=4 csplit=0"]:
        force(spec)
        p, scale = synthetic.q8_weight_problem(200, 384, 3000, "f16", "f32", alpha=2.0, beta=1.0, seed=72,
                                               c_fill="uniform")
        check(ctx, p, scale, f"wide {spec}")
        assert ctx.last_kernel.startswith("q8w_widen_"), ctx.last_kernel


def test_q8_refusals_launch_nothing(ctx):
    X = torch.zeros(4, 64, dtype=torch.float16, device="cuda")
    W = torch.zeros(32, 64, dtype=torch.int8, device="cuda")
    C = torch.zeros(4, 32, dtype=torch.float16, device="cuda")
    s = torch.ones(32, device="cuda")
    before = ctx.launch_count
    bad = [
        (tg.make_desc(4, 32, 64, "f16", "f16", b_dtype="i8", transpose_b=False), tg.TC_ERR_LAYOUT),
        (tg.make_desc(4, 32, 64, "f16", "f16", b_dtype="f16", transpose_b=True), tg.TC_ERR_DTYPE),
        (tg.make_desc(4, 32, 64, "f32", "f32", b_dtype="i8", transpose_b=True), tg.TC_ERR_DTYPE),
        (tg.make_desc(4, 32, 64, "f16", "bf16", b_dtype="i8", transpose_b=True), tg.TC_ERR_DTYPE),
        (tg.make_desc(0, 32, 64, "f16", "f16", b_dtype="i8", transpose_b=True), tg.TC_ERR_DIM),
    ]
    for d, want in bad:
        with pytest.raises(tg.TcError) as err:
            tg.tc_gemm_q8_weight(ctx, d, X, W, C, s)
        assert err.value.status == want
    d = tg.make_desc(4, 32, 64, "f16", "f16", b_dtype="i8", transpose_b=True)
    lib = tg.library()
    import ctypes
    assert lib.tc_gemm_q8_weight(ctx.ptr, ctypes.byref(d), None, X.data_ptr(), W.data_ptr(),
                                 C.data_ptr()) == tg.TC_ERR_NULL
    assert ctx.launch_count == before
