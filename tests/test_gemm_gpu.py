"""Parity of the CUDA path with the CPU oracle, through the C ABI (GB300).

Every case draws seeded inputs (synthetic.py), runs the library and compares
each output element (or, at full size, sampled elements plus the ragged
edges) with the oracle's fp64 value under the bound of tests/parity.py:
|C - R| <= 1e-4 * sum_k|a b| (+ one output ulp for f16/bf16 output), and
1e-5 * sum_k|a b| on the fp32-exact path.  Integer-valued inputs are
compared bitwise.
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


def run_problem(ctx, p, *, lda=0, ldb=0, ldc=0, stream=None):
    A, B, C = p.A.cuda(), p.B.cuda(), p.C.cuda()
    d = tg.make_desc(p.M, p.N, p.K, p.ab_dtype, p.c_dtype, transpose_a=p.transpose_a,
                     transpose_b=p.transpose_b, alpha=p.alpha, beta=p.beta,
                     lda=lda or A.shape[1], ldb=ldb or B.shape[1], ldc=ldc or C.shape[1])
    if stream is None:
        tg.tc_gemm(ctx, d, A, B, C)
    else:
        tg.tc_gemm_async(ctx, d, A, B, C, stream)
        stream.sync()
    return C.cpu()


def check_full(ctx, p, what="", **kw):
    out = run_problem(ctx, p, **kw)
    R, T = oracle.gemm(p)
    got = oracle.decode(out)[:, : p.N]
    return parity.check(got, R, T, p.c_dtype, exact_f32=(p.ab_dtype == "f32"),
                        what=f"{what} {ctx.last_kernel}")


def check_sampled(ctx, p, n=2000, seed=0, what=""):
    out = run_problem(ctx, p)
    rows, cols = parity.sample_points(p.M, p.N, n, np.random.default_rng(seed))
    R, T = oracle.gemm_points(p, rows, cols)
    got = oracle.decode(out)[rows, cols]
    return parity.check(got, R, T, p.c_dtype, exact_f32=(p.ab_dtype == "f32"),
                        what=f"{what} {ctx.last_kernel}")


# ------------------------------------------------------------ small shapes

SHAPES = [(1, 1, 1), (5, 7, 3), (128, 256, 64), (300, 200, 333), (257, 385, 130), (640, 520, 1000)]


@pytest.mark.parametrize("ab,c", DT_PAIRS)
@pytest.mark.parametrize("ta,tb", LAYOUTS)
@pytest.mark.parametrize("shape", SHAPES)
def test_tensor_core_parity(ctx, force, ab, c, ta, tb, shape):
    """Every layout on the tensor-core kernel (NT products with at most 16
    rows on one side would otherwise take the skinny-product kernel, which
    tests/test_skinny_gpu.py covers)."""
    force("gemv=0")
    M, N, K = shape
    p = synthetic.make_problem(M, N, K, ab, c, transpose_a=ta, transpose_b=tb, seed=M * 7 + K,
                               dist="normal")
    check_full(ctx, p, f"{ab}->{c} {p.layout} {shape}")
    assert ctx.last_kernel.startswith("tcgen05_" + p.layout.lower())


@pytest.mark.parametrize("ta,tb", LAYOUTS)
@pytest.mark.parametrize("shape", [(1, 1, 1), (256, 256, 256), (300, 200, 333), (130, 70, 90)])
def test_ffma_parity(ctx, ta, tb, shape):
    M, N, K = shape
    p = synthetic.make_problem(M, N, K, "f32", "f32", transpose_a=ta, transpose_b=tb,
                               alpha=-1.25, beta=0.5, seed=3 + K, dist="uniform", c_fill="uniform")
    check_full(ctx, p, f"f32 {p.layout} {shape}")
    assert ctx.last_kernel.startswith("ffma_f32_" + p.layout.lower())


@pytest.mark.parametrize("shape", [(1, 4, 4), (16, 32, 64), (17, 35, 129), (255, 257, 300), (100, 60, 1000),
                                   (256, 256, 256)])
@pytest.mark.parametrize("beta", [0.0, -0.75])
def test_ffma_small_nn_pipeline(ctx, force, shape, beta):
    """The small-problem NN kernel (16-byte aligned rows): K in chunks of 64
    through a two-buffer cp.async pipeline, zeros past M, N and K; the
    exact-fp32 bound, and bitwise equality with integer data."""
    force("ffma=panel")
    M, N, K = shape
    r4 = lambda x: (x + 3) // 4 * 4      # noqa: E731
    p = synthetic.make_problem(M, N, K, "f32", "f32", alpha=1.5, beta=beta, seed=M + N + K, dist="uniform",
                               c_fill="uniform", lda=r4(K), ldb=r4(N), ldc=N + 1)
    check_full(ctx, p, f"small nn {shape}", lda=r4(K), ldb=r4(N), ldc=N + 1)
    q = synthetic.make_problem(M, N, K, "f32", "f32", alpha=1.0, beta=beta, seed=M + 2 * N + K, dist="int", scale=4,
                               c_fill="int", lda=r4(K), ldb=r4(N))
    out = run_problem(ctx, q, lda=r4(K), ldb=r4(N))
    R, _ = oracle.gemm(q)
    assert np.array_equal(oracle.decode(out)[:, :N], R), ctx.last_kernel


@pytest.mark.parametrize("spec", ["ffma=small", "ffma=large", "ffma=panel"])
@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_ffma_tiles(ctx, force, spec, ta, tb):
    force(spec)
    # K = 1100 spans several 512-wide panels; ragged M and N
    p = synthetic.make_problem(333, 290, 1100, "f32", "f32", transpose_a=ta, transpose_b=tb, seed=5,
                               alpha=0.75, beta=-0.5, c_fill="uniform")
    check_full(ctx, p, spec)


@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (0.5, 1.0), (-2.0, -0.75), (0.0, 1.0)])
@pytest.mark.parametrize("c", ["bf16", "f32"])
def test_alpha_beta(ctx, alpha, beta, c):
    p = synthetic.make_problem(200, 300, 250, "bf16", c, transpose_a=True, alpha=alpha, beta=beta,
                               seed=17, dist="normal", c_fill="uniform")
    check_full(ctx, p, f"alpha={alpha} beta={beta}")


@pytest.mark.parametrize("spec", ["bn=64", "bn=128", "cg=1 bn=192", "bn=256", "bn=128 split=3",
                                  "bn=128 split=3 csplit=0", "bn=64 split=16 csplit=0",
                                  "bn=256 split=7", "bn=64 split=16", "pack=1", "pack=1 split=5",
                                  "grid=3", "group_m=1", "group_m=3 bn=64", "sms=5 tail=2",
                                  "sms=5 tail=3 bn=64", "sms=7 bn=256 tail=2 pack=1", "cg=2",
                                  "cg=2 bn=128", "cg=2 sms=6 tail=2", "cg=2 grid=1 pack=1",
                                  "store=direct", "store=direct cg=2 sms=6 tail=2", "store=direct split=3",
                                  "cg=2 bn=192", "cg=2 bn=192 sms=6 tail=2", "cg=2 bn=192 chunk=0",
                                  "cg=2 bn=192 store=direct", "cg=2 bn=192 pack=1"])
@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_forced_variants(ctx, force, spec, ta, tb):
    force(spec)
    p = synthetic.make_problem(333, 470, 1100, "f16", "f32", transpose_a=ta, transpose_b=tb,
                               alpha=0.75, beta=-1.0, seed=23, dist="normal", c_fill="uniform")
    check_full(ctx, p, spec)


# ----------------------------------------------------- cluster split-K

CSPLIT_SPECS = ["bn=128 split=2", "bn=128 split=3", "bn=64 split=5", "bn=128 split=8", "bn=64 split=16",
                "bn=128 split=16"]


@pytest.mark.parametrize("spec", CSPLIT_SPECS)
@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_cluster_split_equals_memory_split_bitwise(ctx, force, spec, ta, tb):
    """The K slices of a tile reduced on chip by their cluster are the same
    slices, added in the same order, as the partial tiles the reduction
    kernel adds from memory: the two results are equal bit for bit, and
    within the parity bound.  M and N end inside a tile; beta != 0."""
    p = synthetic.make_problem(333, 200, 3000, "bf16", "f32", transpose_a=ta, transpose_b=tb, alpha=0.75,
                               beta=-0.5, seed=131, dist="normal", c_fill="uniform")
    force(spec + " csplit=0")
    ref = run_problem(ctx, p)
    assert "_splitk" in ctx.last_kernel, ctx.last_kernel
    force(spec)
    got = run_problem(ctx, p)
    assert "_csplit" in ctx.last_kernel, ctx.last_kernel
    assert torch.equal(got.view(torch.int32), ref.view(torch.int32)), ctx.last_kernel
    R, T = oracle.gemm(p)
    parity.check(oracle.decode(got), R, T, "f32", what=f"{spec} {ctx.last_kernel}")


@pytest.mark.parametrize("ab,c", DT_PAIRS)
@pytest.mark.parametrize("ldc_pad", [0, 3])
@pytest.mark.parametrize("beta", [0.0, 1.0])
def test_cluster_split_outputs(ctx, force, ab, c, ldc_pad, beta):
    """Every output type of the on-chip reduction: 16-byte / 8-byte stores of
    whole column groups, element stores at the ragged right edge and when
    C's rows are not 16-byte multiples (ldc = N + 3), C_old read or not."""
    force("bn=64 split=7")
    N = 190
    p = synthetic.make_problem(250, N, 2500, ab, c, alpha=1.25, beta=beta, seed=137, dist="normal",
                               c_fill="uniform", ldc=N + ldc_pad if ldc_pad else 0)
    out = run_problem(ctx, p, ldc=N + ldc_pad if ldc_pad else 0)
    assert "_csplit" in ctx.last_kernel and ctx.last_kernel.endswith("_s7"), ctx.last_kernel
    R, T = oracle.gemm(p)
    parity.check(oracle.decode(out)[:, :N], R, T, c, what=f"{ctx.last_kernel}")


def test_padded_leading_dimensions(ctx):
    for ta, tb in LAYOUTS:
        M, N, K = 150, 170, 190
        r8 = lambda x: (x + 7) // 8 * 8      # noqa: E731  (16-byte multiple rows: no repacking)
        p = synthetic.make_problem(M, N, K, "bf16", "f32", transpose_a=ta, transpose_b=tb, seed=31,
                                   dist="normal", beta=1.0, c_fill="uniform",
                                   lda=r8(M if ta else K) + 24, ldb=r8(K if tb else N) + 8, ldc=N + 40)
        check_full(ctx, p, f"padded {p.layout}")
        assert "pack" not in ctx.last_kernel
        q = synthetic.make_problem(M, N, K, "bf16", "f32", transpose_a=ta, transpose_b=tb, seed=32,
                                   dist="normal", lda=(M if ta else K) + 3, ldb=(K if tb else N) + 5,
                                   ldc=N + 1)
        check_full(ctx, q, f"odd-padded {q.layout}")


# ----------------------------------------------------- exactness and edges

@pytest.mark.parametrize("spec", ["", "bn=64", "cg=1 bn=192", "bn=128 split=4", "bn=128 split=4 csplit=0",
                                  "bn=64 split=16", "pack=1 bn=256 split=2",
                                  "sms=5 tail=3", "cg=2", "cg=2 bn=128 sms=4 tail=2", "store=direct",
                                  "cg=2 bn=192", "cg=2 bn=192 sms=4 tail=2", "cg=2 bn=192 chunk=0"])
@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_integer_inputs_bitwise(ctx, force, spec, ta, tb):
    """Integer entries in [-4,4], K=2048: every partial sum is an integer
    below 2^24, so fp32 accumulation is exact in any order."""
    force(spec)
    p = synthetic.make_problem(300, 260, 2048, "bf16", "f32", transpose_a=ta, transpose_b=tb,
                               alpha=0.5, beta=1.0, seed=41, dist="int", scale=4, c_fill="int")
    out = run_problem(ctx, p)
    R, _ = oracle.gemm(p)
    assert np.array_equal(oracle.decode(out), R), ctx.last_kernel


@pytest.mark.parametrize("spec", ["", "cg=2 bn=256", "cg=2 bn=128", "cg=1 bn=256", "cg=1 bn=192", "cg=1 bn=64",
                                  "bn=128 split=3", "cg=2 sms=8 tail=3", "cg=2 bn=192", "cg=2 bn=192 sms=4 tail=2"])
@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_chunked_descriptors_bitwise(ctx, force, spec, ta, tb):
    """An MN-major operand whose extent is a multiple of 64 is read with one
    3-D copy per K block (64-wide chunks as a third dimension); the result
    equals that of one copy per chunk bit for bit (same bytes, same MMAs).
    576 rows and 448 columns end inside a tile, so the last tiles' upper
    chunks lie past the operand and must read as zeros; K = 1000 is ragged."""
    p = synthetic.make_problem(576, 448, 1000, "bf16", "f32", transpose_a=ta, transpose_b=tb, alpha=0.75,
                               beta=0.5, seed=91, dist="normal", c_fill="uniform")
    force((spec + " chunk=0").strip())
    ref = run_problem(ctx, p)
    force(spec)
    got = run_problem(ctx, p)
    assert torch.equal(got.view(torch.int32), ref.view(torch.int32)), ctx.last_kernel
    R, T = oracle.gemm(p)
    parity.check(oracle.decode(got), R, T, "f32", what=f"{spec} {ctx.last_kernel}")



@pytest.mark.parametrize("spec", ["cg=1 bn=192", "cg=1 bn=192 split=3", "cg=1 bn=192 store=direct",
                                  "cg=2 bn=192", "cg=2 bn=192 sms=4 tail=2", "cg=2 bn=192 store=direct"])
@pytest.mark.parametrize("c", ["f16", "f32"])
def test_single_buffer_epilogue_192(ctx, force, spec, c):
    """The 192-wide kernels stage their epilogue in one buffer per warp (for
    one more pipeline stage): TMA-stored C, C through the transpose buffer
    (an odd ldc, beta != 0 so C_old is read back through it too), plain
    stores, and split-K partials all go through that one buffer."""
    force(spec)
    for ldc in (0, 389):
        p = synthetic.make_problem(700, 384, 1500, "f16", c, transpose_b=True, alpha=0.75, beta=-0.5, seed=93,
                                   dist="normal", c_fill="uniform", ldc=ldc)
        out = run_problem(ctx, p, ldc=ldc)
        assert ("256x192_pair" if "cg=2" in spec else "128x192") in ctx.last_kernel, ctx.last_kernel
        R, T = oracle.gemm(p)
        parity.check(oracle.decode(out)[:, :384], R, T, c, what=f"{spec} ldc={ldc} {ctx.last_kernel}")


@pytest.mark.parametrize("bn", [128, 192, 256])
def test_pair_width_first_call_in_fresh_context(force, bn):
    """Each CTA-pair tile width queries its own residency (pairs that fit
    at once) on its first use in a context."""
    c = tg.Context(0)
    try:
        force(f"cg=2 bn={bn}")
        p = synthetic.make_problem(520, 400, 300, "f16", "f32", seed=95, dist="normal")
        out = run_problem(c, p)
        assert f"256x{bn}_pair" in c.last_kernel, c.last_kernel
        R, T = oracle.gemm(p)
        parity.check(oracle.decode(out), R, T, "f32", what=c.last_kernel)
    finally:
        c.close()


@pytest.mark.parametrize("M", [1, 4, 7, 9, 100, 127])
@pytest.mark.parametrize("ta,tb", LAYOUTS)
@pytest.mark.parametrize("spec", ["", "cg=1 bn=128", "bn=128 split=4"])
def test_short_a_copies_bitwise(ctx, force, M, ta, tb, spec):
    """A one-CTA tile over fewer than 128 rows of a K-major A copies only the
    rows that exist (rounded up to 8); the tile's other rows hold stale
    shared memory and feed only output rows beyond M.  The result equals
    that of full 128-row copies bit for bit."""
    p = synthetic.make_problem(M, 700, 2100, "bf16", "f32", transpose_a=ta, transpose_b=tb, alpha=0.75, beta=0.5,
                               seed=M + 95, dist="normal", c_fill="uniform")
    force(spec + " shorta=0 gemv=0")
    ref = run_problem(ctx, p)
    force(spec + " gemv=0")
    got = run_problem(ctx, p)
    assert ctx.last_kernel.startswith("tcgen05_"), ctx.last_kernel
    assert torch.equal(got.view(torch.int32), ref.view(torch.int32)), ctx.last_kernel
    R, T = oracle.gemm(p)
    parity.check(oracle.decode(got), R, T, "f32", what=f"{spec} M={M} {ctx.last_kernel}")


def test_rank_one_exact(ctx):
    for dt in ("f16", "bf16"):
        p = synthetic.make_problem(190, 170, 1, dt, "f32", seed=43, dist="normal")
        out = run_problem(ctx, p)
        R, _ = oracle.gemm(p)
        assert np.array_equal(oracle.decode(out), R)


def test_beta_zero_ignores_nan_c(ctx):
    for ab, c in DT_PAIRS:
        p = synthetic.make_problem(200, 130, 70, ab, c, seed=47, dist="normal", c_fill="nan")
        out = run_problem(ctx, p)
        assert torch.isfinite(out.float()).all(), ctx.last_kernel
    p = synthetic.make_problem(64, 64, 64, "f32", "f32", seed=48, c_fill="nan")
    assert torch.isfinite(run_problem(ctx, p)).all()


def test_worked_example_2x2(ctx):
    """Foundry metal.md "Quick Start": A = {1,2,3,4}, B = {5,6,7,8} -> {19,22,43,50}."""
    for dt in ("f16", "bf16", "f32"):
        for ta, tb in LAYOUTS:
            A = torch.tensor([[1.0, 2.0], [3.0, 4.0]])
            B = torch.tensor([[5.0, 6.0], [7.0, 8.0]])
            p = synthetic.Problem(2, 2, 2, dt, dt, ta, tb, 1.0, 0.0,
                                  (A.T if ta else A).contiguous().to(synthetic.DTYPES[dt]),
                                  (B.T if tb else B).contiguous().to(synthetic.DTYPES[dt]),
                                  torch.zeros(2, 2, dtype=synthetic.DTYPES[dt]))
            out = run_problem(ctx, p)
            assert out.double().flatten().tolist() == [19, 22, 43, 50]


def test_identity_and_permutation(ctx):
    n = 300
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(3))
    P = torch.zeros(n, n)
    P[torch.arange(n), perm] = 1.0
    p = synthetic.make_problem(n, 200, n, "bf16", "f32", seed=5, dist="normal")
    p.A = P.to(torch.bfloat16)
    out = run_problem(ctx, p)
    assert torch.equal(out, p.B.float()[perm])


@pytest.mark.parametrize("spec", ["", "bn=128 split=6", "bn=128 split=6 csplit=0", "bn=64 split=16",
                                  "sms=9 tail=2", "cg=2 sms=8 tail=2"])
def test_determinism(ctx, force, spec):
    force(spec)
    p = synthetic.make_problem(384, 512, 4096, "bf16", "f32", transpose_a=True, seed=53, dist="normal")
    outs = [run_problem(ctx, p) for _ in range(5 if not spec else 10)]
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_transpose_flags_match_explicit_copies(ctx):
    """op() through the flags equals the product of explicitly transposed
    copies, bitwise."""
    base = synthetic.make_problem(300, 260, 520, "f16", "f32", seed=59, dist="normal")
    ref = run_problem(ctx, base)
    for ta, tb in LAYOUTS[1:]:
        q = synthetic.Problem(300, 260, 520, "f16", "f32", ta, tb, 1.0, 0.0,
                              base.A.T.contiguous() if ta else base.A,
                              base.B.T.contiguous() if tb else base.B, torch.zeros(300, 260))
        assert torch.equal(run_problem(ctx, q), ref), (ta, tb)


def test_refused_call_launches_nothing(ctx):
    before = ctx.launch_count
    A = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    d = tg.make_desc(64, 64, 64, "bf16", "bf16", alpha=float("nan"))
    with pytest.raises(tg.TcError):
        tg.tc_gemm(ctx, d, A, A, C)
    d = tg.make_desc(64, 64, 64, "bf16", "bf16")
    with pytest.raises(tg.TcError):
        tg.tc_gemm(ctx, d, A, A, A)          # C overlaps A
    with pytest.raises(ValueError):
        tg.tc_gemm(ctx, tg.make_desc(65, 64, 64, "bf16", "bf16"), A, A, C)   # capacity
    assert ctx.launch_count == before


# ----------------------------------------------------- batched / grouped / streams

@pytest.mark.parametrize("spec", ["", "pack=1", "bn=128 split=3", "cg=2 bn=192"])
def test_batched(ctx, force, spec):
    force(spec)
    M, N, K, batch = 200, 136, 264, 3
    g = torch.Generator().manual_seed(61)
    A = (torch.randn(batch, M, K, generator=g)).to(torch.bfloat16)
    B = (torch.randn(batch, K, N, generator=g)).to(torch.bfloat16)
    C = torch.zeros(batch, M, N)
    Ad, Bd, Cd = A.cuda(), B.cuda(), C.cuda()
    bd = tg.tc_gemm_batched_desc(tg.make_desc(M, N, K, "bf16", "f32"), batch, M * K, K * N, M * N)
    tg.tc_gemm_batched(ctx, bd, Ad, Bd, Cd)
    out = Cd.cpu()
    for i in range(batch):
        p = synthetic.Problem(M, N, K, "bf16", "f32", A=A[i], B=B[i], C=C[i])
        R, T = oracle.gemm(p)
        parity.check(out[i].numpy(), R, T, "f32", what=f"batch {i} {ctx.last_kernel}")
    # one B shared by every entry (stride 0) and a K shorter than lda
    bd = tg.tc_gemm_batched_desc(tg.make_desc(M, N, K - 1, "bf16", "f32", lda=K), batch, M * K, 0, M * N)
    tg.tc_gemm_batched(ctx, bd, Ad, Bd, Cd)
    out = Cd.cpu()
    for i in range(batch):
        R, T = oracle.gemm(synthetic.Problem(M, N, K - 1, "bf16", "f32", A=A[i][:, : K - 1].contiguous(),
                                             B=B[0][: K - 1].contiguous(), C=C[i]))
        parity.check(out[i].numpy(), R, T, "f32", what=f"shared-B batch {i} {ctx.last_kernel}")


def test_grouped_ragged(ctx):
    probs = synthetic.fp16_ragged(count=8, hi=700, seed=71)
    s = tg.Stream(ctx)
    As = [p.A.cuda() for p in probs]
    Bs = [p.B.cuda() for p in probs]
    Cs = [p.C.cuda() for p in probs]
    descs = [tg.make_desc(p.M, p.N, p.K, "f16", "f16") for p in probs]
    tg.tc_gemm_grouped_async(ctx, descs, As, Bs, Cs, s)
    s.sync()
    for p, C in zip(probs, Cs):
        R, T = oracle.gemm(p)
        parity.check(oracle.decode(C.cpu()), R, T, "f16", what=f"ragged {p.M}x{p.N}x{p.K}")
    s.close()


def _shifted(t, off):
    """A device copy of t whose first element sits `off` elements past a
    256-byte aligned allocation (so its base is misaligned for off % 8 != 0)."""
    flat = torch.empty(off + t.numel(), dtype=t.dtype, device="cuda")
    flat[off:] = t.reshape(-1).cuda()
    return flat[off:]


@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_repack_every_misalignment(ctx, ta, tb):
    # every 2-byte offset of the base inside a 16-byte word, with odd leading
    # dimensions: the repack kernel's shifted 16-byte loads and row tails
    M, N, K = 150, 97, 203
    for off in range(8):
        a_cols, b_cols = (M if ta else K), (K if tb else N)
        lda = a_cols + 2 * off + (1 - a_cols % 2)            # odd
        ldb = b_cols + 2 * (7 - off) + (1 - b_cols % 2)      # odd
        p = synthetic.make_problem(M, N, K, "f16", "f32", transpose_a=ta, transpose_b=tb, seed=400 + off,
                                   dist="int", scale=3.0, lda=lda, ldb=ldb)
        A, B, C = _shifted(p.A, off), _shifted(p.B, (off * 3) % 8), p.C.cuda()
        d = tg.make_desc(M, N, K, "f16", "f32", transpose_a=ta, transpose_b=tb, lda=lda, ldb=ldb)
        tg.tc_gemm(ctx, d, A, B, C)
        assert "_packA_packB" in ctx.last_kernel
        R, _ = oracle.gemm(p)
        got = C.cpu().numpy().astype(np.float64)
        assert np.array_equal(got, R), f"offset {off}: {np.argwhere(got != R)[:5]}"


def _grouped_specs():
    """Problems of every dtype pair, layout, alpha/beta, aligned and ragged
    shapes, padded leading dims, plus two fp32 problems; more than one
    table of problems (the launch takes at most 64)."""
    g = torch.Generator().manual_seed(91)
    specs = []
    for i in range(70):
        ab, c = DT_PAIRS[i % 4]
        ta, tb = LAYOUTS[(i // 4) % 4]
        M, N, K = (int(v) for v in torch.randint(1, 400, (3,), generator=g))
        if i % 5 == 0:
            M, N, K = 128 * (1 + i % 3), 64 * (1 + i % 4), 64 * (1 + i % 5)   # TMA-aligned C
        alpha, beta = [(1.0, 0.0), (0.5, 1.0), (-1.5, 0.25)][i % 3]
        pad = (i % 7 == 3)
        specs.append(dict(M=M, N=N, K=K, ab=ab, c=c, ta=ta, tb=tb, alpha=alpha, beta=beta, pad=pad,
                          dist="int" if i % 2 else "normal"))
    specs.append(dict(M=33, N=17, K=65, ab="f32", c="f32", ta=False, tb=True, alpha=1.0, beta=0.0,
                      pad=False, dist="normal"))
    specs.append(dict(M=70, N=90, K=9, ab="f32", c="f32", ta=True, tb=False, alpha=0.5, beta=1.0,
                      pad=False, dist="int"))
    return specs


def _run_grouped(ctx, specs, seed0):
    probs, descs, As, Bs, Cs = [], [], [], [], []
    for j, sp in enumerate(specs):
        a_cols = sp["M"] if sp["ta"] else sp["K"]
        b_cols = sp["K"] if sp["tb"] else sp["N"]
        lda, ldb, ldc = (a_cols + 5, b_cols + 8, sp["N"] + 3) if sp["pad"] else (0, 0, 0)
        p = synthetic.make_problem(sp["M"], sp["N"], sp["K"], sp["ab"], sp["c"], transpose_a=sp["ta"],
                                   transpose_b=sp["tb"], alpha=sp["alpha"], beta=sp["beta"], seed=seed0 + j,
                                   dist=sp["dist"], scale=3.0,
                                   c_fill=("int" if sp["dist"] == "int" else "uniform") if sp["beta"] else "zero",
                                   lda=lda, ldb=ldb, ldc=ldc)
        probs.append(p)
        As.append(p.A.cuda())
        Bs.append(p.B.cuda())
        Cs.append(p.C.cuda())
        descs.append(tg.make_desc(p.M, p.N, p.K, p.ab_dtype, p.c_dtype, transpose_a=p.transpose_a,
                                  transpose_b=p.transpose_b, alpha=p.alpha, beta=p.beta,
                                  lda=p.A.shape[1], ldb=p.B.shape[1], ldc=p.C.shape[1]))
    s = tg.Stream(ctx)
    tg.tc_gemm_grouped_async(ctx, descs, As, Bs, Cs, s)
    s.sync()
    s.close()
    return probs, [C.cpu() for C in Cs]


@pytest.mark.parametrize("spec", ["", "cg=1 bn=128", "cg=2 bn=128", "cg=1 bn=256", "store=direct",
                                  "grouped=0"])
def test_grouped_mixed(ctx, force, spec):
    force(spec)
    specs = _grouped_specs()
    probs, outs = _run_grouped(ctx, specs, 500)
    if spec != "grouped=0":
        assert ctx.last_kernel.startswith("grouped_tcgen05_"), ctx.last_kernel
    for sp, p, out in zip(specs, probs, outs):
        R, T = oracle.gemm(p)
        got = oracle.decode(out)[:, : p.N]
        what = f"{spec or 'default'} {sp} {ctx.last_kernel}"
        if sp["dist"] == "int" and p.c_dtype == "f32" and p.ab_dtype != "f32":
            # integer data with alpha, beta in {1, 0.5, -1.5, 0.25}: exact
            assert np.array_equal(got, R), what
        else:
            parity.check(got, R, T, p.c_dtype, exact_f32=(p.ab_dtype == "f32"), what=what)


def test_grouped_deterministic(ctx):
    specs = _grouped_specs()[:20]
    _, first = _run_grouped(ctx, specs, 700)
    _, second = _run_grouped(ctx, specs, 700)
    bits = lambda t: t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)
    for a, b in zip(first, second):
        assert torch.equal(bits(a), bits(b))


def test_torch_stream_wrap(ctx):
    ts = torch.cuda.Stream()
    s = tg.Stream(ctx, torch_stream=ts)
    p = synthetic.make_problem(256, 256, 512, "bf16", "bf16", seed=73, dist="normal")
    out = run_problem(ctx, p, stream=s)
    R, T = oracle.gemm(p)
    parity.check(oracle.decode(out), R, T, "bf16", what="wrapped stream")
    s.close()


def test_host_buffers(ctx):
    p = synthetic.make_problem(300, 200, 256, "bf16", "f32", beta=1.0, seed=79, dist="normal",
                               c_fill="uniform")
    A, B, C = p.A.pin_memory(), p.B.pin_memory(), p.C.clone().pin_memory()
    d = tg.make_desc(p.M, p.N, p.K, "bf16", "f32", beta=1.0)
    tg.tc_gemm_host(ctx, d, A, B, C)
    R, T = oracle.gemm(p)
    parity.check(C.numpy(), R, T, "f32", what="host buffers")


@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_host_buffers_banded(ctx, ta, tb):
    """M large enough for the host call to move A and C in row bands (the
    last one ragged), with C read (beta != 0) and padded leading dims."""
    M, N, K = 5000, 300, 256
    p = synthetic.make_problem(M, N, K, "bf16", "f32", transpose_a=ta, transpose_b=tb, alpha=0.5, beta=1.0,
                               seed=80, dist="normal", c_fill="uniform", lda=(M if ta else K) + 8,
                               ldb=(K if tb else N) + 3, ldc=N + 5)
    A, B, C = p.A.pin_memory(), p.B.pin_memory(), p.C.clone().pin_memory()
    d = tg.make_desc(M, N, K, "bf16", "f32", transpose_a=ta, transpose_b=tb, alpha=0.5, beta=1.0,
                     lda=A.shape[1], ldb=B.shape[1], ldc=C.shape[1])
    tg.tc_gemm_host(ctx, d, A, B, C)
    R, T = oracle.gemm(p)
    parity.check(C.numpy()[:, :N], R, T, "f32", what=f"host banded {p.layout} {ctx.last_kernel}")
    assert torch.equal(C[:, N:], p.C[:, N:])       # the padding of C is not written


# ----------------------------------------------------- the named workloads

def test_fp32_nn_256(ctx):
    stats = check_full(ctx, synthetic.fp32_nn_256(), "fp32 NN 256^3")
    assert ctx.last_kernel.startswith("ffma_f32_nn")
    assert stats["max_err_over_T"] < 1e-5


def test_bf16_nn_4096(ctx):
    check_sampled(ctx, synthetic.bf16_nn_4096(), what="bf16 NN 4096^3")
    assert "split" not in ctx.last_kernel


@pytest.mark.parametrize("layout", ["TN", "NT"])
def test_bf16_tn_nt_4096x8192(ctx, layout):
    check_sampled(ctx, synthetic.bf16_tn_nt_4096x8192(layout), what=f"bf16 {layout} 4096x4096x8192")


def test_bf16_tn_splitk_256x16384(ctx, force):
    check_full(ctx, synthetic.bf16_tn_splitk_256x16384(), "bf16 TN split-K 256x256x16384")
    assert "_csplit_s" in ctx.last_kernel, ctx.last_kernel
    force("csplit=0")
    check_full(ctx, synthetic.bf16_tn_splitk_256x16384(), "bf16 TN split-K 256x256x16384 through memory")
    assert "_splitk" in ctx.last_kernel, ctx.last_kernel


def test_fp16_nn_narrow_8192x384(ctx):
    check_sampled(ctx, synthetic.fp16_nn_narrow_8192x384x4096(), what="fp16 NN 8192x384x4096")
    assert ctx.last_kernel.endswith("256x192_pair")


@pytest.mark.parametrize("n", synthetic.SQUARE_SIZES)
def test_fp16_square_sweep(ctx, n):
    p = synthetic.fp16_nn_square(n)
    if n <= 512:
        check_full(ctx, p, f"fp16 {n}^3")
    else:
        check_sampled(ctx, p, n=1500, what=f"fp16 {n}^3")


def test_fp16_ragged_64(ctx):
    probs = synthetic.fp16_ragged()
    s = tg.Stream(ctx)
    As = [p.A.cuda() for p in probs]
    Bs = [p.B.cuda() for p in probs]
    Cs = [p.C.cuda() for p in probs]
    tg.tc_gemm_grouped_async(ctx, [tg.make_desc(p.M, p.N, p.K, "f16", "f16") for p in probs],
                             As, Bs, Cs, s)
    s.sync()
    rng = np.random.default_rng(4)
    for p, C in zip(probs, Cs):
        rows, cols = parity.sample_points(p.M, p.N, 200, rng)
        R, T = oracle.gemm_points(p, rows, cols)
        parity.check(oracle.decode(C.cpu())[rows, cols], R, T, "f16",
                     what=f"ragged {p.M}x{p.N}x{p.K}")
    s.close()
