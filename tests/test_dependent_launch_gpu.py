"""Back-to-back launches on one stream, each consuming what the one before
wrote.  The library launches most kernels as programmatic dependents of the
previous kernel in the stream: the next kernel's CTAs start their set-up
while the previous one still runs and wait (griddepcontrol.wait) before any
global access.  A kernel that read its operands, or wrote C, before that
wait would read stale values or overwrite ones still being read; these
chains would then differ from the expected values.

Every link multiplies by a signed permutation (synthetic.signed_permutation)
or accumulates integers, so each expected value is exact: the oracle checks
the first link of each chain, and the later links follow from it by the
same column permutation (for integer data below 2^24 every path is exact)."""
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

LINKS = 6


@pytest.fixture(scope="module")
def ctx():
    c = tg.Context(0)
    yield c
    c.close()


@pytest.fixture
def force(monkeypatch):
    def set_(spec: str):
        monkeypatch.setenv("TC_FORCE_VARIANT", spec)
    yield set_


def ternary(rows, cols, seed, dtype):
    """Integer entries in {-1, 0, 1} (synthetic's "int" draw with scale 1)."""
    return synthetic.make_problem(rows, 1, cols, "f32", "f32", seed=seed, dist="int", scale=1.0).A.to(dtype)


def first_link_by_oracle(X, P, ab, c):
    """X @ P through the oracle (the first link of a chain)."""
    p = synthetic.Problem(X.shape[0], P.shape[1], X.shape[1], ab, c, A=X.cpu(), B=P.to(X.dtype).cpu(),
                          C=torch.zeros(X.shape[0], P.shape[1], dtype=synthetic.DTYPES[c]))
    R, _ = oracle.gemm(p)
    return R


@pytest.mark.parametrize("M,n,ab,spec", [(2048, 2048, "bf16", ""), (4096, 4096, "bf16", ""),
                                         (8192, 384, "f16", ""), (512, 512, "bf16", ""),
                                         (1024, 1024, "f16", ""), (1024, 1024, "f16", "bn=128 split=2 csplit=0"),
                                         (4096, 4096, "bf16", "cg=1 bn=256")])
def test_gemm_chain(ctx, force, M, n, ab, spec):
    """X_{i+1} = X_i @ P_i, ping-ponging between two buffers: each GEMM reads
    the previous one's output (read after write) and overwrites the buffer
    the previous one read (write after read)."""
    force(spec)
    dt = synthetic.DTYPES[ab]
    X0 = ternary(M, n, 100 + n, dt)
    perms = [synthetic.signed_permutation(n, 200 + i) for i in range(LINKS)]
    Ps = [P.to(dt).cuda() for P, _, _ in perms]
    bufs = [X0.cuda(), torch.full((M, n), float("nan"), dtype=dt, device="cuda")]
    st = tg.Stream(ctx)
    d = tg.make_desc(M, n, n, ab, ab)
    for i in range(LINKS):
        tg.tc_gemm_async(ctx, d, bufs[i % 2], Ps[i], bufs[(i + 1) % 2], st)
    st.sync()
    kernel = ctx.last_kernel
    want = first_link_by_oracle(X0, perms[0][0], ab, ab)
    assert np.array_equal(want, (X0.double().numpy()[:, perms[0][1]] * perms[0][2])), "oracle pin"
    for _, perm, s in perms[1:]:
        want = want[:, perm] * s
    got = bufs[LINKS % 2].cpu().double().numpy()
    assert np.array_equal(got, want), (kernel, int((got != want).sum()))


@pytest.mark.parametrize("spec", ["", "csplit=0", "bn=128 split=16"])
def test_splitk_accumulate_chain(ctx, force, spec):
    """C = A^T B + C, LINKS times back to back on the split-K shape (TN,
    256 x 256 x 16384, f32 out): every launch reads the C the previous one
    wrote, through the cluster reduction or the reduction kernel."""
    force(spec)
    p = synthetic.make_problem(256, 256, 16384, "bf16", "f32", transpose_a=True, beta=1.0, seed=31, dist="int",
                               scale=1.0, c_fill="int")
    R, _ = oracle.gemm(p)                       # A^T B + C0, exact
    C0 = p.C.double().numpy()
    want = C0 + LINKS * (R - C0)
    A, B, C = p.A.cuda(), p.B.cuda(), p.C.cuda()
    d = tg.make_desc(256, 256, 16384, "bf16", "f32", transpose_a=True, beta=1.0)
    st = tg.Stream(ctx)
    for _ in range(LINKS):
        tg.tc_gemm_async(ctx, d, A, B, C, st)
    st.sync()
    assert np.array_equal(C.cpu().double().numpy(), want), ctx.last_kernel


@pytest.mark.parametrize("rows", [4096, 5003])
@pytest.mark.parametrize("spec", ["", "gemv_rr=0"])
def test_skinny_chain(ctx, force, rows, spec):
    """x_{i+1} = x_i @ W_i^T (W stored [N, K], a signed permutation) at the
    decode width: the row-range skinny kernel back to back (5003 rows: whole
    16-row blocks per CTA), and the cluster form."""
    force(spec)
    n = rows
    x0 = ternary(4, n, 300 + n, torch.float16)
    perms = [synthetic.signed_permutation(n, 400 + i, torch.float16) for i in range(LINKS)]
    # W = P^T stored [N, K]: x @ W^T = x @ P
    Ws = [P.t().contiguous().cuda() for P, _, _ in perms]
    bufs = [x0.cuda(), torch.full((4, n), float("nan"), dtype=torch.float16, device="cuda")]
    st = tg.Stream(ctx)
    d = tg.make_desc(4, n, n, "f16", "f16", transpose_b=True)
    for i in range(LINKS):
        tg.tc_gemm_async(ctx, d, bufs[i % 2], Ws[i], bufs[(i + 1) % 2], st)
    st.sync()
    assert ctx.last_kernel.startswith("gemv_"), ctx.last_kernel
    want = x0.double().numpy()
    for _, perm, s in perms:
        want = want[:, perm] * s
    assert np.array_equal(bufs[LINKS % 2].cpu().double().numpy(), want), ctx.last_kernel


def test_relaxed_chain(ctx):
    """The relaxed fp32 path (a split pass, then the GEMM over the split
    operands) chained: X_{i+1} = X_i @ P_i in fp32."""
    n = 1024
    X0 = ternary(1024, n, 500, torch.float32)
    perms = [synthetic.signed_permutation(n, 600 + i) for i in range(LINKS)]
    Ps = [P.cuda() for P, _, _ in perms]
    bufs = [X0.cuda(), torch.full((1024, n), float("nan"), device="cuda")]
    st = tg.Stream(ctx)
    d = tg.make_desc(1024, n, n, "f32", "f32")
    for i in range(LINKS):
        tg.tc_gemm_f32_relaxed_async(ctx, d, bufs[i % 2], Ps[i], bufs[(i + 1) % 2], st)
    st.sync()
    want = X0.double().numpy()
    for _, perm, s in perms:
        want = want[:, perm] * s
    assert np.array_equal(bufs[LINKS % 2].cpu().double().numpy(), want), ctx.last_kernel


def test_grouped_chain(ctx):
    """Three problems with odd row lengths (their operands go through the
    repacking pass, then one grouped launch), chained four times."""
    sizes = [(300, 257), (129, 511), (77, 1001)]
    X0s = [ternary(m, n, 700 + n, torch.float16) for m, n in sizes]
    perms = [[synthetic.signed_permutation(n, 800 + 10 * i + j) for j, (_, n) in enumerate(sizes)] for i in range(4)]
    bufs = [[x.cuda() for x in X0s], [torch.full((m, n), float("nan"), dtype=torch.float16, device="cuda")
                                      for m, n in sizes]]
    descs = [tg.make_desc(m, n, n, "f16", "f16") for m, n in sizes]
    st = tg.Stream(ctx)
    groups = []
    for i in range(4):
        Ps = [P.to(torch.float16).cuda() for P, _, _ in perms[i]]
        groups.append(tg.GroupedGemm(descs, bufs[i % 2], Ps, bufs[(i + 1) % 2]))
    for g in groups:
        g.enqueue(ctx, st)
    st.sync()
    for j, x0 in enumerate(X0s):
        want = x0.double().numpy()
        for i in range(4):
            _, perm, s = perms[i][j]
            want = want[:, perm] * s
        assert np.array_equal(bufs[0][j].cpu().double().numpy(), want), (j, ctx.last_kernel)


def test_torch_producer_then_gemm(ctx):
    """A PyTorch kernel writes the operand just before a dependent GEMM is
    enqueued on the same stream (an ordinary kernel never signals early: the
    GEMM's wait covers its whole run)."""
    n = 2048
    P, perm, s = synthetic.signed_permutation(n, 900)
    Pd = P.to(torch.bfloat16).cuda()
    src = ternary(n, n, 901, torch.bfloat16).cuda()
    A = torch.zeros(n, n, dtype=torch.bfloat16, device="cuda")
    C = torch.empty(n, n, dtype=torch.bfloat16, device="cuda")
    ts = torch.cuda.current_stream()
    st = tg.Stream(ctx, torch_stream=ts)
    d = tg.make_desc(n, n, n, "bf16", "bf16")
    for k in range(3):
        A.copy_(src * (k + 1))                    # a torch kernel on the same stream
        tg.tc_gemm_async(ctx, d, A, Pd, C, st)
        torch.cuda.synchronize()
        want = (src.cpu().double().numpy() * (k + 1))[:, perm] * s
        assert np.array_equal(C.cpu().double().numpy(), want), k
