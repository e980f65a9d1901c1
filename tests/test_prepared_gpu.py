"""PreparedGemm (arguments checked and marshalled once, then one C call per
enqueue) against the per-call wrappers: the same entry point on the same
buffers, so every output is bitwise equal, and within the oracle's bound."""
from __future__ import annotations

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


def twice(ctx, st, d, A, B, C, kw, per_call):
    """C from a prepared call (enqueued twice, C zeroed in between) and from
    the per-call wrapper."""
    C1, C2 = C.clone(), C.clone()
    prep = tg.PreparedGemm(ctx, d, A, B, C1, st, **kw)
    prep.enqueue()
    st.sync()
    first = C1.clone()
    C1.copy_(C)
    prep.enqueue()
    st.sync()
    assert torch.equal(first, C1), "a prepared call gives the same bits every time"
    per_call(C2)
    st.sync()
    assert torch.equal(C1, C2), ctx.last_kernel
    return C1


def test_prepared_plain_and_epilogue(ctx):
    st = tg.Stream(ctx)
    p = synthetic.make_problem(300, 200, 333, "bf16", "bf16", alpha=0.5, beta=1.0, seed=51, dist="normal",
                               c_fill="uniform")
    A, B, C = p.A.cuda(), p.B.cuda(), p.C.cuda()
    d = tg.make_desc(p.M, p.N, p.K, "bf16", "bf16", alpha=0.5, beta=1.0)
    out = twice(ctx, st, d, A, B, C, {}, lambda c: tg.tc_gemm_async(ctx, d, A, B, c, st))
    R, T = oracle.gemm(p)
    parity.check(oracle.decode(out.cpu()), R, T, "bf16", what=f"prepared {ctx.last_kernel}")
    bias = torch.randn(p.N, generator=torch.Generator().manual_seed(52)).to(torch.bfloat16).cuda()
    twice(ctx, st, d, A, B, C, {"bias": bias, "activation": "gelu_tanh"},
          lambda c: tg.tc_gemm_epilogue_async(ctx, d, A, B, c, st, bias=bias, activation="gelu_tanh"))
    assert "bias_gelu" in ctx.last_kernel, ctx.last_kernel


def test_prepared_relaxed_i8_q8_and_skinny(ctx):
    st = tg.Stream(ctx)
    p = synthetic.make_problem(256, 192, 320, "f32", "f32", seed=53, dist="uniform")
    A, B, C = p.A.cuda(), p.B.cuda(), p.C.cuda()
    d = tg.make_desc(p.M, p.N, p.K, "f32", "f32")
    twice(ctx, st, d, A, B, C, {"relaxed": True}, lambda c: tg.tc_gemm_f32_relaxed_async(ctx, d, A, B, c, st))
    assert ctx.last_kernel.startswith("relaxed_f32"), ctx.last_kernel

    g = torch.Generator().manual_seed(54)
    A8 = torch.randint(-128, 128, (256, 320), generator=g, dtype=torch.int8).cuda()
    B8 = torch.randint(-128, 128, (320, 192), generator=g, dtype=torch.int8).cuda()
    scale = torch.rand(192, generator=g).cuda()
    C32 = torch.zeros(256, 192, device="cuda")
    d8 = tg.make_desc(256, 192, 320, "i8", "f32")
    twice(ctx, st, d8, A8, B8, C32, {"col_scale": scale},
          lambda c: tg.tc_gemm_i8_dequant_async(ctx, d8, A8, B8, c, scale, st))

    q, qs = synthetic.q8_weight_problem(4, 1000, 4096, "f16", "f16", seed=55)
    X, W, Y, s = q.A.cuda(), q.B.cuda(), q.C.cuda(), qs.cuda()
    dq = tg.make_desc(4, 1000, 4096, "f16", "f16", transpose_b=True, b_dtype="i8")
    twice(ctx, st, dq, X, W, Y, {"q8_scale": s}, lambda c: tg.tc_gemm_q8_weight_async(ctx, dq, X, W, c, s, st))
    assert ctx.last_kernel.startswith("gemv_q8w"), ctx.last_kernel

    f = synthetic.f16_decode(1, 4096, 4096)
    X, W, Y = f.A.cuda(), f.B.cuda(), f.C.cuda()
    df = tg.make_desc(1, 4096, 4096, "f16", "f16", transpose_b=True)
    twice(ctx, st, df, X, W, Y, {}, lambda c: tg.tc_gemm_async(ctx, df, X, W, c, st))
    assert ctx.last_kernel.startswith("gemv_"), ctx.last_kernel
