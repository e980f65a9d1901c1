"""Failure detection on the GPU without a fault: every device wait of the
tensor-core kernel is bounded.  A test hook makes the MMA warp withhold the
first tile's "accumulator ready" signal (a flag that nothing sets), so the
epilogue's wait runs out after a short limit; the kernel records the expiry,
lets its in-flight copies and MMAs land, frees TMEM and returns.  The host
must read TC_ERR_DEVICE_TIMEOUT, and the same context must still compute
correct results afterwards."""
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


# One CTA; a CTA pair (tcgen05.mma.cta_group::2: the even CTA issues the
# MMAs and both CTAs' epilogues wait, then both meet at the cluster barrier
# before TMEM is freed); a cluster split (four K slices, each CTA's epilogue
# waits, then the cluster's two barriers around the on-chip reduction).
@pytest.mark.parametrize("spec,kernel", [("cg=1 bn=128", "128x128"), ("cg=2 bn=256", "256x256_pair"),
                                         ("bn=128 split=4", "128x128_csplit_s4")])
def test_expired_wait_is_reported_and_context_survives(monkeypatch, spec, kernel):
    ctx = tg.Context(0)
    p = synthetic.make_problem(256, 256, 256, "bf16", "f32", seed=5, dist="normal")
    A, B = p.A.cuda(), p.B.cuda()
    C = torch.zeros(256, 256, device="cuda")
    d = tg.make_desc(256, 256, 256, "bf16", "f32")

    monkeypatch.setenv("TC_FORCE_VARIANT", f"{spec} debug_drop=1 debug_timeout_ms=200")
    with pytest.raises(tg.TcError) as err:
        tg.tc_gemm(ctx, d, A, B, C)
    assert err.value.status == tg.TC_ERR_DEVICE_TIMEOUT
    assert kernel in ctx.last_kernel, ctx.last_kernel

    # the status was consumed; the context and the device still work
    monkeypatch.delenv("TC_FORCE_VARIANT")
    torch.cuda.synchronize()
    tg.tc_gemm(ctx, d, A, B, C)
    R, T = oracle.gemm(p)
    parity.check(C.cpu().numpy(), R, T, "f32", what=f"after a reported timeout {ctx.last_kernel}")
    ctx.close()
