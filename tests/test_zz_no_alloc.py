"""tc_gemm_splitk_noalloc: the split-K GEMM that allocates nothing.

Some callers cannot allocate device memory -- their device memory belongs to
another allocator with a fixed budget, or they cannot afford the
device-wide synchronisation of cudaMalloc/cudaFree.  For them the library
keeps the split-K partial tiles in a static device array and needs no
context.  This file checks, through the C ABI, that two calls in a
row give the same output as the ordinary entry point (tc_gemm) within the
parity bound used everywhere in these tests, and that requests beyond the
static array's size are refused.  It is named so that pytest collects it
last.
"""
from __future__ import annotations

import ctypes

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


def _noalloc(d, A, B, C, split, stream):
    """Call the entry point directly through the C ABI."""
    return tg.library().tc_gemm_splitk_noalloc(ctypes.byref(d), A.data_ptr(), B.data_ptr(), C.data_ptr(),
                                               split, ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("case", ["tn_splitk_256x256x16384", "nt_ragged_beta"])
def test_noalloc_matches_tc_gemm_twice(case):
    if case == "tn_splitk_256x256x16384":
        p = synthetic.bf16_tn_splitk_256x16384()
        split = 0
    else:
        p = synthetic.make_problem(300, 200, 3000, "f16", "f16", transpose_b=True, alpha=0.5, beta=-1.0,
                                   seed=101, dist="normal", c_fill="uniform")
        split = 5
    A, B = p.A.cuda(), p.B.cuda()
    d = tg.make_desc(p.M, p.N, p.K, p.ab_dtype, p.c_dtype, transpose_a=p.transpose_a,
                     transpose_b=p.transpose_b, alpha=p.alpha, beta=p.beta)

    ctx = tg.Context(0)
    C_ref = p.C.cuda()
    tg.tc_gemm(ctx, d, A, B, C_ref)                 # the existing entry point
    torch.cuda.synchronize()
    ctx.close()

    R, T = oracle.gemm(p)
    ref = oracle.decode(C_ref.cpu())
    parity.check(ref, R, T, p.c_dtype, what=f"tc_gemm {case}")
    lim = parity.bound(R, T, p.c_dtype)
    stream = torch.cuda.Stream()
    for call in range(2):
        C = p.C.cuda()
        with torch.cuda.stream(stream):
            st = _noalloc(d, A, B, C, split, stream)
        assert st == tg.TC_OK, tg.tc_status_string(st)
        stream.synchronize()
        got = oracle.decode(C.cpu())
        parity.check(got, R, T, p.c_dtype, what=f"noalloc call {call} {case}")
        assert np.all(np.abs(got - ref) <= lim), f"call {call}: differs from tc_gemm beyond the bound"


def test_noalloc_refuses_what_it_cannot_serve():
    stream = torch.cuda.Stream()
    A = torch.zeros(4096, 4096, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(4096, 4096, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(4096, 4096, dtype=torch.float32, device="cuda")
    d = tg.make_desc(4096, 4096, 4096, "bf16", "f32")
    # 1024 output tiles x 2 slices x 64 KiB of partials exceed the static array
    assert _noalloc(d, A, B, C, 2, stream) == tg.TC_ERR_SCRATCH
    d32 = tg.make_desc(64, 64, 64, "f32", "f32")
    assert _noalloc(d32, C, C[64:], C[128:], 0, stream) == tg.TC_ERR_DTYPE
    odd = tg.make_desc(64, 64, 63, "bf16", "f32")      # lda = 63: not TMA-addressable in place
    assert _noalloc(odd, A, B, C, 0, stream) == tg.TC_ERR_ALIGN_UNSUPPORTED
    stream.synchronize()
