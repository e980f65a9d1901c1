"""The C ABI on the host (no GPU needed): the library loads, exports every
symbol the header declares, refuses bad descriptors with the right status
before touching a device, and routes each workload to the intended variant.

Validation order and refusal-without-launch follow the tessl
architecture.md sections "GEMM Pipeline & Kernel Selection" (validate_gemm)
and "The Kernel Library and the nn Boundary" (checked multiply, capacity in
elements, non-zero dims, finite scalars, nothing encoded on error).
"""
from __future__ import annotations

import ctypes
import math
import os
import re

import pytest
import torch

import matrix_multiply_gb300 as tg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tcgemm.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tc_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_binding_surface():
    assert set(declared_functions()) == set(tg.EXPORTED)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(tg.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_ctx_create_without_device_reports_cuda_error():
    p = ctypes.c_void_p(12345)
    st = tg.library().tc_ctx_create(ctypes.byref(p), 0)
    assert st == tg.TC_ERR_CUDA
    assert p.value is None


def test_status_strings():
    for code in tg.STATUS:
        assert tg.tc_status_string(code) not in ("", "unknown status")
    assert tg.tc_status_string(999) == "unknown status"


def desc(**kw):
    base = dict(M=64, N=48, K=32, a_dtype="bf16", c_dtype="bf16")
    base.update(kw)
    M, N, K = base.pop("M"), base.pop("N"), base.pop("K")
    return tg.make_desc(M, N, K, base.pop("a_dtype"), base.pop("c_dtype"), **base)


def test_valid_descriptor_passes():
    assert tg.tc_gemm_validate(desc()) == tg.TC_OK
    for ta in (False, True):
        for tb in (False, True):
            assert tg.tc_gemm_validate(desc(transpose_a=ta, transpose_b=tb)) == tg.TC_OK


@pytest.mark.parametrize("kw,status", [
    (dict(M=0), tg.TC_ERR_DIM), (dict(N=-3), tg.TC_ERR_DIM), (dict(K=0), tg.TC_ERR_DIM),
    (dict(lda=31), tg.TC_ERR_LD), (dict(ldb=47), tg.TC_ERR_LD), (dict(ldc=47), tg.TC_ERR_LD),
    (dict(lda=-1), tg.TC_ERR_LD),
    (dict(transpose_a=True, lda=63), tg.TC_ERR_LD),        # A stored [K,M]: lda >= M
    (dict(transpose_b=True, ldb=31), tg.TC_ERR_LD),        # B stored [N,K]: ldb >= K
    (dict(alpha=math.inf), tg.TC_ERR_SCALAR), (dict(beta=math.nan), tg.TC_ERR_SCALAR),
    (dict(c_dtype="f16"), tg.TC_ERR_DTYPE),                # bf16 in, f16 out
    (dict(a_dtype="f32", c_dtype="bf16"), tg.TC_ERR_DTYPE),
])
def test_refusals(kw, status):
    assert tg.tc_gemm_validate(desc(**kw)) == status


def test_dtype_rules():
    d = desc()
    d.b_dtype = tg.TC_F16
    assert tg.tc_gemm_validate(d) == tg.TC_ERR_DTYPE      # A and B must match
    d = desc()
    d.accum_dtype = tg.TC_F16
    assert tg.tc_gemm_validate(d) == tg.TC_ERR_DTYPE      # fp32 accumulation only
    d = desc()
    d.a_dtype = d.b_dtype = 7
    assert tg.tc_gemm_validate(d) == tg.TC_ERR_DTYPE
    for ab, c in [("f16", "f16"), ("f16", "f32"), ("bf16", "f32"), ("f32", "f32")]:
        assert tg.tc_gemm_validate(desc(a_dtype=ab, c_dtype=c)) == tg.TC_OK


def test_null_pointers():
    assert tg.tc_gemm_validate(None) == tg.TC_ERR_NULL
    assert tg.tc_gemm_validate(desc(), A=0) == tg.TC_ERR_NULL
    assert tg.tc_gemm_validate(desc(), C=0) == tg.TC_ERR_NULL


def test_overlap():
    d = desc(M=64, N=64, K=64)             # A: 64*64*2 = 8192 bytes
    base = 1 << 30
    assert tg.tc_gemm_validate(d, A=base, B=base + (1 << 20), C=base + 8192) == tg.TC_OK
    assert tg.tc_gemm_validate(d, A=base, B=base + (1 << 20), C=base + 8190) == tg.TC_ERR_OVERLAP
    assert tg.tc_gemm_validate(d, A=base, B=base + (1 << 20), C=base + (1 << 20) - 100) == tg.TC_ERR_OVERLAP
    assert tg.tc_gemm_validate(d, A=base + (1 << 20), B=base + (2 << 20), C=base) == tg.TC_OK


def test_overflow_is_refused():
    # (rows-1)*ld + cols elements times the element size overflows int64
    d = desc(M=2**31 - 1, N=2**31 - 1, K=2**31 - 1, a_dtype="f32", c_dtype="f32")
    d.lda = 2**31 - 1
    st = tg.tc_gemm_validate(d, A=1 << 12, B=1 << 62, C=(1 << 62) + (1 << 61))
    assert st in (tg.TC_ERR_OVERFLOW, tg.TC_ERR_OVERLAP)
    bd = tg.tc_gemm_batched_desc(desc(M=1 << 30, N=1 << 30, K=8), 2**31 - 1, 1 << 60, 0, 1 << 61)
    assert tg.tc_gemm_batched_validate(bd) == tg.TC_ERR_OVERFLOW


def test_batched_strides():
    d = desc(M=16, N=16, K=16)
    ok = tg.tc_gemm_batched_desc(d, 4, 256, 256, 256)
    assert tg.tc_gemm_batched_validate(ok) == tg.TC_OK
    shared_b = tg.tc_gemm_batched_desc(d, 4, 256, 0, 256)     # one B for every entry
    assert tg.tc_gemm_batched_validate(shared_b) == tg.TC_OK
    clash = tg.tc_gemm_batched_desc(d, 4, 256, 256, 100)      # outputs overlap
    assert tg.tc_gemm_batched_validate(clash) == tg.TC_ERR_STRIDE
    neg = tg.tc_gemm_batched_desc(d, 4, -256, 256, 256)
    assert tg.tc_gemm_batched_validate(neg) == tg.TC_ERR_STRIDE
    zero = tg.tc_gemm_batched_desc(d, 0, 256, 256, 256)
    assert tg.tc_gemm_batched_validate(zero) == tg.TC_ERR_DIM


# ---------------------------------------------------------------- dispatcher

def plan(M, N, K, ab, c, ta=False, tb=False, A=1 << 20, B=1 << 40, C=1 << 41, **kw):
    return tg.tc_gemm_plan(tg.make_desc(M, N, K, ab, c, transpose_a=ta, transpose_b=tb, **kw),
                           A=A, B=B, C=C, num_sms=152)


def test_plan_fp32_goes_to_ffma():
    assert plan(256, 256, 256, "f32", "f32") == "ffma_f32_nn_16x32_panel"
    assert plan(4096, 4096, 4096, "f32", "f32", tb=True) == "ffma_f32_nt_128x128"


def test_plan_tensor_core_shapes():
    p = plan(4096, 4096, 4096, "bf16", "bf16")
    assert p.startswith("tcgen05_nn_bf16_bf16_256x256_pair") and "split" not in p and "pack" not in p
    assert plan(4096, 4096, 8192, "bf16", "f32", ta=True).startswith("tcgen05_tn_bf16_f32")
    assert plan(4096, 4096, 8192, "bf16", "f32", tb=True).startswith("tcgen05_nt_bf16_f32")


def test_plan_short_k_single_wave_takes_one_cta_tiles():
    """Under 16 K blocks on one wave of tiles: 128 x 64 one-CTA tiles when
    they fit in one wave, else one-CTA tiles of the modelled width; a long K
    loop keeps the CTA pair."""
    assert plan(256, 256, 256, "f16", "f16") == "tcgen05_nn_f16_f16_128x64"
    assert plan(512, 512, 512, "bf16", "bf16") == "tcgen05_nn_bf16_bf16_128x64"
    assert plan(2048, 2048, 512, "bf16", "bf16") == "tcgen05_nn_bf16_bf16_128x256"
    assert plan(2048, 2048, 2048, "f16", "f16") == "tcgen05_nn_f16_f16_256x256_pair"
    assert plan_forced("cg=2", 2048, 2048, 512, "bf16", "bf16") == "tcgen05_nn_bf16_bf16_256x256_pair"


def test_plan_split_k_for_tall_k():
    # the slices of a tile form one cluster (at most 16 CTAs) and are reduced
    # on chip; 64-wide tiles give 8 tiles x 16 slices = 128 CTAs, each with
    # fewer operand bytes to load than 4 128-wide tiles x 16 slices
    p = plan(256, 256, 16384, "bf16", "f32", ta=True)
    assert p == "tcgen05_tn_bf16_f32_128x64_csplit_s16"
    # without the cluster reduction: 128-wide tiles, as many slices as fill the SMs
    q = plan_forced("csplit=0", 256, 256, 16384, "bf16", "f32", ta=True)
    assert "_splitk" in q and q.startswith("tcgen05_tn_bf16_f32_128x128")
    s = int(q.rsplit("_s", 1)[1])
    assert 2 <= s <= 152 // 4
    # a forced split longer than a cluster goes through memory
    assert "_splitk_s20" in plan_forced("split=20", 256, 256, 16384, "bf16", "f32", ta=True)
    assert plan_forced("split=5 bn=128", 256, 256, 16384, "bf16", "f32", ta=True).endswith("128x128_csplit_s5")


def plan_forced(spec, *args, **kw):
    old = os.environ.get("TC_FORCE_VARIANT")
    os.environ["TC_FORCE_VARIANT"] = spec
    try:
        return plan(*args, **kw)
    finally:
        if old is None:
            del os.environ["TC_FORCE_VARIANT"]
        else:
            os.environ["TC_FORCE_VARIANT"] = old


def test_plan_small_split_gives_way_to_64_wide_tiles():
    # 1024^2 with a short K: 128 whole-K 128x64 tiles beat a 2-way split and
    # its reduction; a long K keeps the split, and too few 64-wide tiles
    # (the skinny shapes) keep it too
    assert plan(1024, 1024, 1024, "f16", "f16") == "tcgen05_nn_f16_f16_128x64"
    assert plan(1024, 1024, 8192, "f16", "f16") == "tcgen05_nn_f16_f16_128x128_csplit_s2"
    assert plan_forced("gemv=0", 1, 4096, 4096, "f16", "f16", tb=True).startswith("tcgen05_nt_f16_f16_128x128_csplit")


def test_plan_tail_split():
    # 256 tiles of 256x256 on 76 CTA pairs: 3 whole waves, the last 28 tiles in 2 K slices
    assert plan(4096, 4096, 4096, "bf16", "bf16") == "tcgen05_nn_bf16_bf16_256x256_pair_tail28x2"
    assert "tail" not in plan(2048, 2048, 2048, "bf16", "bf16")       # one wave


def test_plan_narrow_n():
    # a CTA pair on 256 x 192 tiles: each CTA loads 96 columns of B, so the
    # 64 tile rows read B from L2 half as often as one-CTA 128 x 192 tiles
    assert plan(8192, 384, 4096, "f16", "f16") == "tcgen05_nn_f16_f16_256x192_pair"
    assert plan_forced("cg=1", 8192, 384, 4096, "f16", "f16") == "tcgen05_nn_f16_f16_128x192"


def test_plan_repacks_unaligned_operands():
    assert plan(100, 64, 33, "f16", "f16").endswith("_packA")          # lda = 33 elements
    assert plan(100, 63, 64, "f16", "f16").endswith("_packB")          # ldb = 63
    assert "pack" not in plan(100, 64, 64, "f16", "f16")
    assert plan(100, 64, 64, "f16", "f16", A=(1 << 20) + 2).endswith("_packA")   # misaligned base


# ---------------------------------------------------------- fused epilogue

def test_epilogue_validation():
    d = desc(M=64, N=48, K=32)
    assert tg.tc_gemm_epilogue_validate(d, bias=1 << 30, activation="gelu_tanh") == tg.TC_OK
    assert tg.tc_gemm_epilogue_validate(d, bias=None, activation=None) == tg.TC_OK
    assert tg.tc_gemm_epilogue_validate(d, activation=7) == tg.TC_ERR_EPILOGUE
    # the exact-fp32 path is refused (nothing to fuse into)
    assert tg.tc_gemm_epilogue_validate(desc(a_dtype="f32", c_dtype="f32"), activation="gelu_tanh") \
        == tg.TC_ERR_EPILOGUE
    # a bias inside C's byte range (C at 3 << 40, 64 x 48 bf16)
    assert tg.tc_gemm_epilogue_validate(d, bias=(3 << 40) + 64, activation="none") == tg.TC_ERR_OVERLAP
    assert tg.tc_gemm_epilogue_validate(d, bias=(3 << 40) - 96, activation="none") == tg.TC_OK
    # the GEMM's own checks come first
    assert tg.tc_gemm_epilogue_validate(desc(M=0), activation="gelu_tanh") == tg.TC_ERR_DIM
    lib = tg.library()
    assert lib.tc_gemm_epilogue_validate(ctypes.byref(d), None, 1 << 20, 2 << 40, 3 << 40) == tg.TC_ERR_NULL


def test_plan_skinny_products():
    """At most 16 rows on one side of an NT product: the skinny-product
    kernel (its form and K split are chosen at launch); other layouts stay
    on the tensor-core kernel; fp32 on the exact path."""
    assert plan(4, 11008, 4096, "f16", "f16", tb=True) == "gemv_nt_f16_f16_x4"
    assert plan(1, 4096, 4096, "f16", "f16", tb=True) == "gemv_nt_f16_f16_x1"
    assert plan(4096, 3, 4096, "bf16", "f32", tb=True) == "gemv_nt_bf16_f32_x3_swap"
    assert plan(16, 64, 100000, "bf16", "bf16", tb=True) == "gemv_nt_bf16_bf16_x16"
    assert plan(17, 4096, 4096, "f16", "f16", tb=True).startswith("tcgen05_nt_f16_f16_")
    assert plan_forced("gemv=0", 4, 4096, 4096, "f16", "f16", tb=True).startswith("tcgen05_nt_f16_f16_128x128_csplit")
    assert plan(1, 32000, 4096, "bf16", "bf16").startswith("tcgen05_nn_bf16_bf16_128x")
    assert plan(4096, 3, 4096, "bf16", "f32").startswith("tcgen05_nn_bf16_f32_128x")
    assert plan(4, 256, 256, "f32", "f32").startswith("ffma_")


def test_q8_weight_validation():
    """The int8-weight product's own checks, host-only."""
    def q8(**kw):
        base = dict(M=4, N=32, K=64, a="f16", c="f16", b="i8", ta=False, tb=True)
        base.update(kw)
        return tg.make_desc(base["M"], base["N"], base["K"], base["a"], base["c"], b_dtype=base["b"],
                            transpose_a=base["ta"], transpose_b=base["tb"])
    v = tg.tc_gemm_q8_weight_validate
    assert v(q8()) == tg.TC_OK
    assert v(q8(a="bf16", c="f32")) == tg.TC_OK
    assert v(q8(tb=False)) == tg.TC_ERR_LAYOUT
    assert v(q8(ta=True)) == tg.TC_ERR_LAYOUT
    assert v(q8(b="f16")) == tg.TC_ERR_DTYPE
    assert v(q8(a="f32", c="f32")) == tg.TC_ERR_DTYPE
    assert v(q8(a="f16", c="bf16")) == tg.TC_ERR_DTYPE
    assert v(q8(M=0)) == tg.TC_ERR_DIM
    assert v(q8(), scale=0) == tg.TC_ERR_NULL
    # W's byte range is counted in int8 elements: C right after W's 32 x 64 bytes is fine
    assert v(q8(), W=1 << 30, C=(1 << 30) + 32 * 64) == tg.TC_OK
    assert v(q8(), W=1 << 30, C=(1 << 30) + 32 * 64 - 1) == tg.TC_ERR_OVERLAP
    # the scale must not overlap C (4 x 32 f16 at 3 << 40)
    assert v(q8(), scale=(3 << 40) + 16) == tg.TC_ERR_OVERLAP


def test_prepared_call_checks_its_arguments_once_up_front():
    """PreparedGemm runs the same argument checks as the per-call wrappers,
    when it is built: host tensors and short buffers are refused before any
    context or stream is touched."""
    d = tg.make_desc(64, 64, 64, "bf16", "bf16")
    host = torch.zeros(64 * 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        tg.PreparedGemm(None, d, host, host, host, None)
