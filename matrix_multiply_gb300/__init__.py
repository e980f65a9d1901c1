"""Python binding of tcgemm, the GB300 (sm_103a) GEMM library.

C = alpha * op(A) @ op(B) + beta * C, row-major, NN/TN/NT/TT, leading
dimensions, f16/bf16 (tcgen05 tensor cores) or f32 (exact FFMA) inputs with
fp32 accumulation -- the operation of the tensorcore gemm.md page, section
"Surface".

This module only marshals arguments: every step of the computation runs in
the CUDA kernels of ``_lib/libtcgemm.so``.  The functions keep the C names
(``tc_gemm``, ``tc_gemm_async``, ``tc_gemm_batched``, ...) and take either raw
device addresses or torch tensors (PyTorch provides device memory and
streams only).  Where a tensor is given, its capacity is checked in
elements before the call (the tessl architecture.md "nn Boundary" rule: a
view of too few elements is refused, nothing is launched).  ``GroupedGemm``
and ``PreparedGemm`` run those checks once for a group or a single product
that is issued many times; each ``enqueue()`` is then one C call.

There is no fallback: if the library is missing, importing this package
raises.  Build it with ``python -c "import __graft_entry__ as g; g.build()"``.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libtcgemm.so")

# ------------------------------------------------------------------ enums

TC_F16, TC_BF16, TC_F32, TC_I8, TC_I32 = 1, 2, 3, 4, 5
STATUS = {
    0: "TC_OK", 1: "TC_ERR_NULL", 2: "TC_ERR_DIM", 3: "TC_ERR_LD", 4: "TC_ERR_DTYPE",
    5: "TC_ERR_SCALAR", 6: "TC_ERR_OVERLAP", 7: "TC_ERR_OVERFLOW", 8: "TC_ERR_ALIGN_UNSUPPORTED",
    9: "TC_ERR_CUDA", 10: "TC_ERR_DEVICE_TIMEOUT", 11: "TC_ERR_STRIDE", 12: "TC_ERR_VARIANT",
    13: "TC_ERR_SCRATCH", 14: "TC_ERR_EPILOGUE", 15: "TC_ERR_LAYOUT",
}
for _code, _name in STATUS.items():
    globals()[_name] = _code


class tc_gemm_desc(ctypes.Structure):
    _fields_ = [
        ("M", ctypes.c_int32), ("N", ctypes.c_int32), ("K", ctypes.c_int32),
        ("a_dtype", ctypes.c_int), ("b_dtype", ctypes.c_int), ("c_dtype", ctypes.c_int),
        ("accum_dtype", ctypes.c_int),
        ("transpose_a", ctypes.c_bool), ("transpose_b", ctypes.c_bool),
        ("alpha", ctypes.c_float), ("beta", ctypes.c_float),
        ("lda", ctypes.c_int32), ("ldb", ctypes.c_int32), ("ldc", ctypes.c_int32),
    ]


TC_ACT_NONE, TC_ACT_GELU_TANH = 0, 1
_ACTIVATIONS = {None: TC_ACT_NONE, "none": TC_ACT_NONE, "gelu_tanh": TC_ACT_GELU_TANH}


class tc_epilogue(ctypes.Structure):
    """Fused epilogue: bias (device pointer to N values of C's dtype, or
    None) and activation (TC_ACT_*)."""
    _fields_ = [("bias", ctypes.c_void_p), ("activation", ctypes.c_int)]


class tc_gemm_batched_desc(ctypes.Structure):
    _fields_ = [("base", tc_gemm_desc), ("batch", ctypes.c_int32),
                ("stride_a", ctypes.c_int64), ("stride_b", ctypes.c_int64),
                ("stride_c", ctypes.c_int64)]


class TcError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({_lib.tc_status_string(status).decode()})")


# ------------------------------------------------------------------ loading

def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"tcgemm CUDA library not built ({LIB_PATH} missing); run "
            "python -c \"import __graft_entry__ as g; g.build()\"")
    lib = ctypes.CDLL(LIB_PATH)
    vp, st = ctypes.c_void_p, ctypes.c_int
    D = ctypes.POINTER(tc_gemm_desc)
    BD = ctypes.POINTER(tc_gemm_batched_desc)
    E = ctypes.POINTER(tc_epilogue)
    sig = {
        "tc_ctx_create": (st, [ctypes.POINTER(vp), ctypes.c_int]),
        "tc_ctx_destroy": (None, [vp]),
        "tc_stream_create": (st, [vp, ctypes.POINTER(vp)]),
        "tc_stream_wrap": (st, [vp, vp, ctypes.POINTER(vp)]),
        "tc_stream_sync": (st, [vp]),
        "tc_stream_handle": (vp, [vp]),
        "tc_stream_destroy": (None, [vp]),
        "tc_gemm": (st, [vp, D, vp, vp, vp]),
        "tc_gemm_async": (st, [vp, D, vp, vp, vp, vp]),
        "tc_gemm_batched": (st, [vp, BD, vp, vp, vp]),
        "tc_gemm_batched_async": (st, [vp, BD, vp, vp, vp, vp]),
        "tc_gemm_grouped_async": (st, [vp, ctypes.c_int, D, ctypes.POINTER(vp), ctypes.POINTER(vp),
                                       ctypes.POINTER(vp), vp]),
        "tc_gemm_epilogue": (st, [vp, D, E, vp, vp, vp]),
        "tc_gemm_epilogue_async": (st, [vp, D, E, vp, vp, vp, vp]),
        "tc_gemm_epilogue_validate": (st, [D, E, vp, vp, vp]),
        "tc_gemm_f32_relaxed": (st, [vp, D, E, vp, vp, vp]),
        "tc_gemm_i8_dequant": (st, [vp, D, vp, vp, vp, vp]),
        "tc_gemm_i8_dequant_async": (st, [vp, D, vp, vp, vp, vp, vp]),
        "tc_gemm_q8_weight": (st, [vp, D, vp, vp, vp, vp]),
        "tc_gemm_q8_weight_async": (st, [vp, D, vp, vp, vp, vp, vp]),
        "tc_gemm_q8_weight_validate": (st, [D, vp, vp, vp, vp]),
        "tc_gemm_f32_relaxed_async": (st, [vp, D, E, vp, vp, vp, vp]),
        "tc_gemm_host": (st, [vp, D, vp, vp, vp]),
        "tc_gemm_splitk_noalloc": (st, [D, vp, vp, vp, ctypes.c_int, vp]),
        "tc_gemm_validate": (st, [D, vp, vp, vp]),
        "tc_gemm_batched_validate": (st, [BD, vp, vp, vp]),
        "tc_gemm_plan": (st, [D, vp, vp, vp, ctypes.c_int, ctypes.c_char_p, ctypes.c_size_t]),
        "tc_last_kernel": (ctypes.c_char_p, [vp]),
        "tc_launch_count": (ctypes.c_uint64, [vp]),
        "tc_status_string": (ctypes.c_char_p, [st]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()
EXPORTED = (
    "tc_ctx_create", "tc_ctx_destroy", "tc_stream_create", "tc_stream_wrap", "tc_stream_sync",
    "tc_stream_handle", "tc_stream_destroy", "tc_gemm", "tc_gemm_async", "tc_gemm_batched",
    "tc_gemm_batched_async", "tc_gemm_grouped_async", "tc_gemm_host", "tc_gemm_splitk_noalloc",
    "tc_gemm_validate",
    "tc_gemm_batched_validate", "tc_gemm_plan", "tc_last_kernel", "tc_launch_count",
    "tc_status_string", "tc_gemm_epilogue", "tc_gemm_epilogue_async", "tc_gemm_epilogue_validate",
    "tc_gemm_f32_relaxed", "tc_gemm_f32_relaxed_async", "tc_gemm_i8_dequant", "tc_gemm_i8_dequant_async",
    "tc_gemm_q8_weight", "tc_gemm_q8_weight_async", "tc_gemm_q8_weight_validate",
)


def library():
    """The loaded ctypes library (for tests that call the ABI directly)."""
    return _lib


def _check(status: int, what: str):
    if status != 0:
        raise TcError(status, what)


# ------------------------------------------------------------------ helpers

_DT_NAMES = {"f16": TC_F16, "bf16": TC_BF16, "f32": TC_F32, "i8": TC_I8}


def _torch_dtype_code(t) -> int:
    import torch
    return {torch.float16: TC_F16, torch.bfloat16: TC_BF16, torch.float32: TC_F32}[t.dtype]


def _addr(x) -> int:
    """A device address from a torch tensor or an int."""
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return x.data_ptr()


def make_desc(M, N, K, a_dtype, c_dtype=None, *, transpose_a=False, transpose_b=False,
              alpha=1.0, beta=0.0, lda=0, ldb=0, ldc=0, b_dtype=None) -> tc_gemm_desc:
    """A descriptor; B has A's type unless ``b_dtype`` is given (the
    int8-weight product: a_dtype "f16"/"bf16", b_dtype "i8")."""
    a = _DT_NAMES.get(a_dtype, a_dtype)
    b = _DT_NAMES.get(b_dtype, b_dtype) if b_dtype is not None else a
    c = _DT_NAMES.get(c_dtype, c_dtype) if c_dtype is not None else a
    accum = TC_I32 if a == TC_I8 else TC_F32       # int8 x int8 accumulates in int32
    return tc_gemm_desc(M, N, K, a, b, c, accum, bool(transpose_a), bool(transpose_b),
                        float(alpha), float(beta), lda, ldb, ldc)


def _require(t, n_elems: int, what: str):
    """Capacity check in elements (tessl architecture.md, 'nn Boundary')."""
    if t is None or isinstance(t, int):
        return
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    avail = t.untyped_storage().nbytes() // t.element_size() - t.storage_offset()
    if n_elems > avail:
        raise ValueError(f"{what} holds {avail} elements, the descriptor needs {n_elems}")


def _extent(rows, cols, ld):
    return (rows - 1) * ld + cols


def _check_capacity(d: tc_gemm_desc, A, B, C, batch=1, sa=0, sb=0, sc=0):
    lda = d.lda or (d.M if d.transpose_a else d.K)
    ldb = d.ldb or (d.K if d.transpose_b else d.N)
    ldc = d.ldc or d.N
    ar, ac = (d.K, d.M) if d.transpose_a else (d.M, d.K)
    br, bc = (d.N, d.K) if d.transpose_b else (d.K, d.N)
    if min(d.M, d.N, d.K, batch) < 1 or lda < ac or ldb < bc or ldc < d.N:
        return   # the library reports the precise error
    _require(A, (batch - 1) * sa + _extent(ar, ac, lda), "A")
    _require(B, (batch - 1) * sb + _extent(br, bc, ldb), "B")
    _require(C, (batch - 1) * sc + _extent(d.M, d.N, ldc), "C")


# ------------------------------------------------------------------ objects

class Context:
    """A tc_ctx on one CUDA device."""

    def __init__(self, device: int = 0):
        p = ctypes.c_void_p()
        _check(_lib.tc_ctx_create(ctypes.byref(p), device), "tc_ctx_create")
        self.ptr = p.value
        self.device = device

    def close(self):
        if self.ptr:
            _lib.tc_ctx_destroy(self.ptr)
            self.ptr = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def last_kernel(self) -> str:
        return _lib.tc_last_kernel(self.ptr).decode()

    @property
    def launch_count(self) -> int:
        return int(_lib.tc_launch_count(self.ptr))


class Stream:
    """A tc_stream: owned (created by the library) or wrapping a torch stream."""

    def __init__(self, ctx: Context, torch_stream=None):
        p = ctypes.c_void_p()
        if torch_stream is None:
            _check(_lib.tc_stream_create(ctx.ptr, ctypes.byref(p)), "tc_stream_create")
        else:
            _check(_lib.tc_stream_wrap(ctx.ptr, ctypes.c_void_p(torch_stream.cuda_stream),
                                       ctypes.byref(p)), "tc_stream_wrap")
        self.ptr = p.value
        self.ctx = ctx

    @property
    def handle(self) -> int:
        return _lib.tc_stream_handle(self.ptr) or 0

    def sync(self):
        _check(_lib.tc_stream_sync(self.ptr), "tc_stream_sync")

    def close(self):
        if self.ptr:
            _lib.tc_stream_destroy(self.ptr)
            self.ptr = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ------------------------------------------------------------------ C names

def tc_gemm(ctx: Context, d: tc_gemm_desc, A, B, C):
    _check_capacity(d, A, B, C)
    _check(_lib.tc_gemm(ctx.ptr, ctypes.byref(d), _addr(A), _addr(B), _addr(C)), "tc_gemm")


def tc_gemm_async(ctx: Context, d: tc_gemm_desc, A, B, C, stream: Stream):
    _check_capacity(d, A, B, C)
    _check(_lib.tc_gemm_async(ctx.ptr, ctypes.byref(d), _addr(A), _addr(B), _addr(C), stream.ptr),
           "tc_gemm_async")


def tc_gemm_batched(ctx: Context, bd: tc_gemm_batched_desc, A, B, C):
    _check_capacity(bd.base, A, B, C, bd.batch, bd.stride_a, bd.stride_b, bd.stride_c)
    _check(_lib.tc_gemm_batched(ctx.ptr, ctypes.byref(bd), _addr(A), _addr(B), _addr(C)),
           "tc_gemm_batched")


def tc_gemm_batched_async(ctx: Context, bd: tc_gemm_batched_desc, A, B, C, stream: Stream):
    _check_capacity(bd.base, A, B, C, bd.batch, bd.stride_a, bd.stride_b, bd.stride_c)
    _check(_lib.tc_gemm_batched_async(ctx.ptr, ctypes.byref(bd), _addr(A), _addr(B), _addr(C),
                                      stream.ptr), "tc_gemm_batched_async")


class GroupedGemm:
    """The arguments of tc_gemm_grouped_async marshalled once: descriptors
    and operand addresses in C arrays, capacities checked here.  enqueue()
    then costs one C call, so that a group issued many times with the same
    operands does not pay the per-problem Python work each time.  The
    tensors stay referenced (alive) as long as this object."""

    def __init__(self, descs, As, Bs, Cs):
        n = len(descs)
        if not (len(As) == len(Bs) == len(Cs) == n):
            raise ValueError("descs, As, Bs and Cs must have the same length")
        for d, a, b, c in zip(descs, As, Bs, Cs):
            _check_capacity(d, a, b, c)
        self.n = n
        self._keep = (list(As), list(Bs), list(Cs))
        self._descs = (tc_gemm_desc * n)(*descs)
        self._A = (ctypes.c_void_p * n)(*[_addr(x) for x in As])
        self._B = (ctypes.c_void_p * n)(*[_addr(x) for x in Bs])
        self._C = (ctypes.c_void_p * n)(*[_addr(x) for x in Cs])

    def enqueue(self, ctx: Context, stream: Stream):
        _check(_lib.tc_gemm_grouped_async(ctx.ptr, self.n, self._descs, self._A, self._B, self._C, stream.ptr),
               "tc_gemm_grouped_async")


def tc_gemm_grouped_async(ctx: Context, descs, As, Bs, Cs, stream: Stream):
    GroupedGemm(descs, As, Bs, Cs).enqueue(ctx, stream)


class PreparedGemm:
    """One asynchronous product with its arguments checked and marshalled
    once: tc_gemm_async; with ``bias``/``activation`` tc_gemm_epilogue_async;
    with ``relaxed`` tc_gemm_f32_relaxed_async; with ``col_scale``
    tc_gemm_i8_dequant_async; with ``q8_scale`` tc_gemm_q8_weight_async.
    enqueue() is then one C call -- the library still plans the product and
    launches its kernels every time -- for a caller that issues the same
    product on the same buffers many times (the Python checks otherwise
    cost about as much host time per call as the library itself).  The
    tensors stay referenced as long as this object."""

    def __init__(self, ctx: Context, d: tc_gemm_desc, A, B, C, stream: Stream, *, bias=None, activation=None,
                 relaxed: bool = False, col_scale=None, q8_scale=None):
        _check_capacity(d, A, B, C)
        vp = ctypes.c_void_p
        head = (vp(ctx.ptr), ctypes.byref(d))
        abc = (vp(_addr(A)), vp(_addr(B)), vp(_addr(C)), vp(stream.ptr))
        self._e = None
        if q8_scale is not None:
            _require(q8_scale, d.N, "scale")
            self._fn, self._name = _lib.tc_gemm_q8_weight_async, "tc_gemm_q8_weight_async"
            self._args = head + (vp(_addr(q8_scale)),) + abc
        elif col_scale is not None:
            _require(col_scale, d.N, "col_scale")
            self._fn, self._name = _lib.tc_gemm_i8_dequant_async, "tc_gemm_i8_dequant_async"
            self._args = head + (vp(_addr(col_scale)),) + abc
        elif relaxed or bias is not None or activation is not None:
            _check_bias(d, bias)
            self._e = make_epilogue(bias, activation)
            self._name = "tc_gemm_f32_relaxed_async" if relaxed else "tc_gemm_epilogue_async"
            self._fn = getattr(_lib, self._name)
            self._args = head + (ctypes.byref(self._e),) + abc
        else:
            self._fn, self._name = _lib.tc_gemm_async, "tc_gemm_async"
            self._args = head + abc
        self._keep = (ctx, d, A, B, C, stream, bias, col_scale, q8_scale)

    def enqueue(self):
        _check(self._fn(*self._args), self._name)


def make_epilogue(bias=None, activation=None) -> tc_epilogue:
    """bias: a CUDA tensor of N values in C's dtype (or an address, or
    None); activation: None/"none" or "gelu_tanh" (or a TC_ACT_* code)."""
    act = _ACTIVATIONS.get(activation, activation)
    return tc_epilogue(_addr(bias) or None, int(act))


def _check_bias(d: tc_gemm_desc, bias):
    if bias is None or isinstance(bias, int):
        return
    _require(bias, d.N, "bias")
    if d.c_dtype in (TC_F16, TC_BF16, TC_F32) and _torch_dtype_code(bias) != d.c_dtype:
        raise ValueError("bias must have C's dtype")


def tc_gemm_epilogue(ctx: Context, d: tc_gemm_desc, A, B, C, bias=None, activation=None):
    """C = activation(alpha*op(A)@op(B) + beta*C + bias), synchronously."""
    _check_capacity(d, A, B, C)
    _check_bias(d, bias)
    e = make_epilogue(bias, activation)
    _check(_lib.tc_gemm_epilogue(ctx.ptr, ctypes.byref(d), ctypes.byref(e), _addr(A), _addr(B), _addr(C)),
           "tc_gemm_epilogue")


def tc_gemm_epilogue_async(ctx: Context, d: tc_gemm_desc, A, B, C, stream: Stream, bias=None, activation=None):
    _check_capacity(d, A, B, C)
    _check_bias(d, bias)
    e = make_epilogue(bias, activation)
    _check(_lib.tc_gemm_epilogue_async(ctx.ptr, ctypes.byref(d), ctypes.byref(e), _addr(A), _addr(B), _addr(C),
                                       stream.ptr), "tc_gemm_epilogue_async")


def tc_gemm_epilogue_validate(d: tc_gemm_desc, bias=None, activation=None, A=1 << 20, B=2 << 40,
                              C=3 << 40) -> int:
    """Host-only validation status of a fused-epilogue call."""
    e = make_epilogue(bias, activation)
    return int(_lib.tc_gemm_epilogue_validate(ctypes.byref(d), ctypes.byref(e), _addr(A), _addr(B), _addr(C)))


def tc_gemm_f32_relaxed(ctx: Context, d: tc_gemm_desc, A, B, C, bias=None, activation=None):
    """fp32 GEMM on the bf16 tensor cores through a two-part bf16 split of
    each operand (see include/tcgemm.h), synchronously; optional fused
    epilogue."""
    _check_capacity(d, A, B, C)
    _check_bias(d, bias)
    e = make_epilogue(bias, activation)
    _check(_lib.tc_gemm_f32_relaxed(ctx.ptr, ctypes.byref(d), ctypes.byref(e), _addr(A), _addr(B), _addr(C)),
           "tc_gemm_f32_relaxed")


def tc_gemm_f32_relaxed_async(ctx: Context, d: tc_gemm_desc, A, B, C, stream: Stream, bias=None, activation=None):
    _check_capacity(d, A, B, C)
    _check_bias(d, bias)
    e = make_epilogue(bias, activation)
    _check(_lib.tc_gemm_f32_relaxed_async(ctx.ptr, ctypes.byref(d), ctypes.byref(e), _addr(A), _addr(B), _addr(C),
                                          stream.ptr), "tc_gemm_f32_relaxed_async")


def tc_gemm_i8_dequant(ctx: Context, d: tc_gemm_desc, A, B, C, col_scale):
    """int8 x int8 accumulated exactly, then C = alpha * acc * col_scale[n] +
    beta * C (C fp32; col_scale a CUDA tensor of N floats), synchronously."""
    _check_capacity(d, A, B, C)
    _require(col_scale, d.N, "col_scale")
    _check(_lib.tc_gemm_i8_dequant(ctx.ptr, ctypes.byref(d), _addr(col_scale), _addr(A), _addr(B), _addr(C)),
           "tc_gemm_i8_dequant")


def tc_gemm_i8_dequant_async(ctx: Context, d: tc_gemm_desc, A, B, C, col_scale, stream: Stream):
    _check_capacity(d, A, B, C)
    _require(col_scale, d.N, "col_scale")
    _check(_lib.tc_gemm_i8_dequant_async(ctx.ptr, ctypes.byref(d), _addr(col_scale), _addr(A), _addr(B), _addr(C),
                                         stream.ptr), "tc_gemm_i8_dequant_async")


def tc_gemm_q8_weight(ctx: Context, d: tc_gemm_desc, X, W, C, scale):
    """Out = alpha * (X @ W^T) * scale[n] + beta * Out, X [M,K] f16/bf16,
    W [N,K] int8, scale N floats (CUDA tensors), synchronously."""
    _check_capacity(d, X, W, C)
    _require(scale, d.N, "scale")
    _check(_lib.tc_gemm_q8_weight(ctx.ptr, ctypes.byref(d), _addr(scale), _addr(X), _addr(W), _addr(C)),
           "tc_gemm_q8_weight")


def tc_gemm_q8_weight_async(ctx: Context, d: tc_gemm_desc, X, W, C, scale, stream: Stream):
    _check_capacity(d, X, W, C)
    _require(scale, d.N, "scale")
    _check(_lib.tc_gemm_q8_weight_async(ctx.ptr, ctypes.byref(d), _addr(scale), _addr(X), _addr(W), _addr(C),
                                        stream.ptr), "tc_gemm_q8_weight_async")


def tc_gemm_q8_weight_validate(d: tc_gemm_desc, scale=4 << 40, X=1 << 20, W=2 << 40, C=3 << 40) -> int:
    """Host-only validation status of an int8-weight product."""
    return int(_lib.tc_gemm_q8_weight_validate(ctypes.byref(d), _addr(scale), _addr(X), _addr(W), _addr(C)))


def tc_gemm_host(ctx: Context, d: tc_gemm_desc, A_host, B_host, C_host):
    """Host operands (CPU tensors, ideally pinned): copy in, run, copy out."""
    for t in (A_host, B_host, C_host):
        if not isinstance(t, int) and t.is_cuda:
            raise ValueError("tc_gemm_host takes host tensors")
    _check(_lib.tc_gemm_host(ctx.ptr, ctypes.byref(d), _addr(A_host), _addr(B_host), _addr(C_host)),
           "tc_gemm_host")


def tc_gemm_splitk_noalloc(d: tc_gemm_desc, A, B, C, split: int = 0, torch_stream=None):
    """Split-K GEMM whose scratch is the library's static device buffer:
    nothing is allocated (for callers that must not allocate device memory;
    see include/tcgemm.h).  Asynchronous on ``torch_stream`` (default: the
    legacy default stream); calls that overlap on the GPU race."""
    _check_capacity(d, A, B, C)
    handle = torch_stream.cuda_stream if torch_stream is not None else 0
    _check(_lib.tc_gemm_splitk_noalloc(ctypes.byref(d), _addr(A), _addr(B), _addr(C), int(split),
                                       ctypes.c_void_p(handle)), "tc_gemm_splitk_noalloc")


def tc_gemm_validate(d: tc_gemm_desc, A=1 << 20, B=2 << 40, C=3 << 40) -> int:
    """Host-only validation status (no device needed)."""
    return int(_lib.tc_gemm_validate(ctypes.byref(d) if d is not None else None,
                                     _addr(A), _addr(B), _addr(C)))


def tc_gemm_batched_validate(bd: tc_gemm_batched_desc, A=1 << 20, B=2 << 40, C=3 << 40) -> int:
    return int(_lib.tc_gemm_batched_validate(ctypes.byref(bd), _addr(A), _addr(B), _addr(C)))


def tc_gemm_plan(d: tc_gemm_desc, A=1 << 20, B=2 << 40, C=3 << 40, num_sms: int = 152) -> str:
    """The variant the dispatcher picks (host-only)."""
    buf = ctypes.create_string_buffer(256)
    _check(_lib.tc_gemm_plan(ctypes.byref(d), _addr(A), _addr(B), _addr(C), num_sms, buf, 256),
           "tc_gemm_plan")
    return buf.value.decode()


def tc_last_kernel(ctx: Context) -> str:
    return ctx.last_kernel


def tc_launch_count(ctx: Context) -> int:
    return ctx.launch_count


def tc_status_string(status: int) -> str:
    return _lib.tc_status_string(status).decode()


# ------------------------------------------------------------------ tensor API

@dataclass
class _Shapes:
    M: int
    N: int
    K: int


def gemm(ctx: Context, A, B, C, *, transpose_a=False, transpose_b=False, alpha=1.0, beta=0.0,
         stream: Stream | None = None):
    """C = alpha*op(A)@op(B) + beta*C on torch CUDA tensors (2-D, row-major,
    unit column stride; row strides become leading dimensions)."""
    for name, t in (("A", A), ("B", B), ("C", C)):
        if t.dim() != 2 or t.stride(1) != 1:
            raise ValueError(f"{name} must be 2-D with unit column stride")
    M = A.shape[1] if transpose_a else A.shape[0]
    K = A.shape[0] if transpose_a else A.shape[1]
    N = B.shape[0] if transpose_b else B.shape[1]
    d = tc_gemm_desc(M, N, K, _torch_dtype_code(A), _torch_dtype_code(B), _torch_dtype_code(C), TC_F32,
                     bool(transpose_a), bool(transpose_b), float(alpha), float(beta),
                     A.stride(0), B.stride(0), C.stride(0))
    if stream is None:
        tc_gemm(ctx, d, A, B, C)
    else:
        tc_gemm_async(ctx, d, A, B, C, stream)
    return C
