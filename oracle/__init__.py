"""CPU oracle for C = alpha*op(A)@op(B) + beta*C -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product (``matrix_multiply_gb300``) never
does, and the two share no code: this wrapper loads ``oracle.c`` (compiled
here with gcc) and hands it the stored bits of the operands.

Definition followed (see the header of ``oracle.c`` for the citations):
tensorcore gemm.md "Surface" (row-major BLAS layout, ld = 0 means contiguous),
the phobos matmul page ("matmul", "matmul_t", the "sgemm" alpha/beta
epilogue).  Results are fp64 ``R`` plus the absolute-product sum ``T``.

The fused epilogue (tessl architecture.md, "Fused Epilogue": C =
activation(alpha * A@B + beta * C_prev + bias), bias per column, the
GeluTanh activation) is applied here in fp64 on top of the same R, by
``gemm_epilogue`` / ``gemm_epilogue_points``.

The int8-weight product (Foundry metal.md, "Custom Compute Kernels":
fm_sgemm_q8, Out = X @ (W_q8 * scale[n])^T) is the same k-sum over mixed
operand types, scaled per output column: ``gemm_q8_weight`` /
``gemm_q8_weight_points``.

Every function here is pinned by ``tests/test_oracle.py`` against things
other than itself: exact rational brute force, numpy's float64 matmul on
operands decoded by PyTorch, the worked 2x2 input of the Foundry metal.md
"Quick Start", closed forms (identity, permutation, rank one, alpha/beta),
an exhaustive check of the half-precision decoders, and, for the epilogue,
PyTorch's tanh-approximated GELU in float64 and the GELU identities.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")

CODES = {"f16": 1, "bf16": 2, "f32": 3, "i8": 4}


class _Problem(ctypes.Structure):
    _fields_ = [
        ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
        ("a_dtype", ctypes.c_int32), ("b_dtype", ctypes.c_int32), ("c_dtype", ctypes.c_int32),
        ("transpose_a", ctypes.c_int32), ("transpose_b", ctypes.c_int32),
        ("alpha", ctypes.c_double), ("beta", ctypes.c_double),
        ("lda", ctypes.c_int64), ("ldb", ctypes.c_int64), ("ldc", ctypes.c_int64),
        ("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("C", ctypes.c_void_p),
    ]


_lock = threading.Lock()
_lib = None


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile ``src`` into a shared library at ``out`` with gcc."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC",
           *extra_flags, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _bind(lib):
    P = ctypes.POINTER(_Problem)
    i64p = ctypes.POINTER(ctypes.c_int64)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.oracle_gemm_rows.argtypes = [P, ctypes.c_int64, ctypes.c_int64, dp, dp]
    lib.oracle_gemm_rows.restype = ctypes.c_int
    lib.oracle_gemm_points.argtypes = [P, ctypes.c_int64, i64p, i64p, dp, dp]
    lib.oracle_gemm_points.restype = ctypes.c_int
    lib.oracle_decode_array.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, dp]
    lib.oracle_decode_array.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    return lib


def load_library(path: str | None = None):
    """Load the oracle library; build it first if it is missing or stale.
    ``path`` loads another build of it (the mutation tests use this)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if (not os.path.exists(_LIB_PATH)
                    or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
                build()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    assert t.device.type == "cpu"
    return t.data_ptr()


def _dtype_code(t: torch.Tensor) -> int:
    return {torch.float16: 1, torch.bfloat16: 2, torch.float32: 3, torch.int8: 4}[t.dtype]


def _struct(p, lda=None, ldb=None, ldc=None) -> tuple[_Problem, list]:
    """Build the C descriptor from a ``synthetic.Problem``-like object.  The
    stored tensors' row length is the leading dimension unless given."""
    A = p.A.contiguous()
    B = p.B.contiguous()
    C = p.C.contiguous() if p.C is not None else None
    s = _Problem()
    s.M, s.N, s.K = p.M, p.N, p.K
    s.a_dtype, s.b_dtype = _dtype_code(A), _dtype_code(B)
    s.c_dtype = _dtype_code(C) if C is not None else CODES[p.c_dtype]
    s.transpose_a, s.transpose_b = int(p.transpose_a), int(p.transpose_b)
    # alpha/beta reach the GPU as float32: the oracle uses the same values
    s.alpha = float(np.float32(p.alpha))
    s.beta = float(np.float32(p.beta))
    s.lda = A.shape[1] if lda is None else lda
    s.ldb = B.shape[1] if ldb is None else ldb
    s.ldc = (C.shape[1] if C is not None else 0) if ldc is None else ldc
    s.A, s.B, s.C = _ptr(A), _ptr(B), _ptr(C)
    return s, [A, B, C]


def gemm(p, row0: int = 0, row1: int | None = None, lib=None):
    """Rows [row0,row1) of R = alpha*op(A)@op(B) + beta*C_old and of
    T = sum_k |op(A)_ik op(B)_kj|, both fp64 arrays of shape (rows, N)."""
    lib = lib or load_library()
    row1 = p.M if row1 is None else row1
    s, keep = _struct(p)
    R = np.empty((row1 - row0, p.N), dtype=np.float64)
    T = np.empty((row1 - row0, p.N), dtype=np.float64)
    rc = lib.oracle_gemm_rows(ctypes.byref(s), row0, row1,
                              R.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                              T.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    del keep
    if rc != 0:
        raise ValueError(f"oracle_gemm_rows failed ({rc})")
    return R, T


def gemm_points(p, rows, cols, lib=None):
    """R and T at the listed (row, col) positions (1-D fp64 arrays)."""
    lib = lib or load_library()
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    s, keep = _struct(p)
    R = np.empty(rows.shape[0], dtype=np.float64)
    T = np.empty(rows.shape[0], dtype=np.float64)
    i64p = ctypes.POINTER(ctypes.c_int64)
    dp = ctypes.POINTER(ctypes.c_double)
    rc = lib.oracle_gemm_points(ctypes.byref(s), rows.shape[0], rows.ctypes.data_as(i64p),
                                cols.ctypes.data_as(i64p), R.ctypes.data_as(dp),
                                T.ctypes.data_as(dp))
    del keep
    if rc != 0:
        raise ValueError(f"oracle_gemm_points failed ({rc})")
    return R, T


def decode(t: torch.Tensor, lib=None) -> np.ndarray:
    """Exact fp64 values of a stored f16/bf16/f32 tensor, via the oracle's
    own decoders (not PyTorch's casts)."""
    lib = lib or load_library()
    t = t.contiguous()
    out = np.empty(t.numel(), dtype=np.float64)
    rc = lib.oracle_decode_array(_dtype_code(t), t.numel(), t.data_ptr(),
                                 out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    if rc != 0:
        raise ValueError("oracle_decode_array failed")
    return out.reshape(tuple(t.shape))


def num_threads(lib=None) -> int:
    lib = lib or load_library()
    return int(lib.oracle_num_threads())


# ------------------------------------------------------------------ epilogue
# tessl architecture.md, "Fused Epilogue": C = activation(alpha * A@B +
# beta * C_prev + bias); the bias is one value per output column (a
# row-stride-0 view, broadcast over the rows) stored in C's dtype; the
# activation is none or GeluTanh.  The page names a clamped tanh without
# printing it; the oracle uses the exact tanh (clamping only matters where
# tanh is +-1 to working precision).

SQRT_2_OVER_PI = float(np.sqrt(2.0 / np.pi))
GELU_CUBIC = 0.044715
ACTIVATIONS = ("none", "gelu_tanh")


def gelu_tanh(x):
    """GELU, tanh form: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), fp64."""
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + np.tanh(SQRT_2_OVER_PI * (x + GELU_CUBIC * x * x * x)))


def apply_activation(y, activation: str):
    if activation == "none":
        return np.asarray(y, dtype=np.float64)
    if activation == "gelu_tanh":
        return gelu_tanh(y)
    raise ValueError(activation)


def gemm_epilogue(p, bias, activation: str, row0: int = 0, row1: int | None = None, lib=None):
    """Rows [row0,row1) of activation(alpha*op(A)@op(B) + beta*C_old + bias)
    (``bias`` a stored tensor of N values, or None), with T and the
    pre-activation value: returns (R, T, Y) fp64, Y = R before activation."""
    R, T = gemm(p, row0, row1, lib=lib)
    Y = R if bias is None else R + decode(bias, lib=lib).reshape(1, -1)[:, : p.N]
    return apply_activation(Y, activation), T, Y


def gemm_epilogue_points(p, bias, activation: str, rows, cols, lib=None):
    """gemm_epilogue at the listed (row, col) positions (1-D arrays)."""
    R, T = gemm_points(p, rows, cols, lib=lib)
    cols = np.asarray(cols, dtype=np.int64)
    Y = R if bias is None else R + decode(bias, lib=lib).reshape(-1)[cols]
    return apply_activation(Y, activation), T, Y


# -------------------------------------------------------------- int8 GEMM
# tessl architecture.md, "Integer GEMM": int8 x int8 accumulated exactly
# (an integer; refused for K > 131072, where a full-range sum can leave
# int32), then per-column dequantisation.  With this library's alpha/beta:
# C = alpha * (acc[m, n] * scale[n]) + beta * C_old, in fp64.

def gemm_i8_dequant(p, scale, row0: int = 0, row1: int | None = None, lib=None):
    """Rows [row0,row1) of alpha * acc * scale[None, :] + beta * C_old for
    int8 operands, with T and the exact integer accumulation: (R, T, ACC)."""
    import copy
    q = copy.copy(p)
    q.alpha, q.beta = 1.0, 0.0
    ACC, T = gemm(q, row0, row1, lib=lib)
    sc = decode(scale, lib=lib).reshape(1, -1)[:, : p.N]
    R = float(np.float32(p.alpha)) * (ACC * sc)
    if p.beta != 0.0:
        row1 = p.M if row1 is None else row1
        R = R + float(np.float32(p.beta)) * decode(p.C, lib=lib)[row0:row1, : p.N]
    return R, T, ACC



# ------------------------------------------------- int8-weight (Q8) product
# Foundry metal.md, "Custom Compute Kernels": fm_sgemm_q8(X[M,K], W_q8[N,K],
# scales[N]) -- the activations times the transposed int8 weight, each
# weight row n dequantised by its own scale: Out[m, n] = sum_k X[m, k] *
# (W_q8[n, k] * scales[n]).  The tensorcore gemm.md "Kernel variants" table
# runs the same product as an M <= 4 GEMV with fp16 output.  With this
# library's alpha/beta: Out = alpha * (acc[m, n] * scale[n]) + beta * C_old,
# acc = sum_k X[m, k] * W[n, k] (X half precision, W int8: every product is
# exact, and so is the fp64 sum for the sizes tested).  The tolerance scale
# is that of the GEMM over the dequantised weight: T = |scale[n]| * sum_k
# |X[m, k] * W[n, k]|.

def gemm_q8_weight(p, scale, row0: int = 0, row1: int | None = None, lib=None):
    """Rows [row0,row1) of alpha * acc * scale[None, :] + beta * C_old, for
    p.A = X (f16/bf16, stored [M,K]) and p.B = W (int8, stored [N,K],
    transpose_b), with T and the product sum: (R, T, ACC)."""
    import copy
    q = copy.copy(p)
    q.alpha, q.beta = 1.0, 0.0
    ACC, T0 = gemm(q, row0, row1, lib=lib)
    sc = decode(scale, lib=lib).reshape(1, -1)[:, : p.N]
    R = float(np.float32(p.alpha)) * (ACC * sc)
    if p.beta != 0.0:
        row1 = p.M if row1 is None else row1
        R = R + float(np.float32(p.beta)) * decode(p.C, lib=lib)[row0:row1, : p.N]
    return R, T0 * np.abs(sc), ACC


def gemm_q8_weight_points(p, scale, rows, cols, lib=None):
    """gemm_q8_weight at the listed (row, col) positions (1-D arrays)."""
    import copy
    q = copy.copy(p)
    q.alpha, q.beta = 1.0, 0.0
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    ACC, T0 = gemm_points(q, rows, cols, lib=lib)
    sc = decode(scale, lib=lib).reshape(-1)[cols]
    R = float(np.float32(p.alpha)) * (ACC * sc)
    if p.beta != 0.0:
        R = R + float(np.float32(p.beta)) * decode(p.C, lib=lib)[rows, cols]
    return R, T0 * np.abs(sc), ACC
