"""The parity bar between a GEMM result and the oracle's fp64 value.

Per element, with R the oracle's fp64 result and T = sum_k |a_ik b_kj|:
  * fp32 output:            |C - R| <= 1e-4 * T
  * fp16 / bf16 output:     |C - R| <= 1e-4 * T + ulp_out(R)
  * the fp32-exact path:    |C - R| <= 1e-5 * T
The output is decoded exactly before the comparison.  rms_scaled
(||C - R|| / (||R|| + eps), tensorcore gemm.md "Numerical guarantees") is
reported beside it for information.
"""
from __future__ import annotations

import math

import numpy as np

# fraction bits and smallest subnormal spacing of each output encoding
_FRAC_BITS = {"bf16": 7, "f16": 10, "f32": 23}
_MIN_SPACING = {"bf16": 2.0 ** -133, "f16": 2.0 ** -24, "f32": 2.0 ** -149}


def ulp_out(R: np.ndarray, c_dtype: str) -> np.ndarray:
    """Spacing of the output format at |R|: 2^(floor(log2|R|) - frac_bits),
    floored at the format's subnormal spacing."""
    a = np.abs(np.asarray(R, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    u = np.exp2(e - _FRAC_BITS[c_dtype])
    u = np.where(a > 0, u, 0.0)
    return np.maximum(u, _MIN_SPACING[c_dtype])


def bound(R, T, c_dtype: str, exact_f32: bool = False) -> np.ndarray:
    if exact_f32:
        return 1e-5 * T
    b = 1e-4 * T
    if c_dtype in ("bf16", "f16"):
        b = b + ulp_out(R, c_dtype)
    return b


# Largest slope of the tanh-form GELU (near x = 1.5); an error e in its
# argument moves the output by at most GELU_LIPSCHITZ * e.
GELU_LIPSCHITZ = 1.13


def bound_epilogue(R, T, Y, bias_abs, c_dtype: str, activation: str) -> np.ndarray:
    """Bound for C = act(alpha*acc + beta*C_old + bias) against the oracle's
    R = act(Y): the GEMM's 1e-4*T plus the fp32 roundings of the bias add
    (2^-20 of |Y| + |bias|), carried through the activation's slope, plus
    the fp32 evaluation of GELU (2e-6 |Y|: the device forms x / (1 + 2^u),
    u = -2 z log2(e), with approximate ex2 and reciprocal instructions whose
    relative error stays below ~1.5e-6 for the arguments that matter, plus a
    few ulp in u) and one output ulp for f16/bf16."""
    Y = np.abs(np.asarray(Y, dtype=np.float64))
    pre = 1e-4 * T + 2.0 ** -20 * (Y + bias_abs)
    if activation == "gelu_tanh":
        b = GELU_LIPSCHITZ * pre + 2e-6 * Y + 1e-30
    else:
        b = pre
    if c_dtype in ("bf16", "f16"):
        b = b + ulp_out(R, c_dtype)
    return b


def check_epilogue(C, R, T, Y, bias_abs, c_dtype: str, activation: str, what: str = "") -> dict:
    """Assert the fused-epilogue bound per element; return error statistics."""
    C = np.asarray(C, dtype=np.float64)
    err = np.abs(C - R)
    lim = bound_epilogue(R, T, Y, bias_abs, c_dtype, activation)
    bad = ~(err <= lim)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = ", ".join(f"{tuple(int(v) for v in i)}: got {C[tuple(i)]!r} want {R[tuple(i)]!r} "
                           f"(lim={lim[tuple(i)]:.3g})" for i in idx)
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} elements out of bound; {detail}")
    return {"max_err": float(err.max()) if err.size else 0.0, "n": int(err.size)}


def check(C: np.ndarray, R: np.ndarray, T: np.ndarray, c_dtype: str,
          exact_f32: bool = False, what: str = "") -> dict:
    """Assert the per-element bound; return error statistics."""
    C = np.asarray(C, dtype=np.float64)
    err = np.abs(C - R)
    lim = bound(R, T, c_dtype, exact_f32)
    bad = ~(err <= lim)            # NaN counts as bad
    stats = {
        "max_err_over_T": float(np.max(err / np.maximum(T, 1e-300))) if err.size else 0.0,
        "rms_scaled": float(np.linalg.norm(C - R) / (np.linalg.norm(R) + 1e-30)) if err.size else 0.0,
        "n": int(err.size),
    }
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = ", ".join(
            f"{tuple(int(v) for v in i)}: got {C[tuple(i)]!r} want {R[tuple(i)]!r} "
            f"(T={T[tuple(i)]:.3g}, lim={lim[tuple(i)]:.3g})" for i in idx)
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} elements out of bound; {detail}")
    return stats


def sample_points(M: int, N: int, n: int, rng: np.random.Generator):
    """n random (row, col) positions plus the four corners and the last
    row/column tails, so ragged edge tiles are always sampled."""
    rows = list(rng.integers(0, M, n))
    cols = list(rng.integers(0, N, n))
    for r, c in ((0, 0), (0, N - 1), (M - 1, 0), (M - 1, N - 1)):
        rows.append(r)
        cols.append(c)
    for t in range(min(N, 64)):
        rows.append(M - 1)
        cols.append(N - 1 - t)
    for t in range(min(M, 64)):
        rows.append(M - 1 - t)
        cols.append(N - 1)
    return np.array(rows, dtype=np.int64), np.array(cols, dtype=np.int64)


def finite_fraction(x) -> float:
    x = np.asarray(x, dtype=np.float64)
    return float(np.isfinite(x).mean()) if x.size else 1.0


def log2_floor(x: float) -> int:
    return math.floor(math.log2(abs(x)))
