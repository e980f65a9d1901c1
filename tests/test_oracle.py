"""Pins for the CPU oracle (no GPU needed).

The oracle is checked against things other than itself:
  * exhaustive decoding of every binary16 / bfloat16 bit pattern against
    PyTorch's casts (an independent implementation of the encodings);
  * the worked 2x2 input of the Foundry metal.md "Quick Start" and its closed
    form (tests/golden/foundry_quickstart_2x2.txt);
  * exact rational arithmetic (``fractions``) on tiny shapes, every layout,
    padded leading dimensions, alpha/beta;
  * numpy's float64 matmul on operands decoded by PyTorch;
  * closed forms: identity, permutation, rank one (K = 1), alpha/beta on
    integer data, beta = 0 ignoring a NaN-filled C;
  * mutation tests: plausible mistakes planted in a copy of oracle.c (a
    swapped index, a dropped term, a wrong sign, a wrong decoder bias, a
    wrong default leading dimension, a signed T) must each fail a pin.
"""
from __future__ import annotations

import itertools
import os
import re
import subprocess
import tempfile
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synthetic

HERE = os.path.dirname(os.path.abspath(__file__))
LAYOUTS = [(False, False), (True, False), (False, True), (True, True)]


def torch_decode(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def op_a(p, Ad):
    return Ad[: p.K, : p.M].T if p.transpose_a else Ad[: p.M, : p.K]


def op_b(p, Bd):
    return Bd[: p.N, : p.K].T if p.transpose_b else Bd[: p.K, : p.N]


# ---------------------------------------------------------------- decoders

@pytest.mark.parametrize("name,tdt", [("f16", torch.float16), ("bf16", torch.bfloat16)])
def test_decoder_exhaustive(name, tdt):
    bits = torch.arange(0, 65536, dtype=torch.int32).to(torch.int16)
    t = bits.view(tdt)
    mine = oracle.decode(t)
    ref = torch_decode(t)
    nan_m, nan_r = np.isnan(mine), np.isnan(ref)
    assert (nan_m == nan_r).all()
    assert (mine[~nan_m] == ref[~nan_r]).all()
    # signed zeros and infinities keep their sign
    assert (np.signbit(mine[~nan_m]) == np.signbit(ref[~nan_r])).all()


def test_decoder_f32_widening():
    g = torch.Generator().manual_seed(5)
    t = torch.randn(10000, generator=g) * 1e30
    t[:4] = torch.tensor([0.0, -0.0, float("inf"), 1e-45])
    assert (oracle.decode(t) == t.to(torch.float64).numpy()).all()


# ---------------------------------------------------------- worked example

def _read_golden(name):
    vals = {}
    with open(os.path.join(HERE, "golden", name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            vals[k.strip()] = [float(x) for x in v.split()]
    return vals


@pytest.mark.parametrize("dt", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_worked_example_2x2(dt, ta, tb):
    g = _read_golden("foundry_quickstart_2x2.txt")
    M, N, K = (int(v) for v in g["M N K"])
    A = torch.tensor(g["A"]).reshape(M, K)
    B = torch.tensor(g["B"]).reshape(K, N)
    want = np.array(g["C"]).reshape(M, N)
    p = synthetic.Problem(M, N, K, dt, dt, ta, tb, g["alpha beta"][0], g["alpha beta"][1],
                          (A.T if ta else A).contiguous().to(synthetic.DTYPES[dt]),
                          (B.T if tb else B).contiguous().to(synthetic.DTYPES[dt]),
                          torch.zeros(M, N, dtype=synthetic.DTYPES[dt]))
    R, T = oracle.gemm(p)
    assert (R == want).all()
    assert (T == want).all()          # all products positive here


# ------------------------------------------------------ exact brute force

def exact_reference(p):
    """R and T in exact rational arithmetic from PyTorch-decoded operands."""
    Ad, Bd = torch_decode(p.A), torch_decode(p.B)
    a, b = op_a(p, Ad), op_b(p, Bd)
    Cd = torch_decode(p.C)
    alpha = Fraction(float(np.float32(p.alpha)))
    beta = Fraction(float(np.float32(p.beta)))
    R = np.empty((p.M, p.N), dtype=object)
    T = np.empty((p.M, p.N), dtype=object)
    for i in range(p.M):
        for j in range(p.N):
            s = Fraction(0)
            t = Fraction(0)
            for k in range(p.K):
                prod = Fraction(float(a[i, k])) * Fraction(float(b[k, j]))
                s += prod
                t += abs(prod)
            r = alpha * s
            if p.beta != 0:
                r += beta * Fraction(float(Cd[i, j]))
            R[i, j] = r
            T[i, j] = t
    return R, T


def tiny_problems():
    """A fixed family of tiny problems covering every dtype, layout, padded
    leading dimension, alpha/beta choice and a NaN-filled C with beta = 0."""
    out = []
    seed = 100
    for dt, (ta, tb) in itertools.product(["f16", "bf16", "f32"], LAYOUTS):
        for (M, N, K, alpha, beta, fill, pad) in [(3, 5, 4, 1.0, 0.0, "nan", 0),
                                                   (5, 2, 7, -0.75, 1.5, "uniform", 3),
                                                   (1, 6, 1, 2.0, -1.0, "uniform", 1)]:
            seed += 1
            lda = (M if ta else K) + pad if pad else 0
            ldb = (K if tb else N) + pad if pad else 0
            ldc = N + pad if pad else 0
            out.append(synthetic.make_problem(M, N, K, dt, dt, transpose_a=ta, transpose_b=tb,
                                              alpha=alpha, beta=beta, seed=seed, dist="normal",
                                              scale=3.0, c_fill=fill, lda=lda, ldb=ldb, ldc=ldc))
    return out


def pins_pass(lib) -> list[str]:
    """Run the pins against a build of the oracle; return the failures."""
    fails = []
    # exact rational brute force
    for p in tiny_problems():
        R, T = oracle.gemm(p, lib=lib)
        Rx, Tx = exact_reference(p)
        scale = np.array([[float(abs(v)) for v in row] for row in Tx]) + 1.0
        errR = np.array([[abs(float(Fraction(R[i, j]) - Rx[i, j])) if np.isfinite(R[i, j]) else np.inf
                          for j in range(p.N)] for i in range(p.M)])
        errT = np.array([[abs(float(Fraction(T[i, j]) - Tx[i, j])) if np.isfinite(T[i, j]) else np.inf
                          for j in range(p.N)] for i in range(p.M)])
        if not (errR <= 1e-13 * scale).all() or not (errT <= 1e-13 * scale).all():
            fails.append(f"brute force {p.M}x{p.N}x{p.K} {p.ab_dtype} {p.layout}")
        # the single-element path must agree with the row path bitwise
        ii, jj = np.meshgrid(np.arange(p.M), np.arange(p.N), indexing="ij")
        Rp, Tp = oracle.gemm_points(p, ii.ravel(), jj.ravel(), lib=lib)
        if not (np.array_equal(Rp, R.ravel(), equal_nan=True) and np.array_equal(Tp, T.ravel())):
            fails.append(f"points != rows {p.layout}")
    # decoder exhaustive
    for tdt in (torch.float16, torch.bfloat16):
        t = torch.arange(0, 65536, dtype=torch.int32).to(torch.int16).view(tdt)
        mine, ref = oracle.decode(t, lib=lib), torch_decode(t)
        if not np.array_equal(mine, ref, equal_nan=True):
            fails.append(f"decode {tdt}")
    # default (ld = 0) leading dimensions on a non-square problem
    p = synthetic.make_problem(3, 5, 4, "f32", "f32", transpose_a=True, transpose_b=True,
                               alpha=1.0, beta=1.0, seed=7, c_fill="uniform")
    s_rows = oracle.gemm(p, lib=lib)[0]
    s, keep = oracle._struct(p, lda=0, ldb=0, ldc=0)
    import ctypes
    R0 = np.empty((3, 5))
    T0 = np.empty((3, 5))
    dp = ctypes.POINTER(ctypes.c_double)
    lib.oracle_gemm_rows(ctypes.byref(s), 0, 3, R0.ctypes.data_as(dp), T0.ctypes.data_as(dp))
    if not np.array_equal(R0, s_rows):
        fails.append("ld = 0 default")
    return fails


def test_pins_pass_on_oracle():
    assert pins_pass(oracle.load_library()) == []


MUTATIONS = {
    # (regex on oracle.c, replacement): a plausible mistake each
    "transpose_a index swapped": (r"\? k \* lda \+ i : i \* lda \+ k", "? i * lda + k : k * lda + i"),
    "transpose_b ignored": (r"return p->transpose_b \? j \* ldb \+ k : k \* ldb \+ j;",
                            "return k * ldb + j;"),
    "beta term dropped": (r"r \+= p->beta \* load\(p->C, p->c_dtype, i \* ldc \+ j\);\n            S\[j\] = r;",
                          "S[j] = r;"),
    "alpha sign flipped": (r"double r = p->alpha \* S\[j\];", "double r = -p->alpha * S[j];"),
    "f16 exponent bias off by one": (r"e - 25\)", "e - 24)"),
    "bf16 subnormal scale wrong": (r"-133\)", "-126)"),
    "default ldc uses M": (r"\*ldc = p->ldc \? p->ldc : p->N;", "*ldc = p->ldc ? p->ldc : p->M;"),
    "T signed": (r"Ta\[j\] \+= fabs\(prod\);", "Ta[j] += prod;"),
    "last k dropped": (r"for \(int64_t k = 0; k < K; \+\+k\) \{\n            const double a",
                       "for (int64_t k = 0; k < K - 1; ++k) {\n            const double a"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name):
    pat, rep = MUTATIONS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    mutated, n = re.subn(pat, rep, src)
    assert n >= 1, f"mutation {name!r} did not apply"
    with tempfile.TemporaryDirectory() as d:
        cpath = os.path.join(d, "mutant.c")
        with open(cpath, "w") as f:
            f.write(mutated)
        so = oracle.build(cpath, os.path.join(d, "libmutant.so"))
        lib = oracle.load_library(so)
        assert pins_pass(lib) != [], f"planted mistake {name!r} went unnoticed"


# ------------------------------------------------------- library special case

@pytest.mark.parametrize("dt", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_vs_numpy_float64(dt, ta, tb):
    M, N, K = 67, 45, 129
    p = synthetic.make_problem(M, N, K, dt, "f32", transpose_a=ta, transpose_b=tb, alpha=0.5,
                               beta=-2.0, seed=11, dist="normal", c_fill="uniform",
                               lda=(M if ta else K) + 5, ldb=(K if tb else N) + 2, ldc=N + 7)
    R, T = oracle.gemm(p)
    a = op_a(p, torch_decode(p.A))
    b = op_b(p, torch_decode(p.B))
    ref = float(np.float32(0.5)) * (a @ b) + (-2.0) * torch_decode(p.C)[:, :N]
    Tref = np.abs(a) @ np.abs(b)
    assert np.all(np.abs(R - ref) <= 1e-12 * (Tref + 1.0))
    assert np.all(np.abs(T - Tref) <= 1e-12 * Tref)


# -------------------------------------------------------------- closed forms

@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_identity(dt):
    n = 40
    p = synthetic.make_problem(n, 24, n, dt, "f32", seed=3, dist="normal")
    p.A = torch.eye(n).to(synthetic.DTYPES[dt])
    R, _ = oracle.gemm(p)
    assert (R == torch_decode(p.B)).all()


def test_permutation_transposed():
    n = 33
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(9))
    P = torch.zeros(n, n)
    P[torch.arange(n), perm] = 1.0
    p = synthetic.make_problem(n, 17, n, "bf16", "f32", transpose_a=True, seed=4, dist="normal")
    p.A = P.T.contiguous().to(torch.bfloat16)        # stored [K,M]: op(A) = P
    R, _ = oracle.gemm(p)
    assert (R == torch_decode(p.B)[perm]).all()


@pytest.mark.parametrize("dt", ["f16", "bf16", "f32"])
def test_rank_one(dt):
    p = synthetic.make_problem(31, 29, 1, dt, "f32", seed=8, dist="normal")
    R, T = oracle.gemm(p)
    a = torch_decode(p.A)[:, 0]
    b = torch_decode(p.B)[0, :]
    assert (R == np.outer(a, b)).all()
    assert (T == np.abs(np.outer(a, b))).all()


def test_alpha_beta_integer_exact():
    p = synthetic.make_problem(20, 30, 50, "bf16", "f32", transpose_b=True, alpha=0.5, beta=1.0,
                               seed=12, dist="int", scale=4, c_fill="int")
    R, _ = oracle.gemm(p)
    a = op_a(p, torch_decode(p.A)).astype(np.int64)
    b = op_b(p, torch_decode(p.B)).astype(np.int64)
    exact = (a @ b) * 0.5 + torch_decode(p.C)
    assert (R == exact).all()


def test_beta_zero_ignores_nan_c():
    p = synthetic.make_problem(9, 7, 5, "f16", "f16", seed=2, c_fill="nan")
    R, _ = oracle.gemm(p)
    assert np.isfinite(R).all()


def test_linearity_in_alpha_and_beta():
    base = dict(M=12, N=10, K=40, ab_dtype="bf16", c_dtype="f32")
    p1 = synthetic.make_problem(**base, alpha=1.0, beta=0.0, seed=21, c_fill="uniform")
    p2 = synthetic.make_problem(**base, alpha=0.25, beta=0.0, seed=21, c_fill="uniform")
    p3 = synthetic.make_problem(**base, alpha=1.0, beta=2.0, seed=21, c_fill="uniform")
    R1, _ = oracle.gemm(p1)
    R2, _ = oracle.gemm(p2)
    R3, _ = oracle.gemm(p3)
    assert np.array_equal(R2, 0.25 * R1)                 # power-of-two scaling is exact
    assert np.allclose(R3 - R1, 2.0 * torch_decode(p1.C), rtol=0, atol=1e-12)


def test_sub_block_consistency():
    p = synthetic.make_problem(40, 36, 64, "f16", "f32", seed=13, dist="normal")
    R, T = oracle.gemm(p)
    q = synthetic.Problem(10, 12, 64, "f16", "f32", A=p.A[5:15].contiguous(),
                          B=p.B[:, 20:32].contiguous(), C=torch.zeros(10, 12))
    Rq, Tq = oracle.gemm(q)
    assert np.array_equal(Rq, R[5:15, 20:32]) and np.array_equal(Tq, T[5:15, 20:32])


def test_row_band_matches_full():
    p = synthetic.make_problem(30, 20, 50, "bf16", "bf16", seed=14, dist="normal")
    R, T = oracle.gemm(p)
    Rb, Tb = oracle.gemm(p, 7, 19)
    assert np.array_equal(Rb, R[7:19]) and np.array_equal(Tb, T[7:19])


# ---------------------------------------------------------------- epilogue
# tessl architecture.md, "Fused Epilogue": C = activation(alpha * A@B +
# beta * C_prev + bias), bias one value per column, activation GeluTanh.

def epilogue_pins_fail(gelu, epilogue):
    """Failing epilogue pins for the given GELU and epilogue functions
    (the oracle's own, or planted-mistake copies)."""
    fails = []
    # a library routine: PyTorch's tanh-approximated GELU in float64
    x = np.concatenate([np.linspace(-12.0, 12.0, 4001), [0.0, -0.0, 1.0, -1.0, 3.0, 1e-8, -1e-8, 40.0, -40.0]])
    ref = torch.nn.functional.gelu(torch.tensor(x, dtype=torch.float64), approximate="tanh").numpy()
    # (absolute 1e-14: far in the negative tail 1 + tanh rounds to 0 or to
    # a few ulp of 1 depending on the routine; the true value is ~1e-16)
    if not np.allclose(gelu(x), ref, rtol=1e-12, atol=1e-14):
        fails.append("gelu vs torch tanh-GELU")
    # identities: gelu(x) - gelu(-x) = x; gelu(0) = 0; gelu(x) -> x for large x
    y = np.linspace(-6.0, 6.0, 1201)
    if not np.allclose(gelu(y) - gelu(-y), y, rtol=0, atol=1e-14):
        fails.append("odd part")
    if gelu(np.array([0.0]))[0] != 0.0 or abs(gelu(np.array([30.0]))[0] - 30.0) > 1e-12:
        fails.append("gelu(0), gelu(30)")
    # zero A: C = act(beta * C_old + bias), with bias broadcast over rows
    # (M != N so a per-row bias cannot pass)
    M, N, K = 5, 7, 3
    g = torch.Generator().manual_seed(11)
    Cold = (torch.rand(M, N, generator=g) * 4 - 2).to(torch.bfloat16)
    bias = (torch.rand(N, generator=g) * 4 - 2).to(torch.bfloat16)
    p = synthetic.Problem(M, N, K, "bf16", "bf16", False, False, 1.0, 0.5,
                          torch.zeros(M, K, dtype=torch.bfloat16), torch.ones(K, N, dtype=torch.bfloat16), Cold)
    pre = 0.5 * torch_decode(Cold) + torch_decode(bias)[None, :]
    for act, f in (("none", lambda v: v), ("gelu_tanh", lambda v: torch.nn.functional.gelu(
            torch.tensor(v), approximate="tanh").numpy())):
        R, _, Y = epilogue(p, bias, act)
        if not (np.allclose(Y, pre, rtol=1e-15, atol=0) and np.allclose(R, f(pre), rtol=1e-12, atol=1e-15)):
            fails.append(f"zero A, bias, {act}")
    # identity A: C = act(B + bias) on every column
    p = synthetic.Problem(4, 6, 4, "f32", "f32", False, False, 1.0, 0.0, torch.eye(4),
                          torch.arange(24, dtype=torch.float32).reshape(4, 6) / 8 - 1, torch.zeros(4, 6))
    b = torch.tensor([0.5, -1.0, 0.25, 2.0, -3.0, 0.0])
    R, _, _ = epilogue(p, b, "gelu_tanh")
    want = torch.nn.functional.gelu(p.B.double() + b.double()[None, :], approximate="tanh").numpy()
    if not np.allclose(R, want, rtol=1e-12, atol=1e-15):
        fails.append("identity A")
    return fails


def test_epilogue_pins_pass_on_oracle():
    assert epilogue_pins_fail(oracle.gelu_tanh, oracle.gemm_epilogue) == []


def _wrong_cubic(x):
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + np.tanh(oracle.SQRT_2_OVER_PI * (x + 0.0447 * x ** 3)))


def _wrong_scale(x):
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + np.tanh(np.sqrt(2.0) / np.pi * (x + oracle.GELU_CUBIC * x ** 3)))


def _bias_after_activation(p, bias, act):
    R, T = oracle.gemm(p)
    Y = oracle.apply_activation(R, act)
    return (Y if bias is None else Y + oracle.decode(bias).reshape(1, -1)), T, R


def _bias_per_row(p, bias, act):
    R, T = oracle.gemm(p)
    bd = oracle.decode(bias).reshape(-1)
    Y = R + np.resize(bd, p.M)[:, None]
    return oracle.apply_activation(Y, act), T, Y


EPILOGUE_MUTATIONS = {
    "gelu cubic coefficient 0.0447": (_wrong_cubic, oracle.gemm_epilogue),
    "gelu scale sqrt(2)/pi": (_wrong_scale, oracle.gemm_epilogue),
    "bias added after the activation": (oracle.gelu_tanh, _bias_after_activation),
    "bias indexed by row": (oracle.gelu_tanh, _bias_per_row),
}


@pytest.mark.parametrize("name", sorted(EPILOGUE_MUTATIONS))
def test_planted_epilogue_mistake_is_caught(name):
    gelu, epi = EPILOGUE_MUTATIONS[name]
    assert epilogue_pins_fail(gelu, epi) != [], f"planted mistake {name!r} went unnoticed"


def test_epilogue_points_match_rows():
    p = synthetic.make_problem(9, 11, 13, "f16", "f16", alpha=0.5, beta=1.0, seed=12, c_fill="uniform")
    bias = (torch.linspace(-1, 1, 11)).to(torch.float16)
    R, T, Y = oracle.gemm_epilogue(p, bias, "gelu_tanh")
    ii, jj = np.meshgrid(np.arange(9), np.arange(11), indexing="ij")
    Rp, Tp, Yp = oracle.gemm_epilogue_points(p, bias, "gelu_tanh", ii.ravel(), jj.ravel())
    assert np.array_equal(Rp, R.ravel()) and np.array_equal(Tp, T.ravel()) and np.array_equal(Yp, Y.ravel())


# ---------------------------------------------------------------- int8 GEMM
# tessl architecture.md, "Integer GEMM": exact int8 x int8 accumulation,
# per-column dequantisation.

def test_i8_decoder_exhaustive():
    t = torch.arange(-128, 128, dtype=torch.int16).to(torch.int8)
    assert np.array_equal(oracle.decode(t), t.to(torch.float64).numpy())


def _i8_problem(M, N, K, ta, tb, seed, lo=-128, hi=127):
    g = torch.Generator().manual_seed(seed)
    A = torch.randint(lo, hi + 1, (K, M) if ta else (M, K), generator=g).to(torch.int8)
    B = torch.randint(lo, hi + 1, (N, K) if tb else (K, N), generator=g).to(torch.int8)
    return synthetic.Problem(M, N, K, "i8", "f32", ta, tb, 1.0, 0.0, A, B, torch.zeros(M, N))


@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_i8_brute_force(ta, tb):
    p = _i8_problem(3, 4, 5, ta, tb, seed=9)
    Ai = [[int(v) for v in row] for row in p.A.tolist()]
    Bi = [[int(v) for v in row] for row in p.B.tolist()]
    a = (lambda i, k: Ai[k][i]) if ta else (lambda i, k: Ai[i][k])
    b = (lambda k, j: Bi[j][k]) if tb else (lambda k, j: Bi[k][j])
    exact = np.array([[sum(a(i, k) * b(k, j) for k in range(5)) for j in range(4)] for i in range(3)], float)
    R, T = oracle.gemm(p)
    assert np.array_equal(R, exact)
    assert np.array_equal(T, np.array([[sum(abs(a(i, k) * b(k, j)) for k in range(5)) for j in range(4)]
                                       for i in range(3)], float))


def test_i8_full_range_at_the_k_limit():
    """All -128: every product is 2^14; at K = 131072 the sum is 2^31, one
    past the int32 range -- the oracle's fp64 sum is exact."""
    K = 131072
    p = synthetic.Problem(2, 3, K, "i8", "f32", False, False, 1.0, 0.0, torch.full((2, K), -128, dtype=torch.int8),
                          torch.full((K, 3), -128, dtype=torch.int8), torch.zeros(2, 3))
    R, T = oracle.gemm(p)
    assert (R == 2.0 ** 31).all() and (T == 2.0 ** 31).all()


def test_i8_dequant_closed_form():
    """Identity A: acc = B, so C = alpha * B * scale[n] + beta * C_old."""
    N = 6
    B = torch.tensor([[3, -7, 127, -128, 0, 5], [1, 2, 3, 4, 5, 6]], dtype=torch.int8)
    scale = torch.tensor([0.5, 2.0, 1e-3, -0.25, 7.0, 1.0])
    Cold = torch.arange(12, dtype=torch.float32).reshape(2, 6)
    p = synthetic.Problem(2, N, 2, "i8", "f32", False, False, 0.5, 2.0, torch.eye(2, dtype=torch.int8), B, Cold)
    R, _, ACC = oracle.gemm_i8_dequant(p, scale)
    want = 0.5 * B.double().numpy() * scale.double().numpy()[None, :] + 2.0 * Cold.double().numpy()
    assert np.array_equal(ACC, B.double().numpy())
    assert np.allclose(R, want, rtol=1e-15, atol=0)


# ------------------------------------------------- int8-weight (Q8) product
# Foundry metal.md, "Custom Compute Kernels": fm_sgemm_q8(X[M,K], W_q8[N,K],
# scales[N]), Out = X @ (W_q8 * scale[n])^T, with alpha/beta on top.

def _q8_tiny(M, N, K, seed, x_dtype="f16", alpha=1.0, beta=0.0):
    g = torch.Generator().manual_seed(seed)
    X = torch.randn(M, K, generator=g).to(synthetic.DTYPES[x_dtype])
    W = torch.randint(-128, 128, (N, K), generator=g).to(torch.int8)
    scale = (torch.rand(N, generator=g) * 2 - 1) * 1e-2
    C = (torch.rand(M, N, generator=g) * 2 - 1)
    return synthetic.Problem(M, N, K, x_dtype, "f32", False, True, alpha, beta, X, W, C), scale


def q8_pins_fail(fn):
    """Failing pins of an int8-weight product function fn(p, scale) ->
    (R, T, ACC) (the oracle's own, or planted-mistake copies)."""
    fails = []
    # exact rational brute force: alpha * scale[n] * sum_k x w + beta * c
    for x_dtype in ("f16", "bf16"):
        p, scale = _q8_tiny(3, 4, 5, seed=21, x_dtype=x_dtype, alpha=0.75, beta=-0.5)
        X = [[Fraction(float(v)) for v in row] for row in p.A.double().tolist()]
        W = [[int(v) for v in row] for row in p.B.tolist()]
        s = [Fraction(float(v)) for v in scale.tolist()]
        Cf = [[Fraction(float(v)) for v in row] for row in p.C.double().tolist()]
        a, b = Fraction(float(np.float32(0.75))), Fraction(float(np.float32(-0.5)))
        exact = np.array([[float(a * s[j] * sum(X[i][k] * W[j][k] for k in range(5)) + b * Cf[i][j])
                           for j in range(4)] for i in range(3)])
        t_exact = np.array([[float(abs(s[j]) * sum(abs(X[i][k] * W[j][k]) for k in range(5)))
                             for j in range(4)] for i in range(3)])
        R, T, _ = fn(p, scale)
        if not (np.allclose(R, exact, rtol=1e-14, atol=1e-300) and np.allclose(T, t_exact, rtol=1e-14, atol=0)):
            fails.append(f"brute force {x_dtype}")
    # identity weight (N = K): Out = X * scale[n] column by column, exactly
    N = 6
    g = torch.Generator().manual_seed(22)
    X = torch.randn(2, N, generator=g).to(torch.float16)
    scale = torch.tensor([0.5, -2.0, 1e-3, 0.25, 7.0, 1.0])
    p = synthetic.Problem(2, N, N, "f16", "f32", False, True, 1.0, 0.0, X, torch.eye(N, dtype=torch.int8),
                          torch.zeros(2, N))
    R, _, _ = fn(p, scale)
    if not np.array_equal(R, X.double().numpy() * scale.double().numpy()[None, :]):
        fails.append("identity weight")
    # all-ones activations (M != N): Out[m, n] = scale[n] * sum_k W[n, k] on every row
    W = torch.tensor([[1, -2, 3], [127, -128, 0], [5, 5, 5], [-1, 0, 1], [9, -8, 7]], dtype=torch.int8)
    scale = torch.tensor([0.5, 2.0, -1.0, 4.0, 0.125])
    p = synthetic.Problem(2, 5, 3, "bf16", "f32", False, True, 1.0, 0.0, torch.ones(2, 3, dtype=torch.bfloat16),
                          W, torch.zeros(2, 5))
    R, _, _ = fn(p, scale)
    want = (W.double().sum(1) * scale.double()).numpy()
    if not (np.array_equal(R[0], want) and np.array_equal(R[1], want)):
        fails.append("all-ones activations")
    # integer activations, scale 1: the product sum is an exact integer
    g = torch.Generator().manual_seed(23)
    X = torch.randint(-4, 5, (3, 40), generator=g).to(torch.float16)
    W = torch.randint(-128, 128, (7, 40), generator=g).to(torch.int8)
    p = synthetic.Problem(3, 7, 40, "f16", "f32", False, True, 1.0, 0.0, X, W, torch.zeros(3, 7))
    R, _, ACC = fn(p, torch.ones(7))
    want = X.long() @ W.long().T
    if not (np.array_equal(R, want.double().numpy()) and np.array_equal(ACC, want.double().numpy())):
        fails.append("integer activations")
    return fails


def test_q8_pins_pass_on_oracle():
    assert q8_pins_fail(oracle.gemm_q8_weight) == []


def _q8_scale_by_row(p, scale):
    R, T, ACC = oracle.gemm_q8_weight(p, torch.ones(p.N))
    sc = np.resize(scale.double().numpy(), p.M)[:, None]
    return R * sc, T * np.abs(sc), ACC


def _q8_weight_not_transposed(p, scale):
    # the same bytes read as a weight stored [K,N]
    import copy
    q = copy.copy(p)
    q.transpose_b = False
    q.B = p.B.contiguous().reshape(p.K, p.N)
    return oracle.gemm_q8_weight(q, scale)


def _q8_t_unscaled(p, scale):
    R, T, ACC = oracle.gemm_q8_weight(p, scale)
    return R, T / np.abs(np.where(scale.double().numpy() == 0, 1.0, scale.double().numpy()))[None, : p.N], ACC


def _q8_scale_divides(p, scale):
    return oracle.gemm_q8_weight(p, 1.0 / scale)


Q8_MUTATIONS = {
    "scale indexed by row": _q8_scale_by_row,
    "weight read as stored [K,N]": _q8_weight_not_transposed,
    "T without the scale": _q8_t_unscaled,
    "scale divides": _q8_scale_divides,
}


@pytest.mark.parametrize("name", sorted(Q8_MUTATIONS))
def test_planted_q8_mistake_is_caught(name):
    assert q8_pins_fail(Q8_MUTATIONS[name]) != [], f"planted mistake {name!r} went unnoticed"


def test_q8_points_match_rows():
    p, scale = _q8_tiny(6, 9, 33, seed=24, alpha=0.5, beta=2.0)
    R, T, ACC = oracle.gemm_q8_weight(p, scale)
    ii, jj = np.meshgrid(np.arange(6), np.arange(9), indexing="ij")
    Rp, Tp, Ap = oracle.gemm_q8_weight_points(p, scale, ii.ravel(), jj.ravel())
    assert np.array_equal(Rp, R.ravel()) and np.array_equal(Tp, T.ravel()) and np.array_equal(Ap, ACC.ravel())
