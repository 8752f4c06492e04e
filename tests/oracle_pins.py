"""Checks that pin the CPU oracle to facts outside itself (test helper).

Each ``pin_*`` function takes a reference callable
``ref(A16, B16, apply_relu) -> float64 (M, N) array`` and returns a list of
failure messages (empty when the callable passes).  They are run against
the real oracle (all must pass) and against deliberately broken variants of
it (each variant must fail at least one), which shows the pins can see the
mistakes they are meant to catch.

What fixes the expected values, none of it the oracle's own code:
* hand-worked fixtures (tests/golden), exact rationals;
* brute force in exact rational arithmetic (``fractions``) on tiny inputs,
  with binary16 values decoded by numpy (bfloat16 words by a float32 bit
  shift);
* integer inputs whose products and sums are exact in every format,
  checked against numpy int64 matmul;
* closed forms: identity B gives ReLU(A), all-ones A gives ReLU of B's
  column sums;
* invariants: ReLU output non-negative with no -0; zero K-padding changes
  nothing; relu-off is odd in A and homogeneous in B; relu-on equals
  max(relu-off, 0); (A.B)^T equals B^T.A^T;
* a float64 matmul from a library (torch CPU) within the binary64 bound;
* IEEE 754 rules for NaN and infinite operands (a NaN operand or 0 x inf
  makes the product NaN, inf + (-inf) is NaN, a NaN term makes the sum
  NaN), applied term by term with Python floats, and ReLU read as
  x > 0 ? x : +0 (NaN and -inf become +0).
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import torch

from golden_io import all_fixtures

U64 = 2.0 ** -53  # unit roundoff of binary64


class F16:
    """binary16 inputs: numpy float16 arrays, decoded by numpy."""
    name = "f16"

    @staticmethod
    def enc(x):
        return np.asarray(x, dtype=np.float64).astype(np.float16)

    @staticmethod
    def dec(a):
        return np.asarray(a).astype(np.float64)


class BF16:
    """bfloat16 inputs: uint16 words (the top half of a binary32), decoded by
    shifting them into a numpy float32 -- not by the oracle's decoder."""
    name = "bf16"

    @staticmethod
    def enc(x):
        f = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32))
        u = f.view(np.uint32).astype(np.uint64)
        return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)  # round to nearest even

    @staticmethod
    def dec(a):
        return (np.ascontiguousarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _h(x):
    return F16.enc(x)


def _frac(x):
    """Exact rational value of a finite float; None for inf/NaN."""
    x = float(x)
    return Fraction(x) if np.isfinite(x) else None


def _exact_product(A16, B16, fmt=F16):
    """Exact rational A.B (lists of Fractions) from 16-bit inputs."""
    Af = [[Fraction(float(v)) for v in row] for row in fmt.dec(A16)]
    Bf = [[Fraction(float(v)) for v in row] for row in fmt.dec(B16)]
    M, K = len(Af), len(Bf)
    N = B16.shape[1]
    return [[sum((Af[i][k] * Bf[k][j] for k in range(K)), Fraction(0)) for j in range(N)]
            for i in range(M)]


def _bound(A16, B16, fmt=F16):
    """gamma_K * |A|.|B| : a rigorous bound on binary64 accumulation error."""
    K = A16.shape[1]
    gk = K * U64 / (1 - K * U64) if K else 0.0
    return gk * (np.abs(fmt.dec(A16)) @ np.abs(fmt.dec(B16)))


def pin_golden(ref):
    fails = []
    for fx in all_fixtures():
        for relu, key in ((True, "C_relu"), (False, "C_norelu")):
            got = ref(fx["A"], fx["B"], relu)
            exp = fx[key]
            for i, row in enumerate(exp):
                for j, e in enumerate(row):
                    if _frac(got[i, j]) != e:
                        fails.append(f"golden {fx['name']} relu={relu} [{i},{j}]: {got[i, j]} != {e}")
    return fails


def pin_bruteforce(ref, trials=40, seed=123, fmt=F16):
    rng = np.random.default_rng(seed)
    fails = []
    for t in range(trials):
        M, N, K = (int(x) for x in rng.integers(1, 8, size=3))
        A = fmt.enc(rng.standard_normal((M, K)) * 3)
        B = fmt.enc(rng.standard_normal((K, N)) * 3)
        exact = _exact_product(A, B, fmt)
        bnd = _bound(A, B, fmt)
        for relu in (True, False):
            got = ref(A, B, relu)
            for i in range(M):
                for j in range(N):
                    e = exact[i][j]
                    if relu:
                        e = max(e, Fraction(0))
                    g = _frac(got[i, j])
                    if g is None or abs(g - e) > Fraction(float(bnd[i, j])):
                        fails.append(f"bruteforce t={t} ({M},{N},{K}) relu={relu} [{i},{j}]: "
                                     f"{got[i, j]!r} vs {float(e)!r}")
    return fails


def pin_integer_exact(ref, seed=7, fmt=F16):
    rng = np.random.default_rng(seed)
    M, N, K = 33, 47, 300
    Ai = rng.integers(-2, 3, size=(M, K))
    Bi = rng.integers(-2, 3, size=(K, N))
    exact = Ai.astype(np.int64) @ Bi.astype(np.int64)
    fails = []
    for relu in (True, False):
        got = ref(fmt.enc(Ai), fmt.enc(Bi), relu)
        exp = np.maximum(exact, 0) if relu else exact
        if not np.array_equal(got, exp.astype(np.float64)):
            bad = np.argwhere(got != exp)
            fails.append(f"integer relu={relu}: {len(bad)} mismatches, first {bad[0].tolist()}")
    return fails


def pin_identity(ref, seed=11, fmt=F16):
    rng = np.random.default_rng(seed)
    M, K = 9, 13
    A = fmt.enc(rng.standard_normal((M, K)))
    I = fmt.enc(np.eye(K))
    got = ref(A, I, True)
    exp = np.maximum(fmt.dec(A), 0.0)
    return [] if np.array_equal(got, exp) else ["identity B did not give ReLU(A)"]


def pin_ones(ref, seed=12, fmt=F16):
    rng = np.random.default_rng(seed)
    M, N, K = 4, 10, 12
    Ai = np.ones((M, K))
    B = fmt.enc(rng.standard_normal((K, N)))
    Bv = fmt.dec(B)
    fails = []
    colsum = [sum((Fraction(float(Bv[k, j])) for k in range(K)), Fraction(0)) for j in range(N)]
    bnd = _bound(fmt.enc(Ai), B, fmt)
    got = ref(fmt.enc(Ai), B, True)
    for i in range(M):
        for j in range(N):
            e = max(colsum[j], Fraction(0))
            g = _frac(got[i, j])
            if g is None or abs(g - e) > Fraction(float(bnd[i, j])):
                fails.append(f"all-ones A [{i},{j}]: {got[i, j]} vs {float(e)}")
    return fails


def pin_invariants(ref, seed=13, fmt=F16):
    rng = np.random.default_rng(seed)
    fails = []
    M, N, K = 17, 23, 29
    A = fmt.enc(rng.standard_normal((M, K)))
    B = fmt.enc(rng.standard_normal((K, N)))
    on = ref(A, B, True)
    off = ref(A, B, False)
    if (on < 0).any() or np.signbit(on).any():
        fails.append("ReLU output has negatives or -0")
    if not np.array_equal(on, np.where(off > 0, off, 0.0)):
        fails.append("relu-on != max(relu-off, 0)")
    # zero K padding
    Ap = np.concatenate([A, fmt.enc(np.zeros((M, 7)))], axis=1)
    Bp = np.concatenate([B, fmt.enc(np.zeros((7, N)))], axis=0)
    if not np.array_equal(ref(Ap, Bp, False), off):
        fails.append("zero K-tail changed the result")
    # odd in A, homogeneous in B (negation and scaling by 2 are exact)
    if not np.array_equal(ref(fmt.enc(-fmt.dec(A)), B, False), -off):
        fails.append("relu-off not odd in A")
    if not np.array_equal(ref(A, fmt.enc(fmt.dec(B) * 2), False), 2 * off):
        fails.append("relu-off not homogeneous in B")
    # transpose: (A.B)^T == B^T.A^T (same k order per entry => bit-identical)
    if not np.array_equal(ref(np.ascontiguousarray(B.T), np.ascontiguousarray(A.T), False), off.T):
        fails.append("(A.B)^T != B^T.A^T")
    return fails


def pin_torch64(ref, seed=14, fmt=F16):
    rng = np.random.default_rng(seed)
    M, N, K = 40, 50, 300
    A = fmt.enc(rng.standard_normal((M, K)))
    B = fmt.enc(rng.standard_normal((K, N)))
    lib = (torch.from_numpy(fmt.dec(A)) @ torch.from_numpy(fmt.dec(B))).numpy()
    bnd = 2 * _bound(A, B, fmt)  # both sides round in binary64, orders may differ
    fails = []
    for relu in (True, False):
        exp = np.maximum(lib, 0) if relu else lib
        got = ref(A, B, relu)
        if not (np.abs(got - exp) <= bnd).all():
            fails.append(f"torch float64 matmul disagrees (relu={relu}), "
                         f"max err {np.abs(got - exp).max():.3e}")
    return fails


def ieee_expected(Ad, Bd, relu):
    """Exact A.B for decoded inputs holding NaN / infinities, by the IEEE 754
    rules applied to each term: NaN if a product is NaN (a NaN operand or
    0 x inf) or the infinite products have both signs; the infinity of the
    one sign present otherwise; else the exact rational sum.  ReLU: x > 0 ?
    x : +0.  Returns float64 (finite sums rounded once)."""
    M, K = Ad.shape
    N = Bd.shape[1]
    out = np.empty((M, N))
    for i in range(M):
        for j in range(N):
            terms = [float(Ad[i, k]) * float(Bd[k, j]) for k in range(K)]
            if any(t != t for t in terms):
                v = float("nan")
            elif any(t == float("inf") for t in terms) and any(t == float("-inf") for t in terms):
                v = float("nan")
            elif any(t == float("inf") for t in terms):
                v = float("inf")
            elif any(t == float("-inf") for t in terms):
                v = float("-inf")
            else:
                v = float(sum((Fraction(float(Ad[i, k])) * Fraction(float(Bd[k, j])) for k in range(K)),
                              Fraction(0)))
            if relu:
                v = v if v > 0 else 0.0
            out[i, j] = v
    return out


def special_inputs(M, N, K, seed, fmt=F16):
    """Finite random A, B (|x| < 2) with NaN and infinities planted so that
    C holds every case: a NaN row and column, +inf rows and columns whose
    other factor is positive, negative or zero, and dot products with
    +inf and -inf terms (NaN)."""
    rng = np.random.default_rng(seed)
    A = rng.uniform(-2, 2, (M, K))
    B = rng.uniform(-2, 2, (K, N))
    B[rng.random((K, N)) < 0.15] = 0.0
    inf, nan = float("inf"), float("nan")
    A[0, K // 3] = nan
    A[1 % M, 0] = inf
    A[2 % M, K - 1] = -inf
    A[3 % M, 1 % K], A[3 % M, K // 2] = inf, -inf
    B[K // 4, 1 % N] = nan
    B[(K - 1) // 2, 2 % N] = -inf
    B[K - 1, 3 % N] = inf
    return fmt.enc(A), fmt.enc(B)


def pin_ieee_specials(ref, fmt=F16):
    fails = []
    for t, (M, N, K) in enumerate([(5, 6, 7), (4, 9, 16), (6, 4, 33)]):
        A, B = special_inputs(M, N, K, seed=31 + t, fmt=fmt)
        for relu in (True, False):
            exp = ieee_expected(fmt.dec(A), fmt.dec(B), relu)
            got = ref(A, B, relu)
            same_nan = np.isnan(got) == np.isnan(exp)
            fin = np.isfinite(exp)
            same_inf = np.where(np.isinf(exp), got == exp, True)
            close = np.where(fin, np.abs(np.where(fin, got, 0) - np.where(fin, exp, 0))
                             <= 4 * _bound(np.where(np.isfinite(fmt.dec(A)), A, 0).astype(A.dtype),
                                           np.where(np.isfinite(fmt.dec(B)), B, 0).astype(B.dtype), fmt)
                             + 1e-300, True)
            bad = ~(same_nan & same_inf & close)
            if relu:
                bad |= np.signbit(got) & (got == 0)
            if bad.any():
                i, j = np.argwhere(bad)[0]
                fails.append(f"IEEE specials {M}x{N}x{K} relu={relu} [{i},{j}]: {got[i, j]} != {exp[i, j]}")
    return fails


ALL_PINS = [pin_golden, pin_bruteforce, pin_integer_exact, pin_identity, pin_ones,
            pin_invariants, pin_torch64, pin_ieee_specials]
# the pins that take a ``fmt`` (the golden fixtures are binary16 values)
FMT_PINS = [pin_bruteforce, pin_integer_exact, pin_identity, pin_ones, pin_invariants,
            pin_torch64, pin_ieee_specials]
