"""The CPU oracle against its pins, and the pins against planted mistakes.

CPU only (no GPU, no CUDA library).  The planted mistakes are made in the
oracle, on the CPU: each mutant wraps the real oracle with one plausible
bug, and at least one pin must reject it.
"""
import numpy as np
import pytest

import oracle_pins as P
from oracle import matches_ieee as oracle_matches


def _real(oracle_mod):
    return lambda A, B, relu: oracle_mod.gemm_relu(A, B, relu)


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_passes_pin(oracle_mod, pin):
    fails = pin(_real(oracle_mod))
    assert not fails, "\n".join(fails[:10])


def test_half_decode_matches_ieee(oracle_mod):
    # spot values from the binary16 definition
    known = {0x3C00: 1.0, 0xC000: -2.0, 0x7BFF: 65504.0, 0x0001: 2.0 ** -24,
             0x0400: 2.0 ** -14, 0x03FF: 1023 * 2.0 ** -24, 0x3555: 0.333251953125,
             0x0000: 0.0, 0x7C00: float("inf"), 0xFC00: float("-inf")}
    for bits, val in known.items():
        assert oracle_mod.half_to_double(bits) == val, hex(bits)
    assert np.signbit(oracle_mod.half_to_double(0x8000))
    assert np.isnan(oracle_mod.half_to_double(0x7E00))
    # every finite pattern against numpy's conversion
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_mod.half_to_double(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.signbit(got[finite]), np.signbit(ref[finite]))


def test_entries_equal_full_product(oracle_mod):
    rng = np.random.default_rng(5)
    M, N, K = 37, 41, 130
    A = rng.standard_normal((M, K)).astype(np.float16)
    B = rng.standard_normal((K, N)).astype(np.float16)
    full = oracle_mod.gemm_relu(A, B, True)
    rows = rng.integers(0, M, 200)
    cols = rng.integers(0, N, 200)
    ent = oracle_mod.gemm_relu_entries(A, B, rows, cols, True)
    assert np.array_equal(ent, full[rows, cols])


def test_threads_do_not_change_bits(oracle_mod):
    rng = np.random.default_rng(6)
    A = rng.standard_normal((64, 96)).astype(np.float16)
    B = rng.standard_normal((96, 80)).astype(np.float16)
    assert np.array_equal(oracle_mod.gemm_relu(A, B, True, threads=1),
                          oracle_mod.gemm_relu(A, B, True, threads=4))


def test_degenerate_shapes(oracle_mod):
    A = np.zeros((3, 0), np.float16)
    B = np.zeros((0, 5), np.float16)
    c = oracle_mod.gemm_relu(A, B, True)
    assert c.shape == (3, 5) and not c.any() and not np.signbit(c).any()
    assert oracle_mod.gemm_relu(np.zeros((0, 4), np.float16), np.zeros((4, 2), np.float16)).shape == (0, 2)


def test_tolerance_rule():
    # |c - ref| <= 1e-2 + 1e-2 |ref|
    import oracle
    ref = np.array([0.0, 1.0, 100.0, -3.0])
    ok = oracle.within_tolerance(ref + np.array([0.0099, 0.0199, 1.0099, 0.0399]), ref)
    assert ok.tolist() == [True, True, True, True]
    bad = oracle.within_tolerance(ref + np.array([0.0101, 0.0201, 1.02, 0.0401]), ref)
    assert bad.tolist() == [False, False, False, False]


# ---- planted mistakes: each must be caught by at least one pin -------------

def _mutants(oracle_mod):
    g = oracle_mod.gemm_relu

    def drop_last_k(A, B, r):
        if A.shape[1] <= 1:
            return np.zeros((A.shape[0], B.shape[1]))
        return g(np.ascontiguousarray(A[:, :-1]), np.ascontiguousarray(B[:-1, :]), r)

    def transposed_b(A, B, r):  # reads B with the wrong stride
        return g(A, np.ascontiguousarray(B.T).reshape(B.shape), r)

    def relu_as_min(A, B, r):
        off = g(A, B, False)
        return np.minimum(off, 0.0) if r else off

    def relu_ignored(A, B, r):
        return g(A, B, False)

    def rows_shifted(A, B, r):
        return np.roll(g(A, B, r), 1, axis=0)

    def wrong_exponent_bias(A, B, r):
        return g(A, B, r) * 0.25

    def fp16_accumulator(A, B, r):
        M, K = A.shape
        acc = np.zeros((M, B.shape[1]), np.float16)
        for k in range(K):
            acc = (acc.astype(np.float64) + np.outer(A[:, k].astype(np.float64),
                                                     B[k].astype(np.float64))).astype(np.float16)
        out = acc.astype(np.float64)
        return np.where(out > 0, out, 0.0) if r else out

    def first_term_subtracted(A, B, r):
        off = g(A, B, False) - 2 * np.outer(A[:, 0].astype(np.float64), B[0].astype(np.float64))
        return np.where(off > 0, off, 0.0) if r else off

    def negative_zero_kept(A, B, r):
        off = g(A, B, False)
        return np.where(off > 0, off, -0.0) if r else off

    return [drop_last_k, transposed_b, relu_as_min, relu_ignored, rows_shifted,
            wrong_exponent_bias, fp16_accumulator, first_term_subtracted, negative_zero_kept]


@pytest.mark.parametrize("idx", range(9))
def test_pins_catch_planted_mistake(oracle_mod, idx):
    mutant = _mutants(oracle_mod)[idx]
    caught = [pin.__name__ for pin in P.ALL_PINS if pin(mutant)]
    assert caught, f"no pin caught the planted mistake {mutant.__name__}"


def _special_mutants(oracle_mod):
    """Plausible mistakes that only non-finite inputs show."""
    g = oracle_mod.gemm_relu

    def relu_passes_nan(A, B, r):  # max written as x < 0 ? 0 : x
        off = g(A, B, False)
        return np.where(off < 0, 0.0, off) if r else off

    def nan_operands_dropped(A, B, r):
        A2 = np.where(np.isnan(A.astype(np.float64)), 0, A).astype(A.dtype)
        B2 = np.where(np.isnan(B.astype(np.float64)), 0, B).astype(B.dtype)
        return g(A2, B2, r)

    def zero_factor_terms_skipped(A, B, r):  # 0 x inf counted as 0
        a = A.astype(np.float64)
        b = B.astype(np.float64)
        with np.errstate(invalid="ignore"):
            t = a[:, :, None] * b[None, :, :]
            t = np.where((a[:, :, None] == 0) | (b[None, :, :] == 0), 0.0, t)
            off = t.sum(axis=1)
        return np.where(off > 0, off, 0.0) if r else off

    def infinity_saturated(A, B, r):  # a clamping cast instead of IEEE overflow
        return np.clip(g(A, B, r), -oracle_mod.FP16_MAX, oracle_mod.FP16_MAX)

    return [relu_passes_nan, nan_operands_dropped, zero_factor_terms_skipped, infinity_saturated]


@pytest.mark.parametrize("idx", range(4))
def test_pins_catch_planted_mistake_with_specials(oracle_mod, idx):
    mutant = _special_mutants(oracle_mod)[idx]
    caught = [pin.__name__ for pin in P.ALL_PINS if pin(mutant)]
    assert caught, f"no pin caught the planted mistake {mutant.__name__}"


def test_specials_by_hand(oracle_mod):
    """Small cases whose results follow from the IEEE 754 rules alone."""
    inf, nan = float("inf"), float("nan")
    h = np.float16
    # a NaN operand: its row is NaN, +0 after ReLU
    A = np.array([[1, nan], [2, 3]], h)
    B = np.array([[1, 1], [1, 1]], h)
    off = oracle_mod.gemm_relu(A, B, False)
    assert np.isnan(off[0]).all() and off[1].tolist() == [5.0, 5.0]
    on = oracle_mod.gemm_relu(A, B, True)
    assert on[0].tolist() == [0.0, 0.0] and not np.signbit(on[0]).any()
    # inf times a positive, a negative and a zero factor
    A = np.array([[inf, 1]], h)
    B = np.array([[1, -1, 0], [1, 1, 1]], h)
    off = oracle_mod.gemm_relu(A, B, False)
    assert off[0, 0] == inf and off[0, 1] == -inf and np.isnan(off[0, 2])
    assert oracle_mod.gemm_relu(A, B, True)[0].tolist() == [inf, 0.0, 0.0]
    # inf + (-inf) is NaN; inf + inf stays inf
    assert np.isnan(oracle_mod.gemm_relu(np.array([[inf, -inf]], h), np.array([[1], [1]], h), False)[0, 0])
    assert oracle_mod.gemm_relu(np.array([[inf, inf]], h), np.array([[1], [2]], h), False)[0, 0] == inf
    # finite results beyond binary16's range stay finite (the oracle does not round)
    big = oracle_mod.gemm_relu(np.array([[65504, 65504]], h), np.array([[65504], [65504]], h), True)
    assert big[0, 0] == 2 * 65504.0 ** 2


def test_matches_ieee_rule():
    ref = np.array([np.nan, np.inf, -np.inf, 1.0, 0.0])
    assert oracle_matches(np.array([np.nan, np.inf, -np.inf, 1.005, 0.0]), ref).all()
    assert not oracle_matches(np.array([0.0, np.inf, -np.inf, 1.0, 0.0]), ref)[0]
    assert not oracle_matches(np.array([np.nan, -np.inf, -np.inf, 1.0, 0.0]), ref)[1]
    assert not oracle_matches(np.array([np.nan, np.inf, 65504.0, 1.0, 0.0]), ref)[2]
    assert not oracle_matches(np.array([np.nan, np.inf, -np.inf, 1.03, np.nan]), ref)[3:].any()


# ---- B stored (N, K) and bfloat16 elements (oracle_gemm_relu_ex) -----------

def test_bf16_decode_matches_float32_top_half(oracle_mod):
    # a bfloat16 word is the top half of a binary32: decode by shifting
    known = {0x3F80: 1.0, 0xC040: -3.0, 0x7F7F: 3.3895313892515355e38, 0x0001: 2.0 ** -133,
             0x0080: 2.0 ** -126, 0x3EAB: 0.333984375, 0x7F80: float("inf")}
    for bits, val in known.items():
        assert oracle_mod.bf16_to_double(bits) == val, hex(bits)
    assert np.signbit(oracle_mod.bf16_to_double(0x8000))
    assert np.isnan(oracle_mod.bf16_to_double(0x7FC0))
    bits = np.arange(65536, dtype=np.uint16)
    ref = P.BF16.dec(bits)
    got = np.array([oracle_mod.bf16_to_double(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.signbit(got[finite]), np.signbit(ref[finite]))


def _ex_ref(oracle_mod, layout, dtype):
    """ref(A, B_kn, relu) through gemm_relu_ex; for "nk" the (K, N) operand of
    the pins is stored transposed, as an (N, K) row-major matrix."""
    def ref(A, B, relu):
        Bs = np.ascontiguousarray(B.T) if layout == "nk" else B
        return oracle_mod.gemm_relu_ex(A, Bs, relu, b_layout=layout, dtype=dtype)
    return ref


FMTS = {"f16": P.F16, "bf16": P.BF16}


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("pin", P.FMT_PINS, ids=lambda f: f.__name__)
def test_ex_oracle_passes_pin(oracle_mod, layout, dtype, pin):
    fails = pin(_ex_ref(oracle_mod, layout, dtype), fmt=FMTS[dtype])
    assert not fails, "\n".join(fails[:10])


@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_ex_f16_passes_golden(oracle_mod, layout):
    fails = P.pin_golden(_ex_ref(oracle_mod, layout, "f16"))
    assert not fails, "\n".join(fails[:10])


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_ex_layouts_agree_bit_for_bit(oracle_mod, dtype):
    rng = np.random.default_rng(21)
    fmt = FMTS[dtype]
    A = fmt.enc(rng.standard_normal((29, 75)))
    B = fmt.enc(rng.standard_normal((75, 43)))
    kn = oracle_mod.gemm_relu_ex(A, B, True, "kn", dtype)
    nk = oracle_mod.gemm_relu_ex(A, np.ascontiguousarray(B.T), True, "nk", dtype)
    assert np.array_equal(kn, nk)
    if dtype == "f16":
        assert np.array_equal(kn, oracle_mod.gemm_relu(A, B, True))
    rows = rng.integers(0, 29, 50)
    cols = rng.integers(0, 43, 50)
    ent = oracle_mod.gemm_relu_entries_ex(A, np.ascontiguousarray(B.T), rows, cols, True, "nk", dtype)
    assert np.array_equal(ent, kn[rows, cols])


def _ex_mutants(oracle_mod):
    ex = oracle_mod.gemm_relu_ex

    def bf16_read_as_f16(A, B, r):  # element type ignored
        return ex(A, np.ascontiguousarray(B.T), r, "nk", "f16")

    def nk_read_with_kn_strides(A, B, r):  # layout ignored: (N, K) storage walked as (K, N)
        Bs = np.ascontiguousarray(B.T)
        return ex(A, Bs.reshape(B.shape), r, "kn", "bf16")

    def bf16_exponent_off_by_one(A, B, r):
        return ex(A, np.ascontiguousarray(B.T), r, "nk", "bf16") * 2.0

    def nk_last_k_dropped(A, B, r):
        if A.shape[1] <= 1:
            return np.zeros((A.shape[0], B.shape[1]))
        Bs = np.ascontiguousarray(B.T[:, :-1])
        return ex(np.ascontiguousarray(A[:, :-1]), Bs, r, "nk", "bf16")

    return [bf16_read_as_f16, nk_read_with_kn_strides, bf16_exponent_off_by_one, nk_last_k_dropped]


@pytest.mark.parametrize("idx", range(4))
def test_fmt_pins_catch_planted_mistake_in_ex(oracle_mod, idx):
    mutant = _ex_mutants(oracle_mod)[idx]
    caught = [pin.__name__ for pin in P.FMT_PINS if pin(mutant, fmt=P.BF16)]
    assert caught, f"no pin caught the planted mistake {mutant.__name__}"
