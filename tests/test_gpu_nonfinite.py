"""Parity for inputs that hold NaN and infinities, through the C ABI.

The pages say nothing about non-finite inputs; the reading taken is IEEE
754 arithmetic throughout: a NaN operand, or an infinity times zero, makes
that term NaN; infinite terms of both signs sum to NaN; otherwise an
infinite term makes the sum that infinity.  ReLU (x > 0 ? x : +0) turns NaN
and -inf into +0 and keeps +inf.  The oracle follows these rules (pinned by
``oracle_pins.pin_ieee_specials``), and the kernels must agree with it
element by element: NaN where it has NaN, the same infinity where it has
one, and the usual tolerance elsewhere.  The infinities sit at both ends
of K so that split-K and stream-K schedules add them up across their
partial sums.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from tiled_dense_gemm_gb300 import binding
from tiled_dense_gemm_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
THREADS = max(1, len(os.sched_getaffinity(0)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tiled_dense_gemm_gb300 import build
    build.build()
    oracle.build()
    torch.cuda.set_device(DEV)


def planted(M, N, K, seed, dtype=torch.float16):
    """Uniform inputs with NaN and infinities planted in A's rows 5, 7 and 9
    and B's columns 11 and 13, and zeros beside them (inf x 0)."""
    A, B = make_inputs(M, N, K, seed=seed, dist_a="uniform", dist_b="uniform")
    A = A.double()
    B = B.double()
    inf, nan = float("inf"), float("nan")
    A[5, K // 3] = nan
    A[7, 3] = inf
    B[3, ::5] = 0.0
    A[9, 10] = inf
    A[9, K - 20] = -inf
    B[K // 2, 11] = nan
    B[K - 1, 13] = -inf
    A[::4, K - 1] = 0.0
    return A.to(dtype), B.to(dtype)


def check(C, ref, relu, what):
    got = C.double().cpu().numpy()
    ok = oracle.matches_ieee(got, ref)
    if not ok.all():
        i, j = np.argwhere(~ok)[0]
        raise AssertionError(f"{what}: {int((~ok).sum())} mismatches, first [{i},{j}] got {got[i, j]} "
                             f"expected {ref[i, j]}")
    if relu:
        assert not (np.signbit(got) & (got == 0)).any(), f"{what}: -0 after ReLU"
        assert not np.isnan(got).any(), f"{what}: NaN after ReLU"
    # the planted cases are all there
    assert np.isnan(ref).any() or relu
    assert np.isinf(ref).any()


PATHS = [None, "tiled64", "tiled128", "tiled256", "pair", "swap", "tiled128:s3", "tiled64:s3",
         "pair:s2", "pair:s4", "tiled128:c2", "tiled64:c2", "swap:c2", "swap:sk", "tiled128:sk",
         "pair:t2", "pair:pk"]
SHAPES = [(300, 264, 2056), (16, 1000, 1024)]


@pytest.mark.parametrize("force", PATHS, ids=lambda f: f or "auto")
def test_nan_and_infinities_follow_ieee(monkeypatch, force):
    if force:
        monkeypatch.setenv("GEMM_RELU_FORCE_PATH", force)
    for M, N, K in SHAPES:
        A, B = planted(M, N, K, seed=M + N + K)
        a, b = A.to(DEV), B.to(DEV)
        for relu in (True, False):
            C = binding.gemm_relu(a, b, apply_relu=relu)
            binding.check_device_error()
            ref = oracle.gemm_relu(A, B, relu, threads=THREADS)
            check(C, ref, relu, f"{force} {M}x{N}x{K} relu={relu}")


@pytest.mark.parametrize("layout,dtype", [("nk", "f16"), ("kn", "bf16"), ("nk", "bf16")])
def test_nan_and_infinities_ex(layout, dtype):
    M, N, K = 300, 264, 2056
    A, B = planted(M, N, K, seed=7, dtype=torch.bfloat16 if dtype == "bf16" else torch.float16)
    Bs = B.t().contiguous() if layout == "nk" else B
    for relu in (True, False):
        C = binding.gemm_relu_ex(A.to(DEV), Bs.to(DEV), apply_relu=relu, b_layout=layout)
        binding.check_device_error()
        ref = oracle.gemm_relu_ex(A, Bs, relu, b_layout=layout, dtype=dtype, threads=THREADS)
        check(C, ref, relu, f"{layout} {dtype} relu={relu}")
