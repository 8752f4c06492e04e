"""gemm_relu_noalloc checked against the CPU oracle, through the C ABI.

gemm_relu_noalloc serves callers that must not allocate device memory: a
loop that may never stall on cudaMalloc / cudaFree (which can synchronize
the device), or a process whose device memory is all reserved up front by
its own allocator.  It keeps the split-K scratch of the small-M kernel in a
fixed device array instead of a workspace the library allocates.  Each case
runs it twice in a row on different inputs and compares both outputs with
the oracle to the tolerance every parity test here uses,
|c - ref| <= 1e-2 + 1e-2 |ref|.  Further tests check that a call allocates
no device memory, that its error word reports a timed-out device wait
through gemm_relu_noalloc_check_device_error, and that it refuses what its
array cannot hold.

This file is named so that pytest collects it last.
"""
import ctypes
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
GEMM_ERR_TIMEOUT = 6
GEMM_ERR_TOO_LARGE = 8


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tiled_dense_gemm_gb300 import build
    build.build()
    oracle.build()
    torch.cuda.set_device(DEV)


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)


def call_noalloc(a, b, c, relu=True):
    M, K = a.shape
    N = b.shape[1]
    return binding.lib().gemm_relu_noalloc(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K,
                                           int(relu), _stream())


def check_noalloc():
    return binding.lib().gemm_relu_noalloc_check_device_error(_stream())


def assert_close(got, ref, what):
    g = got.double().cpu().numpy()
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    ok = oracle.within_tolerance(g, ref)
    assert ok.all(), f"{what}: {int((~ok).sum())} of {ok.size} outputs outside tolerance of the oracle"


@pytest.mark.parametrize("shape", [(16, 8192, 8192), (100, 1000, 2056), (1, 8, 8), (64, 4096, 1024)])
def test_noalloc_matches_the_oracle_on_two_calls_in_a_row(shape):
    M, N, K = shape
    for call, seed in enumerate((11, 12)):
        A, B = make_inputs(M, N, K, seed=seed + M, scale_b=K ** -0.5)
        a, b = A.to(DEV), B.to(DEV)
        for relu in (True, False):
            ref = oracle.gemm_relu(A, B, relu, threads=THREADS)
            c = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
            assert call_noalloc(a, b, c, relu) == binding.GEMM_OK
            assert check_noalloc() == binding.GEMM_OK
            assert_close(c, ref, f"{shape} call {call + 1} relu={relu}")


def test_noalloc_allocates_no_device_memory():
    """Free device memory is unchanged across a call on a shape no earlier
    call of either entry point has used (after one call that has loaded the
    library's code on the device)."""
    warm_a = torch.zeros(8, 64, dtype=torch.float16, device=DEV)
    warm_b = torch.zeros(64, 64, dtype=torch.float16, device=DEV)
    warm_c = torch.zeros(8, 64, dtype=torch.float16, device=DEV)
    assert call_noalloc(warm_a, warm_b, warm_c) == binding.GEMM_OK
    assert check_noalloc() == binding.GEMM_OK
    M, N, K = 24, 3064, 4104
    A, B = make_inputs(M, N, K, seed=77, scale_b=K ** -0.5)
    a, b = A.to(DEV), B.to(DEV)
    c = torch.empty((M, N), dtype=torch.float16, device=DEV)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info(DEV)[0]
    assert call_noalloc(a, b, c) == binding.GEMM_OK
    assert check_noalloc() == binding.GEMM_OK
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info(DEV)[0]
    assert free_after == free_before, f"device memory changed by {free_before - free_after} bytes"
    assert_close(c, oracle.gemm_relu(A, B, True, threads=THREADS), "fresh shape")


def test_noalloc_reports_a_timed_out_wait(monkeypatch):
    """With the test hook set, every CTA leaves one k-block uncopied and the
    device waits are limited to 1 ms: the wait runs out, the array's error
    word records it, the check reports GEMM_ERR_TIMEOUT once and clears it,
    and the next call on the stream is correct."""
    M, N, K = 16, 1024, 2048
    A, B = make_inputs(M, N, K, seed=5, scale_b=K ** -0.5)
    a, b = A.to(DEV), B.to(DEV)
    ref = oracle.gemm_relu(A, B, True, threads=THREADS)
    c = torch.zeros((M, N), dtype=torch.float16, device=DEV)
    monkeypatch.setenv("GEMM_RELU_TEST_DROP_KB", "1")
    assert call_noalloc(a, b, c) == binding.GEMM_OK
    assert check_noalloc() == GEMM_ERR_TIMEOUT
    assert check_noalloc() == binding.GEMM_OK  # cleared by the first check
    monkeypatch.delenv("GEMM_RELU_TEST_DROP_KB")
    for _ in range(2):
        c = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
        assert call_noalloc(a, b, c) == binding.GEMM_OK
        assert check_noalloc() == binding.GEMM_OK
        assert_close(c, ref, "after the timed-out call")


def test_noalloc_rejects_what_its_scratch_cannot_hold():
    a = torch.zeros(129, 64, dtype=torch.float16, device=DEV)
    b = torch.zeros(64, 64, dtype=torch.float16, device=DEV)
    c = torch.zeros(129, 64, dtype=torch.float16, device=DEV)
    assert call_noalloc(a, b, c) == GEMM_ERR_TOO_LARGE  # M > 128
    assert binding.status_string(GEMM_ERR_TOO_LARGE) == "GEMM_ERR_TOO_LARGE"
    # M = 128, N = 2048, K = 16384: its split-K partials need 11 MiB, more
    # than the array holds
    a2 = torch.zeros(128, 16384, dtype=torch.float16, device=DEV)
    b2 = torch.zeros(16384, 2048, dtype=torch.float16, device=DEV)
    c2 = torch.zeros(128, 2048, dtype=torch.float16, device=DEV)
    assert call_noalloc(a2, b2, c2) == GEMM_ERR_TOO_LARGE
    base = torch.zeros(16 * 64 + 1, dtype=torch.float16, device=DEV)
    assert call_noalloc(base[1:].view(16, 64), b, c[:16]) == 2  # misaligned A
    torch.cuda.synchronize()
