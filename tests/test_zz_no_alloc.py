"""gemm_relu_noalloc checked against gemm_relu, through the C ABI.

gemm_relu_noalloc is for callers that must not allocate device memory
(cudaMalloc / cudaFree can synchronize the device, or all device memory may
already be reserved by another allocator).  It keeps the split-K scratch of
the small-M kernel in a fixed device array instead of a workspace the
library allocates.  Each case runs it twice in a row and compares both
outputs with the regular entry point's output on the same inputs, to the
tolerance every parity test here uses: |c - ref| <= 1e-2 + 1e-2 |ref|.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from tiled_dense_gemm_gb300 import binding
from tiled_dense_gemm_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tiled_dense_gemm_gb300 import build
    build.build()
    torch.cuda.set_device(DEV)


def call_noalloc(a, b, c, relu=True):
    M, K = a.shape
    N = b.shape[1]
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    return binding.lib().gemm_relu_noalloc(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K,
                                           int(relu), stream)


def assert_close(got, ref, what):
    g = got.double().cpu().numpy()
    r = ref.double().cpu().numpy()
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    ok = oracle.within_tolerance(g, r)
    assert ok.all(), f"{what}: {int((~ok).sum())} of {ok.size} outputs differ from gemm_relu"


@pytest.mark.parametrize("shape", [(16, 8192, 8192), (100, 1000, 2056), (1, 8, 8), (64, 4096, 1024)])
def test_noalloc_matches_gemm_relu_on_two_calls_in_a_row(shape):
    M, N, K = shape
    for call, seed in enumerate((11, 12)):
        A, B = make_inputs(M, N, K, seed=seed + M, scale_b=K ** -0.5)
        a, b = A.to(DEV), B.to(DEV)
        for relu in (True, False):
            ref = binding.gemm_relu(a, b, apply_relu=relu)
            c = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
            assert call_noalloc(a, b, c, relu) == binding.GEMM_OK
            torch.cuda.synchronize()
            assert_close(c, ref, f"{shape} call {call + 1} relu={relu}")


def test_noalloc_rejects_what_its_scratch_cannot_hold():
    a = torch.zeros(129, 64, dtype=torch.float16, device=DEV)
    b = torch.zeros(64, 64, dtype=torch.float16, device=DEV)
    c = torch.zeros(129, 64, dtype=torch.float16, device=DEV)
    assert call_noalloc(a, b, c) == 8  # GEMM_ERR_TOO_LARGE: M > 128
    assert binding.status_string(8) == "GEMM_ERR_TOO_LARGE"
    # M = 128, N = 2048, K = 16384: its split-K partials need 11 MiB, more
    # than the array holds
    a2 = torch.zeros(128, 16384, dtype=torch.float16, device=DEV)
    b2 = torch.zeros(16384, 2048, dtype=torch.float16, device=DEV)
    c2 = torch.zeros(128, 2048, dtype=torch.float16, device=DEV)
    assert call_noalloc(a2, b2, c2) == 8
    base = torch.zeros(16 * 64 + 1, dtype=torch.float16, device=DEV)
    assert call_noalloc(base[1:].view(16, 64), b, c[:16]) == 2  # misaligned A
    torch.cuda.synchronize()
