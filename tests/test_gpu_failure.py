"""A bounded device wait that runs out, on the GPU, without a fault.

Every wait of the kernels is bounded; when one runs out the CTA records an
error word, stops its other roles, lets its copies and MMAs in flight land,
frees its tensor memory and returns, so the context stays usable.  The
library's test hook (GEMM_RELU_TEST_DROP_KB=k) makes every CTA leave the
copies of k-block k of its first work item undone -- the stage is armed
for bytes that never arrive, a flag nothing sets -- and limits every wait
to 1 ms.  Each case checks that the host then reports GEMM_ERR_TIMEOUT
once, and that the next call on the same stream, with the hook removed,
matches the oracle on every element (the split-K counters and error word
were reset).
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
GEMM_ERR_INVALID_ARG = 1
GEMM_ERR_TIMEOUT = 6


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tiled_dense_gemm_gb300 import build
    build.build()
    oracle.build()
    torch.cuda.set_device(DEV)


# (force, shape, dropped k-block): one CTA per 128 x 64 tile, data-parallel;
# one CTA per 128 x 128 tile with every tile split in 3 K ranges (global
# partials, tickets and ready flags); swapped operands for small M with
# stream-K over the SMs; one CTA per 128 x 256 tile, several tiles per CTA.
CASES = [("tiled64:dp", (128, 64, 256), 0),
         ("tiled128:s3", (256, 512, 2048), 1),
         ("swap:sk", (16, 1024, 2048), 1),
         ("tiled256:dp", (2048, 8192, 512), 3)]


@pytest.mark.parametrize("force,shape,kb", CASES)
def test_timed_out_wait_is_reported_and_the_next_call_is_correct(monkeypatch, force, shape, kb):
    M, N, K = shape
    A, B = make_inputs(M, N, K, seed=M + N + K, dist_a="uniform", dist_b="uniform")
    a, b = A.to(DEV), B.to(DEV)
    ref = oracle.gemm_relu(A, B, True, threads=THREADS)
    monkeypatch.setenv("GEMM_RELU_FORCE_PATH", force)
    monkeypatch.setenv("GEMM_RELU_TEST_DROP_KB", str(kb))
    c = torch.zeros((M, N), dtype=torch.float16, device=DEV)
    binding.gemm_relu(a, b, c)  # enqueued
    with pytest.raises(binding.GemmReluError) as e:
        binding.check_device_error()
    assert e.value.status == GEMM_ERR_TIMEOUT
    binding.check_device_error()  # reported once, then cleared
    monkeypatch.delenv("GEMM_RELU_TEST_DROP_KB")
    for _ in range(2):
        c = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
        binding.gemm_relu(a, b, c)
        binding.check_device_error()
        got = c.cpu().double().numpy()
        assert np.isfinite(got).all()
        assert oracle.within_tolerance(got, ref).all(), f"{force} {shape}: wrong result after the timeout"


def test_the_hook_is_refused_where_it_does_not_apply(monkeypatch):
    """Plans that run in clusters (CTA pairs, cluster split-K) and k-blocks
    past the end are refused on the host, before any launch."""
    a = torch.zeros(512, 1024, dtype=torch.float16, device=DEV)
    b = torch.zeros(1024, 512, dtype=torch.float16, device=DEV)
    monkeypatch.setenv("GEMM_RELU_TEST_DROP_KB", "0")
    monkeypatch.setenv("GEMM_RELU_FORCE_PATH", "pair")
    with pytest.raises(binding.GemmReluError) as e:
        binding.gemm_relu(a, b)
    assert e.value.status == GEMM_ERR_INVALID_ARG
    monkeypatch.setenv("GEMM_RELU_FORCE_PATH", "tiled128:dp")
    monkeypatch.setenv("GEMM_RELU_TEST_DROP_KB", "8")  # K = 1024: 8 k-blocks of 128
    with pytest.raises(binding.GemmReluError) as e:
        binding.gemm_relu(a, b)
    assert e.value.status == GEMM_ERR_INVALID_ARG
    binding.check_device_error()
