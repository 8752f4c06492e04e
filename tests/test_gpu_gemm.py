"""Parity of the CUDA path with the CPU oracle, through the C ABI.

Every comparison is elementwise |c - ref| <= 1e-2 + 1e-2 |ref| (the GEMM+ReLU
listing's assert_close tolerance, oracle as the expected value), except the
integer cases, which must match bit for bit.  Every test compares every
output element; the oracle's full product of each of the five workloads is
computed once per module (a few seconds on all host cores) and reused by
the tests that run other schedules on the same inputs.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from tiled_dense_gemm_gb300 import binding
from tiled_dense_gemm_gb300.workloads import WORKLOADS, make_inputs, workload_inputs

pytestmark = pytest.mark.gpu

THREADS = max(1, len(os.sched_getaffinity(0)))
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tiled_dense_gemm_gb300 import build
    build.build()
    oracle.build()
    torch.cuda.set_device(DEV)
    yield
    torch.cuda.synchronize()


def gpu_run(A, B, relu=True, stream=None):
    a, b = A.to(DEV), B.to(DEV)
    c = binding.gemm_relu(a, b, apply_relu=relu, stream=stream)
    binding.check_device_error(stream)
    return c.cpu()


def assert_close(c16, ref, what=""):
    c = c16.double().numpy() if hasattr(c16, "double") else np.asarray(c16, np.float64)
    assert np.isfinite(c).all(), f"{what}: non-finite outputs"
    assert np.abs(ref).max(initial=0.0) < oracle.FP16_MAX, f"{what}: invalid workload (fp16 overflow)"
    ok = oracle.within_tolerance(c, ref)
    if not ok.all():
        bad = np.argwhere(~ok)
        i, j = bad[0]
        err = np.abs(c - ref)
        raise AssertionError(f"{what}: {len(bad)} of {ok.size} outside tolerance; first at "
                             f"({i},{j}) gpu={c[i, j]!r} ref={ref[i, j]!r}; max abs err {err.max():.3g}")


def assert_relu_sign(c16, relu):
    if relu:
        bits = c16.contiguous().view(torch.int16)
        assert (bits >= 0).all(), "ReLU output has a sign bit set (negative or -0)"


# ---------------------------------------------------------------- workloads

_FULL = {}


def workload_and_ref(name, relu):
    """Inputs of a workload and the oracle's full product (cached)."""
    key = (name, relu)
    if key not in _FULL:
        A, B = workload_inputs(WORKLOADS[name])
        _FULL[key] = (A, B, oracle.gemm_relu(A, B, relu, threads=THREADS))
    return _FULL[key]


@pytest.mark.parametrize("name", ["c1_256", "c2_1024", "c3_4096", "c4_skinny", "c5_ragged"])
def test_workload_full_parity(name):
    """Every output element of the five workloads (the ragged one with ReLU
    on and off), in the launch configuration the planner picks -- the one
    the benchmark times."""
    w = WORKLOADS[name]
    for relu in w.relu_modes:
        A, B, ref = workload_and_ref(name, relu)
        C = gpu_run(A, B, relu)
        assert_close(C, ref, f"{name} relu={relu}")
        assert_relu_sign(C, relu)


@pytest.mark.parametrize("force", ["pair:t2", "pair:t3", "pair:t4", "tiled256:t2", "tiled128:t3", "pair:dp",
                                   "pair:sk", "tiled128", "pair:npk", "tiled256:pk"])
def test_ragged_other_schedules_full(monkeypatch, force):
    """Other decompositions of the ragged workload -- full waves
    data-parallel with the leftover tiles split along K in 2-4 slots (the
    tail wave), data-parallel only, stream-K over all workers, one CTA per
    128 x 128 tile, without the in-launch copy of A to a 128-byte pitch
    (":npk"; the planner's plan makes it) and with it on one-CTA tiles
    (":pk") -- on every output element, ReLU on and off; the split-K and
    copy counters are left at zero for the next call."""
    monkeypatch.setenv("GEMM_RELU_FORCE_PATH", force)
    for relu in (True, False):
        A, B, ref = workload_and_ref("c5_ragged", relu)
        C = gpu_run(A, B, relu)
        assert_close(C, ref, f"c5_ragged {force} relu={relu}")
        assert_relu_sign(C, relu)


@pytest.mark.parametrize("force", ["pair:dp", "tiled256", "pair:t3"])
def test_square_4096_other_schedules_full(monkeypatch, force):
    """4096^3 without the split tail (data-parallel pairs), on one-CTA
    128 x 256 tiles, and with a 3-way tail split: every output element."""
    monkeypatch.setenv("GEMM_RELU_FORCE_PATH", force)
    A, B, ref = workload_and_ref("c3_4096", True)
    C = gpu_run(A, B, True)
    assert_close(C, ref, f"c3_4096 {force}")
    assert_relu_sign(C, True)


# ---------------------------------------------------------------- exactness

@pytest.mark.parametrize("shape", [(300, 264, 512), (16, 8192, 512), (128, 1024, 4096 // 8),
                                   (1024, 1024, 512), (129, 136, 136)])
def test_integer_inputs_bit_exact(shape):
    M, N, K = shape
    A, B = make_inputs(M, N, K, seed=99, dist_a="intgrid", scale_a=2, dist_b="intgrid", scale_b=2)
    for relu in (True, False):
        C = gpu_run(A, B, relu)
        ref = oracle.gemm_relu(A, B, relu, threads=THREADS)
        assert np.array_equal(C.double().numpy(), ref), f"{shape} relu={relu} not bit-exact"


def test_identity_B_gives_relu_A():
    A, _ = make_inputs(200, 8, 256, seed=5)
    I = torch.eye(256, dtype=torch.float16)
    C = gpu_run(A, I, True)
    assert torch.equal(C, torch.where(A > 0, A, torch.zeros_like(A)))


# ---------------------------------------------------------------- edges

EDGE_M = [1, 8, 127, 128, 129, 255, 257, 300]
EDGE_N = [8, 120, 128, 136, 256, 264]
EDGE_K = [8, 64, 72, 2056]
NAN16 = 0x7E00
CANARY = 0x5A5A
GUARD = 64


@pytest.mark.parametrize("K", EDGE_K)
@pytest.mark.parametrize("M", EDGE_M)
def test_edge_shapes_guarded(M, K):
    for N in EDGE_N:
        A, B = make_inputs(M, N, K, seed=M * 7919 + N * 31 + K, dist_a="uniform", dist_b="uniform")
        total = GUARD + M * N + GUARD
        buf = torch.full((total,), CANARY, dtype=torch.int16, device=DEV)
        buf[GUARD:GUARD + M * N] = NAN16
        c = buf[GUARD:GUARD + M * N].view(torch.float16).view(M, N)
        binding.gemm_relu(A.to(DEV), B.to(DEV), c, apply_relu=True)
        binding.check_device_error()
        host = buf.cpu()
        assert (host[:GUARD] == CANARY).all() and (host[GUARD + M * N:] == CANARY).all(), \
            f"write outside C for {M}x{N}x{K}"
        C = c.cpu()
        assert not torch.isnan(C).any(), f"unwritten outputs for {M}x{N}x{K}"
        ref = oracle.gemm_relu(A, B, True, threads=THREADS)
        assert_close(C, ref, f"{M}x{N}x{K}")
        assert_relu_sign(C, True)


@pytest.mark.parametrize("shape", [(128, 128, 65536), (16, 65536, 512), (20000, 8, 8),
                                   (130, 24, 4104), (64, 4096, 16384)])
def test_extreme_aspect_ratios(shape):
    M, N, K = shape
    A, B = make_inputs(M, N, K, seed=sum(shape), scale_a=1.0, scale_b=K ** -0.5)
    C = gpu_run(A, B, True)
    assert_close(C, oracle.gemm_relu(A, B, True, threads=THREADS), str(shape))


@pytest.mark.parametrize("shape", [(1 << 20, 4096, 64), (1 << 24, 8, 72)])
def test_outputs_beyond_32_bit_element_offsets(shape):
    """C with 2^32 elements (8 GiB; element offsets past 2^31) and a 2^24-row
    problem (131072 row tiles): every row block is written, checked on the
    first and last 128 rows and 64 random rows against the oracle, all
    columns, and on a canary element past the end of C."""
    M, N, K = shape
    A, B = make_inputs(M, N, K, seed=M % 997 + N + K, dist_a="uniform", dist_b="uniform")
    a, b = A.to(DEV), B.to(DEV)
    buf = torch.empty(M * N + 8, dtype=torch.float16, device=DEV)
    buf[M * N:] = 7.0
    c = buf[:M * N].view(M, N)
    binding.gemm_relu(a, b, c)
    binding.check_device_error()
    assert (buf[M * N:] == 7.0).all(), "write past the end of C"
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([np.arange(128), np.arange(M - 128, M), rng.integers(0, M, 64)]))
    idx = torch.from_numpy(rows).to(DEV)
    got = c.index_select(0, idx).cpu()
    ref = oracle.gemm_relu(A[torch.from_numpy(rows)].contiguous(), B, True, threads=THREADS)
    assert_close(got, ref, f"{shape} sampled rows")
    del buf, c
    torch.cuda.empty_cache()


def test_k_zero_writes_positive_zero():
    c = torch.full((37, 40), float("nan"), dtype=torch.float16, device=DEV)
    a = torch.empty((37, 0), dtype=torch.float16, device=DEV)
    b = torch.empty((0, 40), dtype=torch.float16, device=DEV)
    binding.gemm_relu(a, b, c)
    binding.check_device_error()
    assert (c.cpu().view(torch.int16) == 0).all()


def test_empty_output_is_a_noop():
    c = torch.full((0, 16), 1.0, dtype=torch.float16, device=DEV)
    binding.gemm_relu(torch.empty((0, 8), dtype=torch.float16, device=DEV),
                      torch.ones((8, 16), dtype=torch.float16, device=DEV), c)
    binding.check_device_error()


def test_misaligned_pointer_is_rejected():
    base = torch.zeros(64 * 64 + 1, dtype=torch.float16, device=DEV)
    a = base[1:].view(64, 64)
    b = torch.zeros(64, 64, dtype=torch.float16, device=DEV)
    with pytest.raises(binding.GemmReluError) as e:
        binding.gemm_relu(a, b)
    assert e.value.status == 2


# ---------------------------------------------------------------- behaviour

@pytest.mark.parametrize("name", ["c4_skinny", "c5_ragged", "c2_1024"])
def test_deterministic(name):
    A, B = workload_inputs(name)
    a, b = A.to(DEV), B.to(DEV)
    c1 = binding.gemm_relu(a, b)
    c2 = binding.gemm_relu(a, b)
    binding.check_device_error()
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))


def test_side_stream_and_back_to_back_calls():
    A, B = workload_inputs("c2_1024")
    a, b = A.to(DEV), B.to(DEV)
    s = torch.cuda.Stream(DEV)
    outs = []
    with torch.cuda.stream(s):
        for _ in range(3):
            outs.append(binding.gemm_relu(a, b, stream=s))
    s.synchronize()
    binding.check_device_error(s)
    ref = oracle.gemm_relu(A, B, True, threads=THREADS)
    for c in outs:
        assert_close(c.cpu(), ref, "side stream")


def test_cuda_graph_capture_and_replay():
    """After one call of each shape (which sizes the library's workspace),
    gemm_relu can be captured in a CUDA graph: replays on new inputs give
    the oracle's results (a split-tail plan with its fp32 workspace and
    counters, and a small-M cluster split-K plan)."""
    for name in ("c5_ragged", "c4_skinny"):
        A, B, ref = workload_and_ref(name, True)
        a, b = A.to(DEV), B.to(DEV)
        c = torch.empty(ref.shape, dtype=torch.float16, device=DEV)
        s = torch.cuda.Stream(DEV)
        with torch.cuda.stream(s):
            binding.gemm_relu(a, b, c, stream=s)  # warm-up outside the capture
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        a2, b2 = torch.zeros_like(a), torch.zeros_like(b)
        with torch.cuda.graph(g, stream=s):
            binding.gemm_relu(a2, b2, c, stream=torch.cuda.current_stream(DEV))
        a2.copy_(a)
        b2.copy_(b)
        c.fill_(float("nan"))
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        binding.check_device_error()
        assert_close(c.cpu(), ref, f"{name} graph replay")


def test_two_streams_with_split_workspaces_at_once():
    """Split-tail plans on two streams at the same time use separate
    workspaces and counters: both results are the oracle's."""
    A, B, ref = workload_and_ref("c3_4096", True)
    a, b = A.to(DEV), B.to(DEV)
    s1, s2 = torch.cuda.Stream(DEV), torch.cuda.Stream(DEV)
    c1 = torch.empty(ref.shape, dtype=torch.float16, device=DEV)
    c2 = torch.empty(ref.shape, dtype=torch.float16, device=DEV)
    for s, c in ((s1, c1), (s2, c2)):  # size each stream's workspace first
        binding.gemm_relu(a, b, c, stream=s)
    torch.cuda.synchronize()
    c1.fill_(float("nan"))
    c2.fill_(float("nan"))
    for _ in range(3):
        binding.gemm_relu(a, b, c1, stream=s1)
        binding.gemm_relu(a, b, c2, stream=s2)
    binding.check_device_error(s1)
    binding.check_device_error(s2)
    assert_close(c1.cpu(), ref, "stream 1")
    assert_close(c2.cpu(), ref, "stream 2")


def test_host_buffer_entry_point():
    A, B = workload_inputs("c4_skinny")
    C = binding.gemm_relu_host(A.pin_memory(), B.pin_memory())
    assert_close(C, oracle.gemm_relu(A, B, True, threads=THREADS), "host entry point")
    A2, B2 = workload_inputs("c1_256")
    C2 = binding.gemm_relu_host(A2, B2, apply_relu=False)  # pageable memory too
    assert_close(C2, oracle.gemm_relu(A2, B2, False, threads=THREADS), "host entry point pageable")


@pytest.mark.parametrize("name,relu,pinned", [("c3_4096", True, True), ("c5_ragged", False, True),
                                              ("c5_ragged", True, False)])
def test_host_buffer_entry_point_row_blocks(name, relu, pinned):
    """Large problems go through the host-buffer entry point in row blocks
    whose copies in, GEMMs and copies out overlap on three streams (4096^3:
    8 blocks of 512 rows; 3000 rows: 5 blocks of 512 and one of 440):
    every element, twice in a row, pinned and pageable host memory."""
    A, B, ref = workload_and_ref(name, relu)
    a, b = (A.pin_memory(), B.pin_memory()) if pinned else (A, B)
    for _ in range(2):
        C = torch.full(ref.shape, float("nan"), dtype=torch.float16)
        C = C.pin_memory() if pinned else C
        binding.gemm_relu_host(a, b, C, apply_relu=relu)
        assert_close(C, ref, f"{name} host row blocks relu={relu} pinned={pinned}")
        assert_relu_sign(C, relu)


def test_stream_k_counters_are_left_zero():
    """Split tiles reset their arrival counters, so repeated calls stay correct."""
    A, B, ref = workload_and_ref("c4_skinny", True)
    a, b = A.to(DEV), B.to(DEV)
    for _ in range(5):
        c = binding.gemm_relu(a, b)
    binding.check_device_error()
    assert_close(c.cpu(), ref, "after repeats")


# ---------------------------------------------------------------- every kernel shape

FORCED_SHAPES = [(1, 8, 8), (129, 136, 72), (300, 264, 2056), (513, 520, 1000), (1024, 1024, 1024),
                 (257, 1032, 4104), (96, 2048, 3000), (48, 6144, 2048), (8, 4864, 1024),
                 (16, 1000, 1024), (100, 1000, 1032)]


@pytest.mark.parametrize("force", ["tiled256", "tiled128", "pair", "tiled256:dp", "tiled128:dp",
                                   "pair:dp", "swap", "swap:dp", "swap:s7", "tiled128:s3", "pair:s5",
                                   "tiled128:c2", "tiled256:c2", "swap:c2", "swap:sk", "tiled128:sk",
                                   "tiled64", "tiled64:s3", "tiled64:c2", "tiled128:s2", "pair:s2",
                                   "pair:s4", "tiled256:s2", "tiled64:s2", "tiled128:no3d", "pair:no3d",
                                   "swap:no3d", "tiled256:no3d", "pair:t2", "pair:pk", "tiled128:pk",
                                   "pair:s3:pk", "tiled64:c2:pk"])
def test_each_kernel_shape_parity(monkeypatch, force):
    """Every kernel shape (one CTA per 128 x 256 / 128 x 128 / 128 x 64
    tile, 256 x 256 CTA pairs, swapped operands), with and without stream-K,
    split-K and cluster split-K, on ragged shapes."""
    monkeypatch.setenv("GEMM_RELU_FORCE_PATH", force)
    for M, N, K in FORCED_SHAPES:
        A, B = make_inputs(M, N, K, seed=M + N + K, dist_a="uniform", dist_b="uniform")
        for relu in (True, False):
            C = gpu_run(A, B, relu)
            ref = oracle.gemm_relu(A, B, relu, threads=THREADS)
            assert_close(C, ref, f"{force} {M}x{N}x{K} relu={relu}")
            assert_relu_sign(C, relu)
