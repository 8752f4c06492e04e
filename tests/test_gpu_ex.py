"""Parity of gemm_relu_ex -- B stored (N, K), and bfloat16 elements -- with
the CPU oracle, through the C ABI.

Same rule as every parity test here: elementwise |c - ref| <= 1e-2 +
1e-2 |ref| against the oracle's unrounded binary64 result (the rounding of
C to bfloat16, relative 2^-9, sits inside it), bit-exact for integer inputs
whose results are exact in the element type.  Every kernel variant is forced
on ragged shapes; the skinny and square workloads run at full size.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from tiled_dense_gemm_gb300 import binding
from tiled_dense_gemm_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

THREADS = max(1, len(os.sched_getaffinity(0)))
DEV = torch.device("cuda", 0)
TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16}
VARIANTS = [("nk", "f16"), ("kn", "bf16"), ("nk", "bf16")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tiled_dense_gemm_gb300 import build
    build.build()
    oracle.build()
    torch.cuda.set_device(DEV)
    yield
    torch.cuda.synchronize()


def gpu_ex(A, B, layout, relu=True):
    c = binding.gemm_relu_ex(A.to(DEV), B.to(DEV), apply_relu=relu, b_layout=layout)
    binding.check_device_error()
    return c.cpu()


def assert_close(c16, ref, what):
    c = c16.double().numpy()
    assert np.isfinite(c).all(), f"{what}: non-finite outputs"
    ok = oracle.within_tolerance(c, ref)
    if not ok.all():
        bad = np.argwhere(~ok)
        i, j = bad[0]
        raise AssertionError(f"{what}: {len(bad)} of {ok.size} outside tolerance; first at ({i},{j}) "
                             f"gpu={c[i, j]!r} ref={ref[i, j]!r}")


def assert_relu_sign(c16, relu, what):
    if relu:
        assert (c16.contiguous().view(torch.int16) >= 0).all(), f"{what}: sign bit set after ReLU"


_REF = {}


def inputs_and_ref(shape, layout, dtype, relu, seed=31):
    key = (shape, layout, dtype, relu, seed)
    if key not in _REF:
        M, N, K = shape
        A, B = make_inputs(M, N, K, seed, "uniform", 1.0, "uniform", 1.0,
                           dtype=TORCH_DTYPE[dtype], b_layout=layout)
        _REF[key] = (A, B, oracle.gemm_relu_ex(A, B, relu, layout, dtype, threads=THREADS))
    return _REF[key]


SHAPES = [(1, 8, 8), (129, 136, 72), (300, 264, 2056), (513, 520, 1000), (48, 6144, 2048),
          (8, 4864, 1024), (16, 1000, 1024)]
FORCES = ["", "tiled256", "tiled128", "pair", "tiled256:dp", "swap", "swap:dp", "swap:c2", "tiled128:c2",
          "swap:s7", "tiled128:s3", "pair:s5", "swap:sk", "tiled64", "tiled64:c2", "tiled128:no3d", "pair:no3d",
          "swap:no3d", "tiled256:c2", "pair:t2", "pair:pk", "tiled128:pk"]


@pytest.mark.parametrize("force", FORCES)
@pytest.mark.parametrize("layout,dtype", VARIANTS)
def test_ex_each_kernel_shape_parity(monkeypatch, layout, dtype, force):
    """Every kernel variant (forced; "" is the planner's own choice) on
    ragged shapes, for each B layout / element type, ReLU on and off."""
    if force:
        monkeypatch.setenv("GEMM_RELU_FORCE_PATH", force)
    else:
        monkeypatch.delenv("GEMM_RELU_FORCE_PATH", raising=False)
    for shape in SHAPES:
        for relu in (True, False):
            A, B, ref = inputs_and_ref(shape, layout, dtype, relu)
            what = f"{shape} {layout}/{dtype} force={force!r} relu={relu}"
            c = gpu_ex(A, B, layout, relu)
            assert c.dtype == TORCH_DTYPE[dtype]
            assert_close(c, ref, what)
            assert_relu_sign(c, relu, what)


@pytest.mark.parametrize("layout,dtype", VARIANTS)
def test_ex_skinny_full_parity(layout, dtype):
    w = WORKLOADS["c4_skinny"]
    A, B = make_inputs(w.M, w.N, w.K, w.seed, w.dist_a, w.scale_a, w.dist_b, w.scale_b,
                       dtype=TORCH_DTYPE[dtype], b_layout=layout)
    ref = oracle.gemm_relu_ex(A, B, True, layout, dtype, threads=THREADS)
    c = gpu_ex(A, B, layout)
    assert_close(c, ref, f"c4_skinny {layout}/{dtype}")
    assert_relu_sign(c, True, "c4_skinny")


@pytest.mark.parametrize("name", ["c3_4096", "c5_ragged"])
@pytest.mark.parametrize("layout,dtype", VARIANTS)
def test_ex_workload_full_parity(layout, dtype, name):
    """4096^3 and the ragged workload (ReLU on and off) in each B layout /
    element type: every output element against the oracle."""
    w = WORKLOADS[name]
    A, B = make_inputs(w.M, w.N, w.K, w.seed, w.dist_a, w.scale_a, w.dist_b, w.scale_b,
                       dtype=TORCH_DTYPE[dtype], b_layout=layout)
    for relu in w.relu_modes:
        ref = oracle.gemm_relu_ex(A, B, relu, layout, dtype, threads=THREADS)
        c = gpu_ex(A, B, layout, relu)
        assert_close(c, ref, f"{name} {layout}/{dtype} relu={relu}")
        assert_relu_sign(c, relu, name)


@pytest.mark.parametrize("layout,dtype", VARIANTS)
@pytest.mark.parametrize("shape", [(300, 264, 64), (16, 8192, 64), (1024, 1024, 64)])
def test_ex_integer_inputs_bit_exact(layout, dtype, shape):
    """Integers in [-2, 2] with K = 64: |C| <= 256, exact in both element
    types, so the GPU result must equal the oracle's bit for bit."""
    M, N, K = shape
    A, B = make_inputs(M, N, K, 9, "intgrid", 2, "intgrid", 2, dtype=TORCH_DTYPE[dtype], b_layout=layout)
    ref = oracle.gemm_relu_ex(A, B, True, layout, dtype, threads=THREADS)
    c = gpu_ex(A, B, layout).double().numpy()
    assert np.array_equal(c, ref), f"{int((c != ref).sum())} entries differ"


def test_ex_kn_f16_is_gemm_relu():
    M, N, K = 300, 264, 2056
    A, B = make_inputs(M, N, K, 5)
    a, b = A.to(DEV), B.to(DEV)
    c1 = binding.gemm_relu(a, b)
    c2 = binding.gemm_relu_ex(a, b, b_layout="kn")
    binding.check_device_error()
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_ex_layouts_agree(dtype):
    """The same product with B given either way round."""
    M, N, K = 513, 520, 1000
    A, B = make_inputs(M, N, K, 12, dtype=TORCH_DTYPE[dtype])
    c_kn = gpu_ex(A, B, "kn").double().numpy()
    c_nk = gpu_ex(A, B.t().contiguous(), "nk").double().numpy()
    ok = oracle.within_tolerance(c_nk, c_kn, rtol=1e-2, atol=1e-2)
    assert ok.all()
