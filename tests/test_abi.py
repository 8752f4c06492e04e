"""The C ABI without a GPU: symbols, status strings, argument checks.

No compute call is made here; the calls below are rejected by the host-side
checks before any CUDA work (or, on a machine without a GB300, by the device
check).
"""
import ctypes
import subprocess

import pytest
import torch

from tiled_dense_gemm_gb300 import build as B


def test_library_exports_every_declared_symbol(gemm_lib):
    names = gemm_lib.declared_functions()
    assert {"gemm_relu", "gemm_relu_host", "gemm_relu_check_device_error",
            "gemm_relu_status_string", "gemm_relu_shutdown", "gemm_relu_plan",
            "gemm_relu_plan_work_item"} <= set(names)
    L = gemm_lib.lib()
    for n in names:
        assert hasattr(L, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in names if n not in exported]
    assert not missing, missing


def test_library_has_no_cpu_gemm_and_no_oracle_link(gemm_lib):
    out = subprocess.run(["nm", "-D", B.LIB_PATH], capture_output=True, text=True, check=True).stdout
    assert "oracle" not in out
    ldd = subprocess.run(["ldd", B.LIB_PATH], capture_output=True, text=True).stdout
    assert "liboracle" not in ldd and "libcublas" not in ldd


def test_status_strings(gemm_lib):
    for code, name in gemm_lib.STATUS_NAMES.items():
        assert gemm_lib.status_string(code) == name
    assert gemm_lib.status_string(99) == "GEMM_ERR_UNKNOWN"


def _call(L, A, Bp, C, M, N, K, relu=1):
    return L.gemm_relu(A, Bp, C, M, N, K, relu, None)


def test_argument_checks_before_any_cuda_call(gemm_lib):
    L = gemm_lib.lib()
    good = 4096  # a 16-byte aligned fake address: never dereferenced on these paths
    assert _call(L, good, good, good, -1, 8, 8) == 1
    assert _call(L, good, good, good, 8, -1, 8) == 1
    assert _call(L, good, good, good, 8, 8, -1) == 1
    assert _call(L, good, good, good, 1 << 31, 8, 8) == 1
    assert _call(L, None, good, good, 8, 8, 8) == 1
    assert _call(L, good, None, good, 8, 8, 8) == 1
    assert _call(L, good, good, None, 8, 8, 8) == 1
    assert _call(L, good, good, good, 8, 8, 12) == 2   # K % 8
    assert _call(L, good, good, good, 8, 12, 8) == 2   # N % 8
    assert _call(L, good + 2, good, good, 8, 8, 8) == 2
    assert _call(L, good, good + 8, good, 8, 8, 8) == 2
    assert _call(L, good, good, good + 4, 8, 8, 8) == 2
    # empty output: nothing to do, no pointer needed
    assert _call(L, None, None, None, 0, 8, 8) == 0
    assert _call(L, None, None, None, 8, 0, 8) == 0
    # host-buffer entry point: same checks, alignment of host pointers waived
    assert L.gemm_relu_host(None, good, good, 8, 8, 8, 1, None) == 1
    assert L.gemm_relu_host(good, good, good, 8, 8, 12, 1, None) == 2


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks behaviour without a GPU")
def test_no_device_is_reported_not_faked(gemm_lib):
    L = gemm_lib.lib()
    good = 4096
    assert _call(L, good, good, good, 8, 8, 8) == 3  # GEMM_ERR_UNSUPPORTED_DEVICE
    assert L.gemm_relu_host(good, good, good, 8, 8, 8, 1, None) == 3


def test_python_wrapper_rejects_bad_tensors(gemm_lib):
    a = torch.zeros(4, 8, dtype=torch.float16)
    b = torch.zeros(8, 8, dtype=torch.float16)
    with pytest.raises(ValueError):
        gemm_lib.gemm_relu(a, b)  # CPU tensors are not accepted by the device entry point
    with pytest.raises(TypeError):
        gemm_lib.gemm_relu(a.float(), b)
    with pytest.raises(ValueError):
        gemm_lib.gemm_relu(a, torch.zeros(4, 8, dtype=torch.float16))


def test_ex_entry_point_checks(gemm_lib):
    L = gemm_lib.lib()
    good = 4096
    ex = lambda *a: L.gemm_relu_ex(*a, None)  # noqa: E731
    # unknown layout / element type
    assert ex(good, good, good, 8, 8, 8, 1, 2, 0) == 1
    assert ex(good, good, good, 8, 8, 8, 1, -1, 0) == 1
    assert ex(good, good, good, 8, 8, 8, 1, 0, 2) == 1
    # gemm_relu's own checks apply to every layout and type
    for layout in (0, 1):
        for dtype in (0, 1):
            assert ex(good, good, good, -1, 8, 8, 1, layout, dtype) == 1
            assert ex(good, good, good, 8, 8, 12, 1, layout, dtype) == 2
            assert ex(good, good, good, 8, 12, 8, 1, layout, dtype) == 2
            assert ex(good, good + 8, good, 8, 8, 8, 1, layout, dtype) == 2
            assert ex(None, None, None, 0, 8, 8, 1, layout, dtype) == 0
            if not torch.cuda.is_available():
                assert ex(good, good, good, 8, 8, 8, 1, layout, dtype) == 3


def test_ex_python_wrapper_rejects_bad_tensors(gemm_lib):
    a = torch.zeros(4, 8, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        gemm_lib.gemm_relu_ex(a, torch.zeros(8, 8, dtype=torch.float16))  # mixed types
    with pytest.raises(ValueError):
        gemm_lib.gemm_relu_ex(a, torch.zeros(8, 8, dtype=torch.bfloat16), b_layout="tn")
    with pytest.raises(ValueError):
        gemm_lib.gemm_relu_ex(a, torch.zeros(6, 4, dtype=torch.bfloat16), b_layout="nk")  # K differs
    with pytest.raises(ValueError):
        gemm_lib.gemm_relu_ex(a, torch.zeros(16, 8, dtype=torch.bfloat16), b_layout="nk")  # CPU
