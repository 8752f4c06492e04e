"""CPU oracle for C = ReLU(A . B) -- TEST INFRASTRUCTURE, not the product.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and
has no CPU fallback; this package never imports the CUDA library either.

The arithmetic lives in ``oracle_gemm_relu.c`` (plain C, binary64
accumulation, i-k-j loop, its own binary16 decoder).  This module only
compiles that file with gcc and marshals numpy arrays to it.

Definition followed: the GEMM+ReLU worked example of "Writing
High-Performance Kernels in TileLang" (atlascloud.ai guide, GEMM section,
listing ``matmul_relu_kernel``): clear the accumulator, accumulate A.B over
all of K, apply max(x, 0), write C.  Checked against: ``torch.relu(a @ b)``
with rtol = atol = 1e-2 (same listing's closing assert).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_gemm_relu.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lock = threading.Lock()
_lib = None

# fp16 overflow threshold: an exact result beyond this would not survive the
# cast to binary16, so a workload that reaches it is invalid for parity.
FP16_MAX = 65504.0


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no CUDA involved).  Returns the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp",
           "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, dp, vp = ctypes.c_int64, ctypes.POINTER(ctypes.c_double), ctypes.c_void_p
        lib.oracle_half_to_double.restype = ctypes.c_double
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_gemm_relu.restype = ctypes.c_int
        lib.oracle_gemm_relu.argtypes = [vp, vp, vp, i64, i64, i64, ctypes.c_int,
                                         vp, vp, ctypes.c_int]
        lib.oracle_gemm_relu_entries.restype = ctypes.c_int
        lib.oracle_gemm_relu_entries.argtypes = [vp, vp, i64, i64, i64, ctypes.c_int,
                                                 vp, vp, i64, vp, ctypes.c_int]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_gemm_relu_ex.restype = ctypes.c_int
        lib.oracle_gemm_relu_ex.argtypes = [vp, vp, vp, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, vp, vp, ctypes.c_int]
        lib.oracle_gemm_relu_entries_ex.restype = ctypes.c_int
        lib.oracle_gemm_relu_entries_ex.argtypes = [vp, vp, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                                    ctypes.c_int, vp, vp, i64, vp, ctypes.c_int]
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        del dp
        _lib = lib
        return lib


def _as_half_bits(x) -> np.ndarray:
    """Accept float16 / uint16 numpy arrays or CPU torch fp16 / bf16 tensors;
    return a C-contiguous uint16 view of the raw 16-bit words."""
    if hasattr(x, "detach"):  # torch tensor
        import torch
        t = x.detach().cpu().contiguous()
        x = t.view(torch.int16).numpy().view(np.uint16).reshape(tuple(t.shape))
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        x = x.view(np.uint16)
    if x.dtype != np.uint16:
        raise TypeError(f"oracle inputs must be binary16 bits, got {x.dtype}")
    return x


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def half_to_double(bits: int) -> float:
    return float(_load().oracle_half_to_double(int(bits) & 0xFFFF))


def gemm_relu(A, B, apply_relu: bool = True, threads: int | None = None) -> np.ndarray:
    """Exact-as-binary64 C = ReLU(A.B) (or A.B when apply_relu is False).

    A: (M, K) binary16, B: (K, N) binary16, both row-major.  Returns an
    (M, N) float64 array, not rounded to binary16.
    """
    a = _as_half_bits(A)
    b = _as_half_bits(B)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[0]:
        raise ValueError(f"shape mismatch {a.shape} . {b.shape}")
    M, K = a.shape
    N = b.shape[1]
    c = np.empty((M, N), dtype=np.float64)
    ad = np.empty(max(M * K, 1), dtype=np.float64)
    bd = np.empty(max(K * N, 1), dtype=np.float64)
    nt = threads if threads is not None else 1
    rc = _load().oracle_gemm_relu(a.ctypes.data, b.ctypes.data, c.ctypes.data,
                                  M, N, K, int(bool(apply_relu)),
                                  ad.ctypes.data, bd.ctypes.data, int(nt))
    if rc != 0:
        raise ValueError("oracle_gemm_relu rejected its arguments")
    return c


def gemm_relu_entries(A, B, rows, cols, apply_relu: bool = True,
                      threads: int | None = None) -> np.ndarray:
    """The entries (rows[t], cols[t]) of ReLU(A.B), each summed in k order
    exactly as :func:`gemm_relu` does.  For sampled checks at full size."""
    a = _as_half_bits(A)
    b = _as_half_bits(B)
    M, K = a.shape
    K2, N = b.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    r = np.ascontiguousarray(rows, dtype=np.int64)
    cc = np.ascontiguousarray(cols, dtype=np.int64)
    if r.shape != cc.shape:
        raise ValueError("rows/cols length differ")
    out = np.empty(r.shape, dtype=np.float64)
    nt = threads if threads is not None else 1
    rc = _load().oracle_gemm_relu_entries(a.ctypes.data, b.ctypes.data, M, N, K,
                                          int(bool(apply_relu)), r.ctypes.data,
                                          cc.ctypes.data, r.size, out.ctypes.data, int(nt))
    if rc != 0:
        raise ValueError("oracle_gemm_relu_entries rejected its arguments")
    return out


# B layouts and element types of the _ex functions
B_LAYOUTS = {"kn": 0, "nk": 1}
DTYPES = {"f16": 0, "bf16": 1}


def bf16_to_double(bits: int) -> float:
    return float(_load().oracle_bf16_to_double(int(bits) & 0xFFFF))


def gemm_relu_ex(A, B, apply_relu: bool = True, b_layout: str = "kn", dtype: str = "f16",
                 threads: int | None = None) -> np.ndarray:
    """C = ReLU(A.B) with B given as (K, N) ("kn") or as (N, K) ("nk", then
    C = ReLU(A.B^T) of the stored matrix), elements binary16 ("f16") or
    bfloat16 ("bf16") words.  Returns an (M, N) float64 array, unrounded."""
    a = _as_half_bits(A)
    b = _as_half_bits(B)
    if a.ndim != 2 or b.ndim != 2:
        raise ValueError("A and B must be 2-D")
    M, K = a.shape
    if b_layout == "kn":
        K2, N = b.shape
    elif b_layout == "nk":
        N, K2 = b.shape
    else:
        raise ValueError(f"unknown B layout {b_layout!r}")
    if K2 != K:
        raise ValueError(f"shape mismatch {a.shape} . {b.shape} ({b_layout})")
    c = np.empty((M, N), dtype=np.float64)
    ad = np.empty(max(M * K, 1), dtype=np.float64)
    bd = np.empty(max(K * N, 1), dtype=np.float64)
    nt = threads if threads is not None else 1
    rc = _load().oracle_gemm_relu_ex(a.ctypes.data, b.ctypes.data, c.ctypes.data, M, N, K,
                                     int(bool(apply_relu)), B_LAYOUTS[b_layout], DTYPES[dtype],
                                     ad.ctypes.data, bd.ctypes.data, int(nt))
    if rc != 0:
        raise ValueError("oracle_gemm_relu_ex rejected its arguments")
    return c


def gemm_relu_entries_ex(A, B, rows, cols, apply_relu: bool = True, b_layout: str = "kn",
                         dtype: str = "f16", threads: int | None = None) -> np.ndarray:
    """Entries (rows[t], cols[t]) of :func:`gemm_relu_ex`, each summed in k order."""
    a = _as_half_bits(A)
    b = _as_half_bits(B)
    M, K = a.shape
    N = b.shape[1] if b_layout == "kn" else b.shape[0]
    K2 = b.shape[0] if b_layout == "kn" else b.shape[1]
    if K != K2:
        raise ValueError("inner dimensions differ")
    r = np.ascontiguousarray(rows, dtype=np.int64)
    cc = np.ascontiguousarray(cols, dtype=np.int64)
    if r.shape != cc.shape:
        raise ValueError("rows/cols length differ")
    out = np.empty(r.shape, dtype=np.float64)
    nt = threads if threads is not None else 1
    rc = _load().oracle_gemm_relu_entries_ex(a.ctypes.data, b.ctypes.data, M, N, K,
                                             int(bool(apply_relu)), B_LAYOUTS[b_layout],
                                             DTYPES[dtype], r.ctypes.data, cc.ctypes.data, r.size,
                                             out.ctypes.data, int(nt))
    if rc != 0:
        raise ValueError("oracle_gemm_relu_entries_ex rejected its arguments")
    return out


def within_tolerance(c_test, ref, rtol: float = 1e-2, atol: float = 1e-2) -> np.ndarray:
    """Elementwise |c - ref| <= atol + rtol * |ref| (the listing's
    assert_close rule with the oracle as the expected value)."""
    c_test = np.asarray(c_test, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return np.abs(c_test - ref) <= atol + rtol * np.abs(ref)


def matches_ieee(c_test, ref, rtol: float = 1e-2, atol: float = 1e-2) -> np.ndarray:
    """Elementwise comparison that also covers non-finite results (inputs
    holding NaN or infinities): a NaN expected value must be NaN, an
    infinite one the same infinity, a finite one within_tolerance.  The
    expected values follow the IEEE 754 rules (a NaN operand or 0 x inf
    makes a NaN term, inf + (-inf) is NaN) and ReLU's x > 0 ? x : +0."""
    c_test = np.asarray(c_test, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    fin = np.isfinite(ref)
    with np.errstate(invalid="ignore"):
        close = np.abs(np.where(fin, c_test, 0.0) - np.where(fin, ref, 0.0)) <= atol + rtol * np.abs(np.where(fin, ref, 0.0))
    return np.where(np.isnan(ref), np.isnan(c_test), np.where(np.isinf(ref), c_test == ref, close & np.isfinite(c_test)))
