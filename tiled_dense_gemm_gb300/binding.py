"""ctypes binding to libgemmrelu.so (argument marshalling only).

Every step of the computation runs in the CUDA library; this module checks
tensor properties, passes raw pointers, sizes and the current CUDA stream,
and turns status codes into exceptions.  There is no CPU fallback: if the
library is missing or the device is not a GB300 (sm_103a), calls raise.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from .build import INCLUDE, LIB_PATH

GEMM_OK = 0
STATUS_NAMES = {
    0: "GEMM_OK", 1: "GEMM_ERR_INVALID_ARG", 2: "GEMM_ERR_ALIGNMENT",
    3: "GEMM_ERR_UNSUPPORTED_DEVICE", 4: "GEMM_ERR_OUT_OF_MEMORY", 5: "GEMM_ERR_LAUNCH",
    6: "GEMM_ERR_TIMEOUT", 7: "GEMM_ERR_CUDA", 8: "GEMM_ERR_TOO_LARGE",
}


class GemmReluError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}" if what else
                         STATUS_NAMES.get(status, str(status)))


class Plan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "path", "mma_m", "mma_n", "tile_m", "tile_n", "tiles_m", "tiles_n", "num_tiles",
        "num_kb", "block_k", "group_m", "grid", "cluster", "dp_tiles", "sk_tiles", "sk_q", "sk_r",
        "splits", "max_slots", "num_stages", "stage_bytes", "smem_bytes", "tmem_cols", "pack_a")] + [
        ("workspace_bytes", ctypes.c_int64), ("counter_count", ctypes.c_int64)]

    def as_dict(self) -> dict:
        return {n: getattr(self, n) for n, _ in self._fields_}


_lock = threading.Lock()
_lib = None


class Boxes(ctypes.Structure):
    """gemm_relu_boxes_t: the TMA boxes of one ring stage's copies."""
    _fields_ = [("a_3d", ctypes.c_int32), ("a_box", ctypes.c_uint32 * 3), ("b_3d", ctypes.c_int32),
                ("b_box", ctypes.c_uint32 * 3), ("b2_box", ctypes.c_uint32 * 2), ("b_view_inner", ctypes.c_int64)]

    def as_dict(self) -> dict:
        return {"a_3d": self.a_3d, "a_box": list(self.a_box), "b_3d": self.b_3d, "b_box": list(self.b_box),
                "b2_box": list(self.b2_box), "b_view_inner": self.b_view_inner}


def declared_functions() -> list[str]:
    """Names of the functions include/gemm_relu.h declares."""
    text = open(os.path.join(INCLUDE, "gemm_relu.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_relu\w*)\s*\(", text)))


def lib():
    """Load libgemmrelu.so (built by ``__graft_entry__.build()`` or
    ``python -m tiled_dense_gemm_gb300.build``).  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing; build it first "
                               "(python -m tiled_dense_gemm_gb300.build)")
        L = ctypes.CDLL(LIB_PATH)
        i64, vp, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        L.gemm_relu.restype = i32
        L.gemm_relu.argtypes = [vp, vp, vp, i64, i64, i64, i32, vp]
        L.gemm_relu_ex.restype = i32
        L.gemm_relu_ex.argtypes = [vp, vp, vp, i64, i64, i64, i32, i32, i32, vp]
        L.gemm_relu_host.restype = i32
        L.gemm_relu_host.argtypes = [vp, vp, vp, i64, i64, i64, i32, vp]
        L.gemm_relu_noalloc.restype = i32
        L.gemm_relu_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, i32, vp]
        L.gemm_relu_noalloc_check_device_error.restype = i32
        L.gemm_relu_noalloc_check_device_error.argtypes = [vp]
        L.gemm_relu_check_device_error.restype = i32
        L.gemm_relu_check_device_error.argtypes = [vp]
        L.gemm_relu_status_string.restype = ctypes.c_char_p
        L.gemm_relu_status_string.argtypes = [i32]
        L.gemm_relu_shutdown.restype = None
        L.gemm_relu_shutdown.argtypes = []
        L.gemm_relu_plan.restype = i32
        L.gemm_relu_plan.argtypes = [i64, i64, i64, i32, ctypes.POINTER(Plan)]
        p32 = ctypes.POINTER(ctypes.c_int32)
        L.gemm_relu_plan_boxes.restype = i32
        L.gemm_relu_plan_boxes.argtypes = [ctypes.POINTER(Plan), i64, i64, i64, i32, ctypes.POINTER(Boxes)]
        L.gemm_relu_plan_work_item.restype = i32
        L.gemm_relu_plan_work_item.argtypes = [ctypes.POINTER(Plan), i32, i32] + [p32] * 7
        _lib = L
        return L


def status_string(status: int) -> str:
    return lib().gemm_relu_status_string(int(status)).decode()


def plan(M: int, N: int, K: int, num_sms: int) -> Plan:
    p = Plan()
    rc = lib().gemm_relu_plan(M, N, K, num_sms, ctypes.byref(p))
    if rc != GEMM_OK:
        raise GemmReluError(rc, "gemm_relu_plan")
    return p


def plan_work_items(p: Plan, cta: int) -> list[dict]:
    """Work items of one CTA, as the kernel walks them."""
    out = []
    vals = [ctypes.c_int32() for _ in range(7)]
    idx = 0
    while True:
        rc = lib().gemm_relu_plan_work_item(ctypes.byref(p), cta, idx,
                                            *[ctypes.byref(v) for v in vals])
        if rc < 0:
            raise GemmReluError(GEMM_OK + 1, "gemm_relu_plan_work_item")
        if rc == 0:
            return out
        out.append(dict(zip(("tile", "tm", "tn", "kb0", "kb1", "slot", "nslots"),
                            (v.value for v in vals))))
        idx += 1


def plan_boxes(p: Plan, M: int, N: int, K: int, b_layout: str = "kn") -> Boxes:
    """The TMA boxes the kernel's copies use for one ring stage under plan ``p``."""
    out = Boxes()
    rc = lib().gemm_relu_plan_boxes(ctypes.byref(p), M, N, K, B_LAYOUTS[b_layout], ctypes.byref(out))
    if rc != GEMM_OK:
        raise GemmReluError(rc, "gemm_relu_plan_boxes")
    return out


def _stream_handle(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _on_device(device, fn, *args):
    """Call fn(*args) with `device` current (no device switch when it
    already is: the switch costs more host time than the call itself)."""
    import torch
    if device.index is None or device.index == torch.cuda.current_device():
        return fn(*args)
    with torch.cuda.device(device):
        return fn(*args)


def gemm_relu(a, b, c=None, apply_relu: bool = True, stream=None):
    """C = ReLU(a @ b) (or a @ b) for CUDA fp16 tensors a (M, K), b (K, N).

    ``c`` (M, N) fp16 is written in place when given, else allocated.  Runs
    asynchronously on ``stream`` (default: torch's current stream)."""
    import torch
    if not (isinstance(a, torch.Tensor) and isinstance(b, torch.Tensor)):
        raise TypeError("a and b must be torch tensors")
    if a.dtype != torch.float16 or b.dtype != torch.float16:
        raise TypeError("a and b must be float16")
    if a.dim() != 2 or b.dim() != 2 or a.shape[1] != b.shape[0]:
        raise ValueError(f"bad shapes {tuple(a.shape)} @ {tuple(b.shape)}")
    if not (a.is_cuda and b.is_cuda) or a.device != b.device:
        raise ValueError("a and b must be CUDA tensors on the same device")
    if not (a.is_contiguous() and b.is_contiguous()):
        raise ValueError("a and b must be contiguous row-major (call .contiguous())")
    M, K = a.shape
    N = b.shape[1]
    if c is None:
        c = torch.empty((M, N), dtype=torch.float16, device=a.device)
    elif (c.dtype != torch.float16 or tuple(c.shape) != (M, N) or c.device != a.device
          or not c.is_contiguous()):
        raise ValueError("c must be a contiguous float16 (M, N) tensor on a's device")
    rc = _on_device(a.device, lib().gemm_relu, a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K,
                    int(bool(apply_relu)), _stream_handle(stream, a.device))
    if rc != GEMM_OK:
        raise GemmReluError(rc, "gemm_relu")
    return c


B_LAYOUTS = {"kn": 0, "nk": 1}  # gemm_b_layout_t


def gemm_relu_ex(a, b, c=None, apply_relu: bool = True, b_layout: str = "kn", stream=None):
    """C = ReLU(a @ b) for b_layout "kn" (b is (K, N)) or ReLU(a @ b.T) for
    "nk" (b is (N, K)); a, b and c are CUDA tensors of one element type,
    float16 or bfloat16.  ``c`` (M, N) is written in place when given."""
    import torch
    if not (isinstance(a, torch.Tensor) and isinstance(b, torch.Tensor)):
        raise TypeError("a and b must be torch tensors")
    dtypes = {torch.float16: 0, torch.bfloat16: 1}
    if a.dtype not in dtypes or b.dtype != a.dtype:
        raise TypeError("a and b must both be float16 or both bfloat16")
    if b_layout not in B_LAYOUTS:
        raise ValueError(f"b_layout must be 'kn' or 'nk', not {b_layout!r}")
    if a.dim() != 2 or b.dim() != 2:
        raise ValueError("a and b must be 2-D")
    M, K = a.shape
    N, Kb = (b.shape[1], b.shape[0]) if b_layout == "kn" else (b.shape[0], b.shape[1])
    if Kb != K:
        raise ValueError(f"bad shapes {tuple(a.shape)} and {tuple(b.shape)} ({b_layout})")
    if not (a.is_cuda and b.is_cuda) or a.device != b.device:
        raise ValueError("a and b must be CUDA tensors on the same device")
    if not (a.is_contiguous() and b.is_contiguous()):
        raise ValueError("a and b must be contiguous row-major (call .contiguous())")
    if c is None:
        c = torch.empty((M, N), dtype=a.dtype, device=a.device)
    elif (c.dtype != a.dtype or tuple(c.shape) != (M, N) or c.device != a.device
          or not c.is_contiguous()):
        raise ValueError("c must be a contiguous (M, N) tensor of a's type on a's device")
    rc = _on_device(a.device, lib().gemm_relu_ex, a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K,
                    int(bool(apply_relu)), B_LAYOUTS[b_layout], dtypes[a.dtype],
                    _stream_handle(stream, a.device))
    if rc != GEMM_OK:
        raise GemmReluError(rc, "gemm_relu_ex")
    return c


def gemm_relu_host(a, b, c=None, apply_relu: bool = True, stream=None, device=None):
    """Same operation on CPU fp16 tensors (pinned memory is fastest): the
    library copies them to the GPU, computes, and copies C back before
    returning."""
    import torch
    if a.dtype != torch.float16 or b.dtype != torch.float16 or a.is_cuda or b.is_cuda:
        raise TypeError("a and b must be CPU float16 tensors")
    if a.dim() != 2 or b.dim() != 2 or a.shape[1] != b.shape[0]:
        raise ValueError(f"bad shapes {tuple(a.shape)} @ {tuple(b.shape)}")
    if not (a.is_contiguous() and b.is_contiguous()):
        raise ValueError("a and b must be contiguous")
    M, K = a.shape
    N = b.shape[1]
    if c is None:
        c = torch.empty((M, N), dtype=torch.float16, pin_memory=a.is_pinned())
    cur = torch.cuda.current_device()
    dev = torch.device("cuda", cur) if device is None else torch.device(device)
    args = (a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, int(bool(apply_relu)), _stream_handle(stream, dev))
    if dev.index is None or dev.index == cur:
        rc = lib().gemm_relu_host(*args)
    else:
        with torch.cuda.device(dev):
            rc = lib().gemm_relu_host(*args)
    if rc != GEMM_OK:
        raise GemmReluError(rc, "gemm_relu_host")
    return c


def check_device_error(stream=None, device=None):
    """Synchronize ``stream`` and raise if a kernel of this library reported
    a timed-out wait since the last check."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        rc = lib().gemm_relu_check_device_error(_stream_handle(stream, dev))
    if rc != GEMM_OK:
        raise GemmReluError(rc, "device")


def gemm_relu_noalloc(a, b, c, apply_relu: bool = True, stream=None):
    """gemm_relu through the entry point that allocates no device memory
    (small M only; its split-K scratch is a fixed device array of the
    library).  ``c`` must be given: this call allocates nothing."""
    import torch
    if a.dtype != torch.float16 or b.dtype != torch.float16 or c.dtype != torch.float16:
        raise TypeError("a, b and c must be float16")
    if a.dim() != 2 or b.dim() != 2 or a.shape[1] != b.shape[0] or tuple(c.shape) != (a.shape[0], b.shape[1]):
        raise ValueError(f"bad shapes {tuple(a.shape)} @ {tuple(b.shape)} -> {tuple(c.shape)}")
    if not (a.is_cuda and b.is_cuda and c.is_cuda) or a.device != b.device or c.device != a.device:
        raise ValueError("a, b and c must be CUDA tensors on one device")
    if not (a.is_contiguous() and b.is_contiguous() and c.is_contiguous()):
        raise ValueError("a, b and c must be contiguous row-major")
    M, K = a.shape
    N = b.shape[1]
    rc = _on_device(a.device, lib().gemm_relu_noalloc, a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K,
                    int(bool(apply_relu)), _stream_handle(stream, a.device))
    if rc != GEMM_OK:
        raise GemmReluError(rc, "gemm_relu_noalloc")
    return c


def noalloc_check_device_error(stream=None, device=None):
    """Synchronize ``stream`` and raise if a gemm_relu_noalloc kernel
    reported a timed-out wait since the last check."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        rc = lib().gemm_relu_noalloc_check_device_error(_stream_handle(stream, dev))
    if rc != GEMM_OK:
        raise GemmReluError(rc, "device (noalloc)")


def shutdown():
    lib().gemm_relu_shutdown()
