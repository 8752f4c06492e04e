"""GB300-native C = ReLU(A . B): fp16 inputs, fp32 accumulation, fp16 output.

The compute path is a hand-written sm_103a CUDA library behind a C ABI
(``include/gemm_relu.h``); ``binding`` marshals torch tensors to it.  The
library is loaded lazily on first use so that importing this package (for
example to draw the seeded workloads in ``workloads``) needs no GPU.
"""
import importlib

__all__ = ["gemm_relu", "gemm_relu_host", "binding", "workloads"]


def __getattr__(name):
    if name in ("binding", "build", "workloads"):
        return importlib.import_module(f".{name}", __name__)
    if name in ("gemm_relu", "gemm_relu_host", "check_device_error"):
        return getattr(importlib.import_module(".binding", __name__), name)
    raise AttributeError(name)
