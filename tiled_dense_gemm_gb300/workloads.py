"""Seeded synthetic inputs for C = ReLU(A . B).

This module only draws random binary16 (or bfloat16) matrices; it holds none of the
product's arithmetic, so both the CUDA path and the CPU oracle can consume
the same bytes without sharing any compute code.

Recipe (the same for every workload): a CPU ``torch.Generator`` seeded with
the workload's seed draws A first, then B, in float32, scales them, and
rounds once to binary16 (round-to-nearest-even).  ``normal`` draws
``randn``; ``uniform`` draws ``rand * 2 - 1`` (U(-1, 1)); ``intgrid`` draws
integers uniformly from [-r, r] (exact in binary16).

The shapes and distributions are the five workloads this library is
measured and checked on:

* ``c1_256``   256^3, A, B ~ N(0, 1), seed 0 -- small case.
* ``c2_1024``  1024^3, A, B ~ N(0, 1), seed 1 -- the worked size of the
  GEMM+ReLU tutorial listing ("Writing High-Performance Kernels in
  TileLang", GEMM section: M = N = K = 1024, torch.randn inputs).
* ``c3_4096``  4096^3, A, B ~ N(0, 1) * 4096**-0.25, seed 2 -- square,
  tensor-core bound; per-element std K^-1/4 keeps outputs O(1).
* ``c4_skinny`` M=16, N=K=8192, A ~ N(0, 1), B ~ N(0, 1/K), seed 3 --
  decode-like, HBM bound.
* ``c5_ragged`` M=3000, N=5000, K=2056, A, B ~ U(-1, 1), seed 4 -- no
  dimension a multiple of 128; checked with ReLU on and off.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dist_a: str          # "normal" | "uniform" | "intgrid"
    scale_a: float
    dist_b: str
    scale_b: float
    seed: int
    relu_modes: tuple = (True,)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def algorithmic_bytes(self) -> int:
        """A and B read once, C written once, binary16 each."""
        return 2 * (self.M * self.K + self.K * self.N + self.M * self.N)


WORKLOADS = {
    w.name: w for w in [
        Workload("c1_256", 256, 256, 256, "normal", 1.0, "normal", 1.0, 0),
        Workload("c2_1024", 1024, 1024, 1024, "normal", 1.0, "normal", 1.0, 1),
        Workload("c3_4096", 4096, 4096, 4096, "normal", 4096 ** -0.25,
                 "normal", 4096 ** -0.25, 2),
        Workload("c4_skinny", 16, 8192, 8192, "normal", 1.0, "normal", 8192 ** -0.5, 3),
        Workload("c5_ragged", 3000, 5000, 2056, "uniform", 1.0, "uniform", 1.0, 4,
                 relu_modes=(True, False)),
    ]
}


def _draw(g: torch.Generator, shape, dist: str, scale: float, dtype=torch.float16) -> torch.Tensor:
    if dist == "normal":
        x = torch.randn(shape, generator=g, dtype=torch.float32)
    elif dist == "uniform":
        x = torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    elif dist == "intgrid":
        r = int(scale)
        return torch.randint(-r, r + 1, shape, generator=g, dtype=torch.int32).to(dtype)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return (x * scale).to(dtype)


def make_inputs(M: int, N: int, K: int, seed: int, dist_a: str = "normal",
                scale_a: float = 1.0, dist_b: str = "normal", scale_b: float = 1.0,
                dtype=torch.float16, b_layout: str = "kn"):
    """Return (A, B): CPU tensors of shapes (M, K) and (K, N), rounded once to
    ``dtype`` (binary16 or bfloat16).  With ``b_layout="nk"`` B is returned
    stored as its (N, K) transpose, same values (drawn in the (K, N) order)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    a = _draw(g, (M, K), dist_a, scale_a, dtype).contiguous()
    b = _draw(g, (K, N), dist_b, scale_b, dtype).contiguous()
    if b_layout == "nk":
        b = b.t().contiguous()
    elif b_layout != "kn":
        raise ValueError(f"unknown B layout {b_layout!r}")
    return a, b


def workload_inputs(name_or_workload, seed_offset: int = 0):
    """(A, B) for one of the named workloads.  ``seed_offset`` gives extra,
    independent input sets of the same shape and distribution (used to keep
    the benchmark's inputs out of L2)."""
    w = WORKLOADS[name_or_workload] if isinstance(name_or_workload, str) else name_or_workload
    return make_inputs(w.M, w.N, w.K, w.seed + 1000003 * seed_offset,
                       w.dist_a, w.scale_a, w.dist_b, w.scale_b)
