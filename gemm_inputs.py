"""Seeded synthetic inputs for the fp32 GEMM workloads.

Shared by the tests, the smoke check and the benchmark.  It only draws
random numbers; it holds none of the product's arithmetic, so both the CUDA
path and the CPU oracle can be fed from it without sharing method code.

Recipe: a CPU ``torch.Generator`` seeded with the workload's seed draws A
(M x K) and then B (K x N) in float32.  "uniform" is ``rand*2-1`` (values in
[-1, 1)), "normal" is ``randn`` (mean 0, variance 1), "int" draws integers
in [-8, 8] (exact test inputs).  A workload that names two shapes reseeds the
generator for each shape.

16-bit inputs (``make_ab16``): the same float32 draws, rounded to the
nearest float16 or bfloat16 by torch's CPU conversion.  The 16-bit values
are the inputs; both sides read the same patterns.
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
    seed: int
    dist: str  # "uniform" | "normal"

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


# The named workloads: every shape the benchmark and the parity tests use.
WORKLOADS = {
    "masked_100x72x80": Workload("masked_100x72x80", 100, 72, 80, 0, "uniform"),
    "square_1024": Workload("square_1024", 1024, 1024, 1024, 1, "normal"),
    "square_4096": Workload("square_4096", 4096, 4096, 4096, 2, "uniform"),
    "ragged_4097x3001x2053": Workload("ragged_4097x3001x2053", 4097, 3001, 2053,
                                      3, "normal"),
    "square_8192": Workload("square_8192", 8192, 8192, 8192, 4, "uniform"),
    "skinny_65536x128x4096": Workload("skinny_65536x128x4096", 65536, 128,
                                      4096, 4, "uniform"),
}


def _draw(shape, dist: str, g: torch.Generator) -> torch.Tensor:
    if dist == "uniform":
        return torch.rand(shape, generator=g, dtype=torch.float32) * 2 - 1
    if dist == "normal":
        return torch.randn(shape, generator=g, dtype=torch.float32)
    if dist == "int":
        return torch.randint(-8, 9, shape, generator=g).to(torch.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def make_ab(M: int, N: int, K: int, seed: int, dist: str = "uniform"):
    """(A, B) as contiguous float32 CPU tensors: A is M x K, B is K x N."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    A = _draw((M, K), dist, g).contiguous()
    B = _draw((K, N), dist, g).contiguous()
    return A, B


def make_workload(w: Workload | str):
    if isinstance(w, str):
        w = WORKLOADS[w]
    return make_ab(w.M, w.N, w.K, w.seed, w.dist)


def make_ab16(M: int, N: int, K: int, seed: int, dist: str = "uniform",
              dtype: str = "bf16"):
    """(A, B) as contiguous CPU tensors of torch.bfloat16 ("bf16") or
    torch.float16 ("f16"): the float32 draws of make_ab, rounded."""
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16}[dtype]
    A, B = make_ab(M, N, K, seed, dist)
    return A.to(tdt).contiguous(), B.to(tdt).contiguous()
