"""Torch operator registrations for the library's products.

Importing this module registers ``torch.ops.mt.sgemm(a, b)`` and
``torch.ops.mt.gemm_bias(a, b, bias)`` as torch custom operators: the same
C-ABI calls as ``sgemm`` / ``gemm(..., bias=...)``, visible to torch's
dispatcher, graph capture and tracing (each has a shape-only fake
implementation, so tracing needs no GPU).  Marshalling only: the products
run in the library's kernels.
"""
from __future__ import annotations

import torch

from . import gemm, sgemm


@torch.library.custom_op("mt::sgemm", mutates_args=())
def sgemm_op(a: torch.Tensor, b: torch.Tensor) -> torch.Tensor:
    """a @ b (float32, CUDA, row-major) through mt_sgemm_ex."""
    return sgemm(a.contiguous(), b.contiguous())


@sgemm_op.register_fake
def _sgemm_fake(a: torch.Tensor, b: torch.Tensor) -> torch.Tensor:
    torch._check(a.dim() == 2 and b.dim() == 2 and a.shape[1] == b.shape[0],
                 lambda: "mt::sgemm needs (M, K) @ (K, N)")
    return a.new_empty((a.shape[0], b.shape[1]))


@torch.library.custom_op("mt::gemm_bias", mutates_args=())
def gemm_bias_op(a: torch.Tensor, b: torch.Tensor, bias: torch.Tensor) -> torch.Tensor:
    """a @ b + bias (bias: N values added to every row) through
    mt_sgemm_general_bias."""
    return gemm(a.contiguous(), b.contiguous(), bias=bias.contiguous())


@gemm_bias_op.register_fake
def _gemm_bias_fake(a: torch.Tensor, b: torch.Tensor, bias: torch.Tensor) -> torch.Tensor:
    torch._check(a.dim() == 2 and b.dim() == 2 and a.shape[1] == b.shape[0],
                 lambda: "mt::gemm_bias needs (M, K) @ (K, N)")
    torch._check(bias.dim() == 1 and bias.shape[0] == b.shape[1],
                 lambda: "mt::gemm_bias needs a bias of N values")
    return a.new_empty((a.shape[0], b.shape[1]))
