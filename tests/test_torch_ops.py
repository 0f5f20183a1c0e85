"""The torch operator registrations (tiled_fp32_gemm_gb300.torch_ops).

CPU: the operators exist and their fake implementations give the output
shape, device and dtype without running anything (tracing needs no GPU).
GPU: each operator returns exactly what the direct binding returns; both
replay correctly from a CUDA graph, including a plan whose call allocates
workspace (the transposing copy of A) inside the capture; dynamo traces
them as single calls.
"""
import numpy as np
import pytest
import torch
from torch._subclasses.fake_tensor import FakeTensorMode

import oracle
import tiled_fp32_gemm_gb300 as mt
import tiled_fp32_gemm_gb300.torch_ops  # noqa: F401  (registers torch.ops.mt.*)


def test_operators_registered_with_shape_only_fakes():
    with FakeTensorMode():
        a = torch.empty(8, 5, device="cuda")
        b = torch.empty(5, 3, device="cuda")
        bias = torch.empty(3, device="cuda")
        for out in (torch.ops.mt.sgemm(a, b), torch.ops.mt.gemm_bias(a, b, bias)):
            assert tuple(out.shape) == (8, 3) and out.dtype == torch.float32
            assert out.device.type == "cuda"
        with pytest.raises(Exception):
            torch.ops.mt.sgemm(a, torch.empty(4, 3, device="cuda"))
        with pytest.raises(Exception):
            torch.ops.mt.gemm_bias(a, b, torch.empty(4, device="cuda"))


@pytest.mark.gpu
def test_operators_match_the_binding_and_replay_from_a_graph():
    g = torch.Generator().manual_seed(50)
    M, N, K = 512, 2048, 1024          # N >= 2048, 2^30 multiply-adds: A is copied K-major
    assert mt.plan(M, N, K)["pack_a"] == 5
    A = torch.randn(M, K, generator=g)
    B = torch.randn(K, N, generator=g)
    bias = torch.randn(N, generator=g)
    a, b, bd = A.cuda(), B.cuda(), bias.cuda()
    assert torch.equal(torch.ops.mt.sgemm(a, b), mt.sgemm(a, b))
    assert torch.equal(torch.ops.mt.gemm_bias(a, b, bd), mt.gemm(a, b, bias=bd))
    torch.cuda.synchronize()
    # Captured: the copy of A, its workspace, the GEMM and the bias epilogue.
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        torch.ops.mt.gemm_bias(a, b, bd)   # warm up on the capture stream
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        out = torch.ops.mt.gemm_bias(a, b, bd)
    a.mul_(-1.0)
    graph.replay()
    torch.cuda.synchronize()
    Cref, W = oracle.sgemm((-A).numpy(), B.numpy(), with_w=True)
    want = Cref.astype(np.float64) + bias.numpy()[None, :]
    err = np.abs(out.cpu().numpy().astype(np.float64) - want)
    assert np.all(err <= 1e-5 * (W + np.abs(bias.numpy())[None, :]))
    assert mt.mt_device_status(0) == mt.MT_OK


@pytest.mark.gpu
def test_dynamo_traces_the_operators():
    torch._dynamo.reset()

    def layer(x, w, b):
        return torch.relu(torch.ops.mt.gemm_bias(x, w, b))

    g = torch.Generator().manual_seed(51)
    x = torch.randn(100, 80, generator=g).cuda()
    w = torch.randn(80, 72, generator=g).cuda()
    b = torch.randn(72, generator=g).cuda()
    compiled = torch.compile(layer, backend="eager", fullgraph=True)
    assert torch.equal(compiled(x, w, b), layer(x, w, b))
