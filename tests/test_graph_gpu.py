"""The library's calls inside a CUDA graph.

Stream capture records every launch a call makes (pack kernels, the GEMM,
split-tail reduce, stream-ordered workspace allocation and free) into a
graph; replaying the graph recomputes the products.  The 16-bit call's TMA
descriptors are kernel parameters, encoded once at capture time.
"""
import numpy as np
import pytest
import torch

import gemm_inputs
import oracle
import tiled_fp32_gemm_gb300 as mt

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    from tiled_fp32_gemm_gb300 import build
    build.build()
    return mt.lib()


def test_captured_calls_replay_to_the_same_results():
    M, N, K = 1000, 1100, 700
    A, B = gemm_inputs.make_ab(M, N, K, 31, "normal")
    A16, B16 = gemm_inputs.make_ab16(M, N, K, 32, "normal", "bf16")
    a, b, a16, b16 = A.cuda(), B.cuda(), A16.cuda(), B16.cuda()
    outs = [torch.empty(M, N, device="cuda") for _ in range(3)]
    calls = [lambda s: mt.sgemm(a, b, out=outs[0], stream=s),
             lambda s: mt.sgemm(a, b, out=outs[1], stream=s, variant="tf32x3"),
             lambda s: mt.gemm_mixed(a16, b16, outs[2], stream=s)]
    # Warm up outside capture: first calls set kernel attributes and look up
    # the tensor-map encoder, which are not stream work.
    for f in calls:
        f(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for f in calls:
            f(stream.cuda_stream)
    for o in outs:
        o.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert mt.mt_device_status(0) == mt.MT_OK
    Cref, W = oracle.sgemm(A.numpy(), B.numpy(), with_w=True)
    C16, W16 = oracle.gemm_mixed_general(oracle.BF16, A16, B16, np.zeros(M * N, np.float32),
                                         M, N, K, K, N, N, with_w=True)
    for got, want, w, tol in ((outs[0], Cref, W, 1e-5), (outs[1], Cref, W, 5e-5),
                              (outs[2], C16.reshape(M, N), W16, 5e-5)):
        err = np.abs(got.cpu().numpy().astype(np.float64) - want)
        assert np.all(err <= tol * w)
    # Replaying again after changing the inputs in place uses the new values.
    a.mul_(2.0)
    graph.replay()
    torch.cuda.synchronize()
    err = np.abs(outs[0].cpu().numpy().astype(np.float64) - 2.0 * Cref)
    assert np.all(err <= 2e-5 * W)
