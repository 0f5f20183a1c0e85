"""The allocation-free 3xTF32 entry point against the allocating one.

mt_sgemm_tf32x3_noalloc serves callers that must not allocate device memory
while they run (memory owned by a host application or a caching allocator,
real-time loops that reserve everything up front): its scratch is a static
device array inside the library.  This file is collected last on purpose,
so a run that stops at the first failure has run every other test first.
"""
import numpy as np
import pytest
import torch

import gemm_inputs
import oracle
import tiled_fp32_gemm_gb300 as mt

pytestmark = pytest.mark.gpu

TOL = 5e-5  # the 3xTF32 tolerance the other tests use: |C - C_ref| <= TOL * |A|*|B|


@pytest.fixture(scope="module", autouse=True)
def library():
    from tiled_fp32_gemm_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    return mt.lib()


def allocating_call(a, b, M, N, K, stream):
    c = torch.full((M, N), float("nan"), device="cuda")
    st = mt.mt_sgemm_ex(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, stream,
                        mt.make_config(variant="tf32x3"))
    assert st == mt.MT_OK
    return c


def test_noalloc_matches_allocating_entry_point_on_two_calls_in_a_row():
    stream = torch.cuda.current_stream().cuda_stream
    # The larger problem first, then a smaller ragged one: the second call
    # runs on scratch still holding the first call's data.
    for name in ("square_1024", "masked_100x72x80"):
        w = gemm_inputs.WORKLOADS[name]
        A, B = gemm_inputs.make_workload(w)
        a, b = A.cuda(), B.cuda()
        ref = allocating_call(a, b, w.M, w.N, w.K, stream)
        c = torch.full((w.M, w.N), float("nan"), device="cuda")
        st = mt.mt_sgemm_tf32x3_noalloc(a.data_ptr(), b.data_ptr(), c.data_ptr(),
                                        w.M, w.N, w.K, stream)
        assert st == mt.MT_OK, mt.mt_status_string(st)
        torch.cuda.synchronize()
        _, W = oracle.sgemm(A.numpy(), B.numpy(), with_w=True)
        got = c.cpu().numpy().astype(np.float64)
        want = ref.cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        assert np.all(np.abs(got - want) <= TOL * W), name
    assert mt.mt_device_status(0) == mt.MT_OK


def test_noalloc_rejects_problems_beyond_its_scratch():
    M = N = K = 4096  # needs 128 MiB of packed copies
    assert mt.plan(M, N, K, variant="tf32x3")["workspace_bytes"] > mt.MT_NOALLOC_SCRATCH_BYTES
    a = torch.zeros((M, K), device="cuda")
    b = torch.zeros((K, N), device="cuda")
    c = torch.full((M, N), 3.0, device="cuda")
    st = mt.mt_sgemm_tf32x3_noalloc(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K,
                                    torch.cuda.current_stream().cuda_stream)
    assert st == mt.MT_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert torch.all(c == 3.0)  # nothing launched
