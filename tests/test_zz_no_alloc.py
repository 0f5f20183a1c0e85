"""The allocation-free 3xTF32 entry point against the allocating one and the oracle.

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


def offset_view(A):
    """A's values in device memory 4 bytes past a 16-byte boundary: the
    tensor-memory copy cannot read A there, so the call packs A too."""
    M, K = A.shape
    store = torch.empty(M * K + 1, device="cuda")
    a = store[1:].view(M, K)
    a.copy_(A)
    return a


# (M, N, K, seed, A 16-byte aligned?, the plan it must take).  The first two
# split A inside the GEMM kernel and pack only B; the third packs A as well
# (one CTA per tile); the last packs both operands for the CTA-pair kernel
# and splits its last partial round over K, so the partial tiles live in
# the static scratch too.
CASES = [
    (1024, 1024, 1024, 1, True, dict(pack_a=2, bm=128)),
    (100, 72, 80, 0, True, dict(pack_a=2, bm=128)),
    (300, 200, 160, 5, False, dict(pack_a=1, bm=128)),
    (2304, 2304, 256, 6, False, dict(pack_a=1, bm=256)),
]


def test_noalloc_matches_allocating_entry_point_on_calls_in_a_row():
    stream = torch.cuda.current_stream().cuda_stream
    # Larger problems before smaller ones, each call on scratch that still
    # holds the previous call's data; the sequence runs twice.
    for _ in range(2):
        for M, N, K, seed, aligned, want in CASES:
            A, B = gemm_inputs.make_ab(M, N, K, seed=seed, dist="uniform")
            a = A.cuda() if aligned else offset_view(A.cuda())
            b = B.cuda()
            p = mt.plan(M, N, K, a=a, b=b, variant="tf32x3")
            assert {k: p[k] for k in want} == want, p
            assert p["workspace_bytes"] <= mt.MT_NOALLOC_SCRATCH_BYTES
            ref = allocating_call(a, b, M, N, K, stream)
            c = torch.full((M, N), float("nan"), device="cuda")
            st = mt.mt_sgemm_tf32x3_noalloc(a.data_ptr(), b.data_ptr(), c.data_ptr(),
                                            M, N, K, stream)
            assert st == mt.MT_OK, mt.mt_status_string(st)
            torch.cuda.synchronize()
            got = c.cpu().numpy()
            # The same plan and kernels on another buffer: the same bits.
            assert np.array_equal(got, ref.cpu().numpy()), (M, N, K)
            Cref, W = oracle.sgemm(A.numpy(), B.numpy(), with_w=True)
            err = np.abs(got.astype(np.float64) - Cref)
            assert np.all(err <= TOL * W), (M, N, K, float((err / np.maximum(W, 1e-300)).max()))
    assert mt.mt_check_device_status(0) == mt.MT_OK


def test_noalloc_rejects_problems_beyond_its_scratch():
    M = N = K = 4096  # the packed copies of A and B alone are 256 MiB
    assert mt.plan(M, N, K, variant="tf32x3")["workspace_bytes"] > mt.MT_NOALLOC_SCRATCH_BYTES
    a = torch.zeros((M, K), device="cuda")
    b = torch.zeros((K, N), device="cuda")
    c = torch.full((M, N), 3.0, device="cuda")
    st = mt.mt_sgemm_tf32x3_noalloc(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K,
                                    torch.cuda.current_stream().cuda_stream)
    assert st == mt.MT_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert torch.all(c == 3.0)  # nothing launched
