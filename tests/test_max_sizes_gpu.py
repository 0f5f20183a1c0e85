"""GPU: operands past 2^31 elements (64-bit indexing).

Three products, each with one operand longer than 2^31 elements, so every
index that a kernel forms from row * leading dimension must be 64-bit:

* A: 524325 x 4100 (2.15e9 elements; N = 72, so A is gathered K-major by
  the FFMA kernel and split inside the 3xTF32 kernel);
* C: 46341 x 46341 (K = 8; A copied K-major, 128 x 128 tiles);
* B: 65541 x 32771 (M = 8; N is not a multiple of 4, so B is copied into
  padded rows first, itself 2.15e9 elements).

Inputs are small integers given by a formula, built on the device with
torch arithmetic (never by this library) and rebuilt on the host for the
sampled rows and columns; every partial sum stays below 2^24, so each
variant's result is exact and must equal the oracle's bit for bit.  The
bounds-checked build runs every case first and must find no access outside
its buffers.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import tiled_fp32_gemm_gb300 as mt

pytestmark = pytest.mark.gpu

CASES = {"A": (524325, 72, 4100), "C": (46341, 46341, 8), "B": (8, 32771, 65541)}
VARIANTS = [dict(), dict(variant="tf32x3"), dict(variant="p18")]


def a_formula(i, k):
    return ((3 * i + 7 * k) % 17 - 8).astype(np.float32)


def b_formula(k, j):
    return ((5 * k + 11 * j) % 13 - 6).astype(np.float32)


def device_matrix(rows, cols, formula_id):
    """The formula's rows x cols matrix on the device, built in row chunks."""
    out = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
    cols_i = torch.arange(cols, device="cuda", dtype=torch.int64)
    step = max(1, (1 << 27) // cols)
    for r0 in range(0, rows, step):
        r = torch.arange(r0, min(rows, r0 + step), device="cuda", dtype=torch.int64)[:, None]
        if formula_id == "a":
            v = (3 * r + 7 * cols_i[None, :]) % 17 - 8
        else:
            v = (5 * r + 11 * cols_i[None, :]) % 13 - 6
        out[r0:r0 + r.shape[0]] = v.to(torch.float32)
    return out


@pytest.fixture(scope="module")
def checked():
    from tiled_fp32_gemm_gb300 import build
    build.build(checked=True)
    h = mt.checked_lib()
    mt.bounds_status(h)
    return h


def call(h, a, b, c, M, N, K, cfg):
    conf = mt.make_config(**cfg) if cfg else None
    st = h.mt_sgemm_ex(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K,
                       torch.cuda.current_stream().cuda_stream,
                       ctypes.byref(conf) if conf is not None else None)
    assert st == mt.MT_OK, mt.mt_status_string(st)
    torch.cuda.synchronize()


def samples(M, N, K):
    """Output positions whose row (of A or C) or column (of B) lies past
    2^31 elements into its operand, plus the corners."""
    rows = {0, M - 1, M // 2}
    cols = {0, N - 1, N // 2}
    if M * K > 2 ** 31:
        rows |= {2 ** 31 // K, 2 ** 31 // K + 1}
    if M * N > 2 ** 31:
        rows |= {2 ** 31 // N, 2 ** 31 // N + 1}
    if K * N > 2 ** 31:
        cols |= {(2 ** 31 % N) - 1, 2 ** 31 % N, N - 2}
    return sorted(r for r in rows if r < M), sorted(c for c in cols if 0 <= c < N)


@pytest.mark.parametrize("case", sorted(CASES))
def test_operands_past_two_to_the_31(case, checked):
    M, N, K = CASES[case]
    assert max(M * K, K * N, M * N) > 2 ** 31
    a = device_matrix(M, K, "a")
    b = device_matrix(K, N, "b")
    c = torch.empty((M, N), dtype=torch.float32, device="cuda")
    rows, cols = samples(M, N, K)
    ks = np.arange(K, dtype=np.int64)
    want = np.empty((len(rows), len(cols)), np.float64)
    for x, i in enumerate(rows):
        a_row = a_formula(np.int64(i), ks)[None, :]
        for y, j in enumerate(cols):
            b_col = b_formula(ks, np.int64(j))[:, None]
            want[x, y] = oracle.sgemm(a_row, b_col)[0, 0]  # the 1 x 1 product
    rsel = torch.tensor(rows, device="cuda")
    csel = torch.tensor(cols, device="cuda")
    for handle, name in ((checked, "checked"), (mt.lib(), "normal")):
        for cfg in VARIANTS:
            c.fill_(float("nan"))
            call(handle, a, b, c, M, N, K, cfg)
            got = c[rsel][:, csel].cpu().numpy()
            assert np.array_equal(got, want), (case, name, cfg)
            assert not torch.isnan(c[-1]).any()
            if handle is checked:
                rec = mt.bounds_status(checked)
                assert rec["count"] == 0, (case, cfg, rec)
    del a, b, c
    torch.cuda.empty_cache()
