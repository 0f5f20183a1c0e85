"""GPU: the bounds-checked build.

libmtsgemm_checked.so is the library built with MT_BOUNDS_CHECK=1: before
every global or shared access, the FFMA GEMM kernel (all staging forms,
tiles, pipeline depths and K splits), its operand copies, the K-slice reduce,
the C scaling kernel and the one-warp kernel test the access against the
extent of the buffer it belongs to, and so do the tensor-core paths' own
accesses (the 3xTF32 packers, the 16-bit repack, the TMEM-to-C epilogue and
its partial tiles; their operands reach the MMAs through TMA, which bounds
every copy by its tensor map); an access outside is skipped and counted
(mt_bounds_status).  It takes the place of a memory checker, which cannot run
here.  These tests run the plans through that build and require (1) no
access outside any buffer and (2) the oracle's results within the variant's
tolerance (FFMA 1e-5 * W, tensor cores 5e-5 * W), so the checks did not skip
anything that mattered.  A mistake planted on the host (C declared one element shorter
than it is) shows that the record does catch an access outside: the last
store is reported and skipped, and no access leaves the real buffer.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

import gemm_inputs
import oracle
import tiled_fp32_gemm_gb300 as mt

pytestmark = pytest.mark.gpu

TOL = 1e-5

# FFMA-path plans: every staging form of A (row-major as stored / from a
# copy, K-major gathered / from a copy / as stored), tile, pipeline depth,
# K groups of warps, explicit and automatic K splits, stream-K runs and their
# fix-up, and the one-warp kernel.
CONFIGS = [dict(), dict(pack_a=1), dict(pack_a=2), dict(pack_a=4), dict(pack_a=5),
           dict(bm=64, bn=128, pack_a=4), dict(bm=64, bn=64, pack_a=5),
           dict(bm=64, bn=128, stages=3, pack_a=5),
           dict(bm=128, bn=128, bk=32, stages=3, fma=2),
           dict(bm=128, bn=128, bk=16, stages=1), dict(bm=128, bn=128, bk=16, stages=2),
           dict(pack_a=4, split_k=3), dict(bm=128, bn=128, bk=32, stages=3, no_pad=True),
           dict(schedule=2), dict(bm=128, bn=128, bk=16, stages=4, wm=64, pack_a=5, schedule=2),
           dict(bm=64, bn=64, pack_a=4, schedule=2),
           dict(variant="p18"), dict(variant="p18", stages=1)]


def ids(cfgs):
    return ["-".join(f"{k}{v}" for k, v in c.items()) or "auto" for c in cfgs]


@pytest.fixture(scope="module", autouse=True)
def checked():
    from tiled_fp32_gemm_gb300 import build
    build.build(checked=True)
    assert torch.cuda.is_available()
    h = mt.checked_lib()
    mt.bounds_status(h)  # start from a clear record
    return h


def stored(g, rows, cols, ld):
    """rows x cols normal values inside a rows x ld buffer of NaN."""
    buf = np.full((rows, ld), np.nan, np.float32)
    buf[:, :cols] = g.standard_normal((rows, cols))
    return buf


def general(h, ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C0, ldc, bias=None, **cfg):
    a, b, c = (torch.from_numpy(x).cuda() for x in (A, B, C0))
    bz = torch.from_numpy(bias).cuda() if bias is not None else None
    conf = mt.make_config(**cfg) if cfg else None
    st = h.mt_sgemm_general_bias(ta, tb, M, N, K, alpha, a.data_ptr(), lda, b.data_ptr(), ldb,
                                 beta, bz.data_ptr() if bz is not None else None, c.data_ptr(),
                                 ldc, torch.cuda.current_stream().cuda_stream,
                                 ctypes.byref(conf) if conf is not None else None)
    if st == mt.MT_ERR_UNSUPPORTED:
        pytest.skip("this tile has no kernel for these transposes (as in the normal build)")
    assert st == mt.MT_OK, mt.mt_status_string(st)
    torch.cuda.synchronize()
    return c.cpu().numpy()


def assert_clean(h, what):
    rec = mt.bounds_status(h)
    assert rec["count"] == 0, f"{what}: {rec}"


@pytest.mark.parametrize("cfg", CONFIGS, ids=ids(CONFIGS))
@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("shape,pads", [((133, 97, 71), (3, 5, 7)),
                                        ((260, 300, 96), (4, 8, 4)),
                                        ((33, 17, 2100), (0, 1, 2))])
def test_checked_general_form_stays_inside_its_buffers(checked, cfg, ta, tb, shape, pads):
    if cfg.get("pack_a") == 4 and ta:
        pytest.skip("gathered K-major A needs A stored M x K")
    M, N, K = shape
    g = np.random.default_rng(M + 7 * N + 13 * K + 2 * ta + tb)
    lda = (M if ta else K) + pads[0]
    ldb = (K if tb else N) + pads[1]
    ldc = N + pads[2]
    A = stored(g, K if ta else M, M if ta else K, lda)
    B = stored(g, N if tb else K, K if tb else N, ldb)
    C0 = stored(g, M, N, ldc)
    bias = g.standard_normal(N).astype(np.float32)
    alpha, beta = 1.75, -0.5
    got = general(checked, ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C0, ldc, bias, **cfg)
    assert_clean(checked, f"{shape} {cfg} ta={ta} tb={tb}")
    want, W = oracle.sgemm_general(A, B, C0, M, N, K, lda, ldb, ldc, alpha, beta, ta, tb,
                                   with_w=True, bias=bias)
    want = want.reshape(M, ldc)
    err = np.abs(got[:, :N].astype(np.float64) - want[:, :N])
    assert np.all(err <= TOL * W)  # W counts |bias| too
    assert np.isnan(got[:, N:]).all()


def sampled(M, extra=24):
    g = np.random.default_rng(M)
    rows = {0, M - 1, M // 2} | set(g.integers(0, M, extra).tolist())
    return np.array(sorted(rows), np.int64)


@pytest.mark.parametrize("name", ["masked_100x72x80", "square_1024", "ragged_4097x3001x2053",
                                  "square_4096", "skinny_65536x128x4096"])
def test_checked_workloads_automatic_plans(checked, name):
    """The benchmark's and the parity tests' workloads in their automatic
    plans (transposing copy of A, gathered A, copied B, split tails)."""
    w = gemm_inputs.WORKLOADS[name]
    A, B = gemm_inputs.make_workload(w)
    a, b = A.cuda(), B.cuda()
    c = torch.full((w.M, w.N), float("nan"), device="cuda")
    st = checked.mt_sgemm(a.data_ptr(), b.data_ptr(), c.data_ptr(), w.M, w.N, w.K,
                          torch.cuda.current_stream().cuda_stream)
    assert st == mt.MT_OK
    torch.cuda.synchronize()
    assert_clean(checked, name)
    rows = sampled(w.M)
    Cr, Wr = oracle.sgemm_rows(A.numpy(), B.numpy(), rows, with_w=True)
    got = c[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - Cr) <= TOL * Wr), name
    # The same bits as the normal build (the checks change no arithmetic).
    ref = mt.sgemm(a, b)
    torch.cuda.synchronize()
    assert torch.equal(c, ref)


@pytest.mark.parametrize("cfg", [dict(), dict(variant="p18")], ids=["ffma", "p18"])
def test_checked_scaling_path_and_empty_product(checked, cfg):
    """K = 0 and alpha = 0 run the C scaling kernel (C = beta*C + bias)."""
    g = np.random.default_rng(3)
    M, N, ldc = 70, 45, 51
    C0 = stored(g, M, N, ldc)
    bias = g.standard_normal(N).astype(np.float32)
    A = np.zeros((M, 8), np.float32)
    B = np.zeros((8, N), np.float32)
    for K, alpha in ((0, 1.0), (8, 0.0)):
        got = general(checked, 0, 0, M, N, K, alpha, A, max(K, 1), B, N, 0.5, C0, ldc, bias,
                      **cfg)
        assert_clean(checked, f"K={K} alpha={alpha}")
        want = 0.5 * C0[:, :N].astype(np.float64) + bias[None, :]
        assert np.allclose(got[:, :N], want, rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("cfg,site", [(dict(), mt.MT_SITE_C_STORE),
                                      (dict(variant="p18"), mt.MT_SITE_P18)],
                         ids=["ffma", "p18"])
def test_checked_record_catches_a_planted_short_extent(checked, cfg, site, monkeypatch):
    """With C declared one element short (a host-side test hook of the
    checked build), the store of C's last element counts as outside: it is
    reported at the C store and skipped, and every other output is right."""
    M, N, K = 100, 72, 80
    A, B = gemm_inputs.make_workload("masked_100x72x80")
    a, b = A.cuda(), B.cuda()
    c = torch.full((M, N), float("nan"), device="cuda")
    conf = mt.make_config(**cfg) if cfg else None
    monkeypatch.setenv("MT_CHECKED_SHRINK_C_EXTENT", "1")
    st = checked.mt_sgemm_ex(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K,
                             torch.cuda.current_stream().cuda_stream,
                             ctypes.byref(conf) if conf is not None else None)
    monkeypatch.delenv("MT_CHECKED_SHRINK_C_EXTENT")
    assert st == mt.MT_OK
    torch.cuda.synchronize()
    rec = mt.bounds_status(checked)
    width = 1 if cfg else 4  # the FFMA kernel stores C in float4s here (N % 4 == 0)
    assert rec["count"] == 1, rec
    assert (rec["site"], rec["extent"], rec["offset"]) == (site, M * N - 1, M * N - width)
    got = c.cpu().numpy()
    assert np.isnan(got[-1, N - width:]).all()  # the skipped store
    Cref, W = oracle.sgemm(A.numpy(), B.numpy(), with_w=True)
    mask = np.ones((M, N), bool)
    mask[-1, N - width:] = False
    assert np.all(np.abs(got[mask].astype(np.float64) - Cref[mask]) <= TOL * W[mask])
    assert mt.bounds_status(checked)["count"] == 0  # the read cleared it
    assert os.environ.get("MT_CHECKED_SHRINK_C_EXTENT") is None


TC_TOL = 5e-5
TF32_CONFIGS = [dict(variant="tf32x3"), dict(variant="tf32x3", bn=64),
                dict(variant="tf32x3", bm=256), dict(variant="tf32x3", pack_a=1),
                dict(variant="tf32x3", pack_a=2),
                # stream-K runs: pieces in partial slots, added by the fix-up
                dict(variant="tf32x3", schedule=2), dict(variant="tf32x3", bm=256, schedule=2)]


@pytest.mark.parametrize("cfg", TF32_CONFIGS, ids=ids(TF32_CONFIGS))
@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("shape,pads", [((133, 97, 71), (3, 5, 7)),
                                        ((300, 520, 257), (4, 8, 4))])
def test_checked_tf32x3_stays_inside_its_buffers(checked, cfg, ta, tb, shape, pads):
    M, N, K = shape
    g = np.random.default_rng(11 * M + N + K + 2 * ta + tb)
    lda = (M if ta else K) + pads[0]
    ldb = (K if tb else N) + pads[1]
    ldc = N + pads[2]
    A = stored(g, K if ta else M, M if ta else K, lda)
    B = stored(g, N if tb else K, K if tb else N, ldb)
    C0 = stored(g, M, N, ldc)
    bias = g.standard_normal(N).astype(np.float32)
    got = general(checked, ta, tb, M, N, K, 1.25, A, lda, B, ldb, 0.5, C0, ldc, bias, **cfg)
    assert_clean(checked, f"{shape} {cfg} ta={ta} tb={tb}")
    want, W = oracle.sgemm_general(A, B, C0, M, N, K, lda, ldb, ldc, 1.25, 0.5, ta, tb,
                                   with_w=True, bias=bias)
    err = np.abs(got[:, :N].astype(np.float64) - want.reshape(M, ldc)[:, :N])
    assert np.all(err <= TC_TOL * W)
    assert np.isnan(got[:, N:]).all()


@pytest.mark.parametrize("name", ["square_4096", "skinny_65536x128x4096",
                                  "ragged_4097x3001x2053"])
def test_checked_tf32x3_workloads(checked, name):
    """Automatic 3xTF32 plans: CTA pairs with a split tail, the split-A
    kernel, padded packing of ragged operands."""
    w = gemm_inputs.WORKLOADS[name]
    A, B = gemm_inputs.make_workload(w)
    a, b = A.cuda(), B.cuda()
    c = torch.full((w.M, w.N), float("nan"), device="cuda")
    conf = mt.make_config(variant="tf32x3")
    st = checked.mt_sgemm_ex(a.data_ptr(), b.data_ptr(), c.data_ptr(), w.M, w.N, w.K,
                             torch.cuda.current_stream().cuda_stream, ctypes.byref(conf))
    assert st == mt.MT_OK
    torch.cuda.synchronize()
    assert_clean(checked, name)
    ref = mt.sgemm(a, b, variant="tf32x3")
    torch.cuda.synchronize()
    assert torch.equal(c, ref)  # the same bits as the normal build
    rows = sampled(w.M, extra=8)
    Cr, Wr = oracle.sgemm_rows(A.numpy(), B.numpy(), rows, with_w=True)
    got = c[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - Cr) <= TC_TOL * Wr), name


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("tile", [dict(), dict(bm=128), dict(bn=128), dict(bm=256),
                                  dict(bm=128, schedule=2), dict(bm=256, schedule=2)],
                         ids=["auto", "single", "bn128", "pair", "single-streamk",
                              "pair-streamk"])
@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 1)])
@pytest.mark.parametrize("lds", ["direct", "repack"])
def test_checked_16bit_inputs_stay_inside_their_buffers(checked, dt, tile, ta, tb, lds):
    """16-bit inputs read by TMA in place ("direct": row pitch a multiple
    of 8 elements) or first copied into padded scratch ("repack")."""
    code, tdt = {"bf16": (mt.MT_DTYPE_BF16, torch.bfloat16),
                 "f16": (mt.MT_DTYPE_F16, torch.float16)}[dt]
    M, N, K = 300, 520, 200
    g = np.random.default_rng(M + 3 * ta + tb + (lds == "repack"))

    def ld_for(cols):
        return (cols + 1 + 7) // 8 * 8 if lds == "direct" else cols + 3

    ra, ca = (K, M) if ta else (M, K)
    rb, cb = (N, K) if tb else (K, N)
    lda, ldb, ldc = ld_for(ca), ld_for(cb), N + 5
    A = torch.full((ra, lda), float("nan"), dtype=tdt)
    A[:, :ca] = torch.from_numpy(g.standard_normal((ra, ca)).astype(np.float32)).to(tdt)
    B = torch.full((rb, ldb), float("nan"), dtype=tdt)
    B[:, :cb] = torch.from_numpy(g.standard_normal((rb, cb)).astype(np.float32)).to(tdt)
    C0 = stored(g, M, N, ldc)
    bias = g.standard_normal(N).astype(np.float32)
    a, b, c = A.cuda(), B.cuda(), torch.from_numpy(C0).cuda()
    bz = torch.from_numpy(bias).cuda()
    conf = mt.make_config(**tile) if tile else None
    st = checked.mt_gemm_mixed_general_bias(code, ta, tb, M, N, K, 1.5, a.data_ptr(), lda,
                                            b.data_ptr(), ldb, -0.5, bz.data_ptr(),
                                            c.data_ptr(), ldc,
                                            torch.cuda.current_stream().cuda_stream,
                                            ctypes.byref(conf) if conf is not None else None)
    assert st == mt.MT_OK, mt.mt_status_string(st)
    torch.cuda.synchronize()
    assert_clean(checked, f"{dt} {tile} ta={ta} tb={tb} {lds}")
    want, W = oracle.gemm_mixed_general(code, A.view(torch.int16).numpy(),
                                        B.view(torch.int16).numpy(), C0, M, N, K, lda, ldb,
                                        ldc, 1.5, -0.5, ta, tb, with_w=True, bias=bias)
    got = c.cpu().numpy()
    err = np.abs(got[:, :N].astype(np.float64) - want.reshape(M, ldc)[:, :N])
    assert np.all(err <= TC_TOL * W)
    assert np.isnan(got[:, N:]).all()
