"""GPU parity of the general form C = alpha*op(A)*op(B) + beta*C.

Leading dimensions, transposed storage and the alpha/beta update through
mt_sgemm_general, for every variant, against the oracle's general form
(oracle_sgemm_general: the same fp64 sum, one rounding).  Tolerance scale:
W = |alpha| * |op(A)|*|op(B)| + |beta| * |C|; FFMA and P18 within 1e-5 * W,
3xTF32 within 5e-5 * W, integer-valued inputs bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
import tiled_fp32_gemm_gb300 as mt

pytestmark = pytest.mark.gpu

VARIANTS = [(dict(), 1e-5), (dict(bm=128, bn=128), 1e-5), (dict(bm=64, bn=64), 1e-5),
            (dict(variant="p18"), 1e-5), (dict(variant="tf32x3"), 5e-5),
            (dict(variant="tf32x3", bn=64), 5e-5), (dict(variant="tf32x3", bm=256), 5e-5),
            (dict(pack_a=1), 1e-5), (dict(pack_a=2), 1e-5),
            (dict(pack_a=4), 1e-5), (dict(pack_a=5), 1e-5),
            (dict(bm=64, bn=128, pack_a=4), 1e-5), (dict(bm=64, bn=128, pack_a=5), 1e-5),
            (dict(bm=64, bn=64, pack_a=5), 1e-5), (dict(pack_a=4, split_k=3), 1e-5),
            (dict(bm=64, bn=128, stages=3, pack_a=4), 1e-5),
            (dict(bm=64, bn=128, stages=3, pack_a=5), 1e-5)]
VIDS = ["ffma", "ffma128", "ffma64", "p18", "tf32x3", "tf32x3-bn64", "tf32x3-pair",
        "ffma-copied", "ffma-rowmajor", "ffma-kgather", "ffma-kcopy", "ffma64x128-kgather",
        "ffma64x128-kcopy", "ffma64-kcopy", "ffma-kgather-split3", "ffma-kslices2-gather",
        "ffma-kslices2-copy"]


def supported(cfg, ta):
    """A gathered K-major A tile reads A stored M x K only."""
    return not (cfg.get("pack_a") == 4 and ta)


@pytest.fixture(scope="module", autouse=True)
def library():
    from tiled_fp32_gemm_gb300 import build
    build.build()
    return mt.lib()


def stored(g, rows, cols, ld, dist="normal"):
    """A rows x cols matrix inside a rows x ld buffer whose extra columns are NaN."""
    buf = np.full((rows, ld), np.nan, np.float32)
    if dist == "int":
        buf[:, :cols] = g.integers(-8, 9, (rows, cols))
    else:
        buf[:, :cols] = g.standard_normal((rows, cols))
    return buf


def run_general(ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C0, ldc, **cfg):
    a, b, c = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), torch.from_numpy(C0).cuda()
    st = mt.mt_sgemm_general(ta, tb, M, N, K, alpha, a.data_ptr(), lda, b.data_ptr(), ldb, beta,
                             c.data_ptr(), ldc, torch.cuda.current_stream().cuda_stream,
                             mt.make_config(**cfg) if cfg else None)
    assert st == mt.MT_OK, mt.mt_status_string(st)
    torch.cuda.synchronize()
    return c.cpu().numpy()


@pytest.mark.parametrize("cfg,tol", VARIANTS, ids=VIDS)
@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("shape,pads", [((133, 97, 71), (3, 5, 7)), ((260, 300, 96), (4, 8, 4)),
                                        ((31, 17, 300), (0, 1, 2))])
def test_general_matches_oracle(cfg, tol, ta, tb, shape, pads):
    if not supported(cfg, ta):
        pytest.skip("gathered K-major A needs A stored M x K")
    M, N, K = shape
    g = np.random.default_rng(M + 7 * N + 13 * K + 2 * ta + tb)
    lda = (M if ta else K) + pads[0]
    ldb = (K if tb else N) + pads[1]
    ldc = N + pads[2]
    A = stored(g, K if ta else M, M if ta else K, lda)
    B = stored(g, N if tb else K, K if tb else N, ldb)
    C0 = stored(g, M, N, ldc)
    alpha, beta = 1.75, -0.5
    got = run_general(ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C0, ldc, **cfg)
    want, W = oracle.sgemm_general(A, B, C0, M, N, K, lda, ldb, ldc, alpha, beta, ta, tb,
                                   with_w=True)
    want = want.reshape(M, ldc)
    err = np.abs(got[:, :N].astype(np.float64) - want[:, :N])
    assert np.all(err <= tol * W), f"max err/W {(err / np.maximum(W, 1e-30)).max():.3g}"
    assert np.isnan(got[:, N:]).all()  # C's padding columns untouched


@pytest.mark.parametrize("cfg,tol", VARIANTS, ids=VIDS)
def test_general_integers_exact(cfg, tol):
    M, N, K = 70, 90, 130
    g = np.random.default_rng(5)
    for ta, tb in [(0, 0), (1, 1)]:
        if not supported(cfg, ta):
            continue
        lda, ldb, ldc = (M if ta else K) + 2, (K if tb else N) + 3, N + 1
        A = stored(g, K if ta else M, M if ta else K, lda, "int")
        B = stored(g, N if tb else K, K if tb else N, ldb, "int")
        C0 = stored(g, M, N, ldc, "int")
        got = run_general(ta, tb, M, N, K, 2.0, A, lda, B, ldb, -3.0, C0, ldc, **cfg)
        want = oracle.sgemm_general(A, B, C0, M, N, K, lda, ldb, ldc, 2.0, -3.0, ta, tb)
        assert np.array_equal(got[:, :N], want.reshape(M, ldc)[:, :N])


@pytest.mark.parametrize("cfg,tol", VARIANTS, ids=VIDS)
def test_beta_zero_never_reads_c_and_alpha_zero_never_reads_ab(cfg, tol):
    M, N, K = 40, 44, 36
    g = np.random.default_rng(6)
    A = stored(g, M, K, K)
    B = stored(g, K, N, N)
    C0 = np.full((M, N), np.nan, np.float32)
    got = run_general(0, 0, M, N, K, 1.0, A, K, B, N, 0.0, C0, N, **cfg)
    want, W = oracle.sgemm(A, B, with_w=True)
    assert np.isfinite(got).all() and np.all(np.abs(got - want) <= tol * W)
    # alpha == 0: C = beta * C, A and B (all NaN here) are not read.
    Cb = stored(g, M, N, N)
    nanA = np.full((M, K), np.nan, np.float32)
    nanB = np.full((K, N), np.nan, np.float32)
    got = run_general(0, 0, M, N, K, 0.0, nanA, K, nanB, N, 0.5, Cb, N, **cfg)
    assert np.array_equal(got, (0.5 * Cb).astype(np.float32))
    # K == 0 with beta: the same.
    got = run_general(0, 0, M, N, 0, 1.0, A, 1, B, N, 2.0, Cb, N, **cfg)
    assert np.array_equal(got, (2.0 * Cb).astype(np.float32))


def test_packed_general_is_the_plain_call_bit_for_bit():
    M, N, K = 300, 260, 200
    g = np.random.default_rng(7)
    A = g.standard_normal((M, K)).astype(np.float32)
    B = g.standard_normal((K, N)).astype(np.float32)
    a, b = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    plain = mt.sgemm(a, b)
    general = mt.gemm(a, b)
    torch.cuda.synchronize()
    assert torch.equal(plain, general)


def test_torch_views_and_transposes():
    g = torch.Generator().manual_seed(8)
    big = torch.randn(300, 400, generator=g).cuda()
    a = big[10:110, 20:170]          # 100 x 150, row stride 400
    b = torch.randn(150, 90, generator=g).cuda()
    c = torch.zeros(100, 128).cuda()[:, :90]
    mt.gemm(a, b, c)
    at = a.t().contiguous()          # stored 150 x 100
    c2 = mt.gemm(at, b, trans_a=True)
    torch.cuda.synchronize()
    A, B = a.cpu().numpy(), b.cpu().numpy()
    want, W = oracle.sgemm(np.ascontiguousarray(A), np.ascontiguousarray(B), with_w=True)
    assert np.all(np.abs(c.cpu().numpy() - want) <= 1e-5 * W)
    assert np.all(np.abs(c2.cpu().numpy() - want) <= 1e-5 * W)


def test_ffma_transposes_need_a_tile_built_for_them():
    a = torch.zeros(64, 64, device="cuda")
    c = torch.zeros(64, 64, device="cuda")
    st = mt.mt_sgemm_general(1, 0, 64, 64, 64, 1.0, a.data_ptr(), 64, a.data_ptr(), 64, 0.0,
                             c.data_ptr(), 64, 0, mt.make_config(bm=256, bn=128))
    assert st == mt.MT_ERR_UNSUPPORTED


@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("shape", [(257, 130, 77), (300, 260, 200)])
def test_ffma_operand_copy_is_bit_identical(ta, tb, shape):
    """Copying operands into padded row-major scratch (pack_a = 1) changes
    the staging, not the arithmetic: the same FMA chain per output."""
    M, N, K = shape
    g = np.random.default_rng(M + N + K + ta + 2 * tb)
    lda, ldb, ldc = (M if ta else K) + 3, (K if tb else N) + 1, N + 2
    A = stored(g, K if ta else M, M if ta else K, lda)
    B = stored(g, N if tb else K, K if tb else N, ldb)
    C0 = stored(g, M, N, ldc)
    assert mt.plan(M, N, K, pack_a=1)["pack_a"] == (1 if (K % 4 or N % 4) else 0)
    copied = run_general(ta, tb, M, N, K, 1.25, A, lda, B, ldb, 0.5, C0, ldc, pack_a=1)
    stored_ = run_general(ta, tb, M, N, K, 1.25, A, lda, B, ldb, 0.5, C0, ldc, pack_a=2)
    assert np.array_equal(copied, stored_, equal_nan=True)
    want, W = oracle.sgemm_general(A, B, C0, M, N, K, lda, ldb, ldc, 1.25, 0.5, ta, tb,
                                   with_w=True)
    err = np.abs(copied.reshape(M, ldc)[:, :N].astype(np.float64) - want.reshape(M, ldc)[:, :N])
    assert np.all(err <= 1e-5 * W)


@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("shape,lda_pad", [((257, 130, 77), 3), ((300, 260, 200), 0),
                                           ((1000, 2200, 96), 4)])
@pytest.mark.parametrize("tile", [dict(), dict(bm=64, bn=128), dict(bm=64, bn=64)],
                         ids=["128x128", "64x128", "64x64"])
def test_ffma_kmajor_a_is_bit_identical(ta, tb, shape, lda_pad, tile):
    """A staged K-major (read as stored K x M, gathered from M x K inside
    the kernel, or from a K x M copy) changes which rows a float4 holds, not
    the arithmetic: every source gives the row-major tiles' FMA chain bit for
    bit.  Padding columns of A hold NaN: a 16-byte chunk that reaches past M
    only feeds rows that are never stored."""
    M, N, K = shape
    g = np.random.default_rng(M + N + K + ta + 2 * tb)
    lda, ldb, ldc = (M if ta else K) + lda_pad, (K if tb else N) + 1, N + 2
    A = stored(g, K if ta else M, M if ta else K, lda)
    B = stored(g, N if tb else K, K if tb else N, ldb)
    C0 = stored(g, M, N, ldc)
    # Reference: row-major A tiles of the default tile, staged as stored.
    # Every FFMA tile sums each output over k in order with one fused
    # multiply-add per k, so the tile does not change the bits either.
    ref = run_general(ta, tb, M, N, K, 1.25, A, lda, B, ldb, 0.5, C0, ldc, pack_a=2)
    for pack in (3, 4, 5):
        if pack == 4 and ta:
            continue
        got = run_general(ta, tb, M, N, K, 1.25, A, lda, B, ldb, 0.5, C0, ldc, pack_a=pack,
                          **tile)
        assert np.array_equal(got, ref, equal_nan=True), pack
    want, W = oracle.sgemm_general(A, B, C0, M, N, K, lda, ldb, ldc, 1.25, 0.5, ta, tb,
                                   with_w=True)
    err = np.abs(ref.reshape(M, ldc)[:, :N].astype(np.float64) - want.reshape(M, ldc)[:, :N])
    assert np.all(err <= 1e-5 * W)


@pytest.mark.parametrize("cfg,tol", VARIANTS, ids=VIDS)
@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 1)])
def test_bias_epilogue_matches_oracle(cfg, tol, ta, tb):
    """C = alpha*op(A)*op(B) + beta*C + bias[j], bias fused into every
    variant's epilogue (and its K-slice reduce).  Tolerance scale W grows by
    |bias[j]|; integer inputs are exact."""
    if not supported(cfg, ta):
        pytest.skip("gathered K-major A needs A stored M x K")
    M, N, K = 133, 97, 71
    g = np.random.default_rng(40 + 2 * ta + tb)
    lda, ldb, ldc = (M if ta else K) + 3, (K if tb else N) + 5, N + 7
    A = stored(g, K if ta else M, M if ta else K, lda)
    B = stored(g, N if tb else K, K if tb else N, ldb)
    C0 = stored(g, M, N, ldc)
    bias = g.standard_normal(N).astype(np.float32)
    a, b, c = (torch.from_numpy(x).cuda() for x in (A, B, C0))
    bias_d = torch.from_numpy(bias).cuda()
    st = mt.mt_sgemm_general_bias(ta, tb, M, N, K, 1.75, a.data_ptr(), lda, b.data_ptr(), ldb,
                                  -0.5, bias_d.data_ptr(), c.data_ptr(), ldc,
                                  torch.cuda.current_stream().cuda_stream,
                                  mt.make_config(**cfg))
    assert st == mt.MT_OK, mt.mt_status_string(st)
    got = c.cpu().numpy()
    want, W = oracle.sgemm_general(A, B, C0, M, N, K, lda, ldb, ldc, 1.75, -0.5, ta, tb,
                                   with_w=True, bias=bias)
    err = np.abs(got[:, :N].astype(np.float64) - want.reshape(M, ldc)[:, :N])
    assert np.all(err <= tol * W), f"max err/W {(err / np.maximum(W, 1e-30)).max():.3g}"
    assert np.isnan(got[:, N:]).all()
    # Integer inputs: exact.
    Ai = stored(g, K if ta else M, M if ta else K, lda, "int")
    Bi = stored(g, N if tb else K, K if tb else N, ldb, "int")
    Ci = stored(g, M, N, ldc, "int")
    bi = g.integers(-9, 10, N).astype(np.float32)
    # Device copies held in names for the whole call (a temporary's memory
    # could be handed to the next allocation before the kernel reads it).
    ai, bi_, biasi, c = (torch.from_numpy(x).cuda() for x in (Ai, Bi, bi, Ci))
    st = mt.mt_sgemm_general_bias(ta, tb, M, N, K, 2.0, ai.data_ptr(), lda, bi_.data_ptr(), ldb,
                                  -3.0, biasi.data_ptr(), c.data_ptr(), ldc,
                                  torch.cuda.current_stream().cuda_stream,
                                  mt.make_config(**cfg))
    torch.cuda.synchronize()
    assert st == mt.MT_OK
    want = oracle.sgemm_general(Ai, Bi, Ci, M, N, K, lda, ldb, ldc, 2.0, -3.0, ta, tb, bias=bi)
    assert np.array_equal(c.cpu().numpy()[:, :N], want.reshape(M, ldc)[:, :N])


@pytest.mark.parametrize("shape", [(4096, 4096, 4096), (65536, 128, 4096)])
def test_bias_on_split_plans_and_empty_product(shape):
    """The automatic plans of the benchmark shapes (K-major A, K slices in
    the last partial wave, the transposing copy) with a bias, on sampled
    rows; alpha = 0 and K = 0 give beta*C + bias."""
    M, N, K = shape
    g = torch.Generator().manual_seed(41)
    A = torch.rand(M, K, generator=g) * 2 - 1
    B = torch.rand(K, N, generator=g) * 2 - 1
    bias = torch.randn(N, generator=g)
    a, b, bd = A.cuda(), B.cuda(), bias.cuda()
    c = mt.gemm(a, b, bias=bd)
    torch.cuda.synchronize()
    rows = np.array(sorted({0, 1, 127, 128, M // 2, M - 1}))
    Cr, Wr = oracle.sgemm_rows(A.numpy(), B.numpy(), rows, with_w=True)
    got = c[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64)
    want = Cr.astype(np.float64) + bias.numpy()[None, :]
    assert np.all(np.abs(got - want) <= 1e-5 * (Wr + np.abs(bias.numpy())[None, :]) + 1e-7)
    c0 = torch.randn(64, 48, generator=g).cuda()
    bd2 = torch.randn(48, generator=g).cuda()
    x = torch.zeros(64, 0, device="cuda")
    y = torch.zeros(0, 48, device="cuda")
    out = mt.gemm(x, y, c0.clone(), beta=0.5, bias=bd2)
    torch.cuda.synchronize()
    assert torch.equal(out, 0.5 * c0 + bd2)


def test_binding_refuses_operands_off_the_device():
    """A host c (or bias) beside device operands is refused before any call:
    its pointer would otherwise reach a kernel."""
    a = torch.zeros((8, 4), device="cuda")
    b = torch.zeros((4, 6), device="cuda")
    with pytest.raises(TypeError):
        mt.gemm(a, b, c=torch.zeros((8, 6)))
    with pytest.raises((TypeError, ValueError)):
        mt.gemm(a, b, bias=torch.zeros(6))
    with pytest.raises(TypeError):
        mt.sgemm(a, b, out=torch.zeros((8, 6)))
    a16, b16 = a.to(torch.bfloat16), b.to(torch.bfloat16)
    with pytest.raises(TypeError):
        mt.gemm_mixed(a16, b16, c=torch.zeros((8, 6)))
