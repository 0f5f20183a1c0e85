"""GPU parity of the 16-bit-input product (mt_gemm_mixed*, tcgen05 kind::f16).

C = alpha * op(A) * op(B) + beta * C with A and B stored as fp16 or bf16 and
C in fp32, against the oracle's oracle_gemm_mixed_general (the values the
16-bit patterns encode, an fp64 sum, one rounding).  Both sides read the same
16-bit patterns.  Tolerance scale W = |alpha| * |op(A)|*|op(B)| + |beta| * |C|:
within 5e-5 * W, the bar of the other tensor-core path (a product of two
16-bit values is exact in fp32, so only the fp32 accumulation rounds), and
bit-exact on integer-valued inputs.

Operands are read by TMA in place when their row pitch is a multiple of 8
elements and their base 16-byte aligned ("direct"); otherwise the call copies
them into padded scratch first ("repack").  Both paths are covered.
"""
import numpy as np
import pytest
import torch

import gemm_inputs
import oracle
import tiled_fp32_gemm_gb300 as mt

pytestmark = pytest.mark.gpu

TOL = 5e-5
# Tile plans: automatic, one CTA per 128 x 256 or 128 x 128 tile, a CTA pair
# per 256 x 256 tile (cta_group::2).
TILES = {"auto": {}, "single": dict(bm=128), "bn128": dict(bn=128), "pair": dict(bm=256)}
DTYPES = {"bf16": (mt.MT_DTYPE_BF16, torch.bfloat16), "f16": (mt.MT_DTYPE_F16, torch.float16)}
assert (oracle.F16, oracle.BF16) == (mt.MT_DTYPE_F16, mt.MT_DTYPE_BF16)


@pytest.fixture(scope="module", autouse=True)
def library():
    from tiled_fp32_gemm_gb300 import build
    build.build()
    return mt.lib()


def draw(g, shape, dist):
    if dist == "int":
        return g.integers(-8, 9, shape).astype(np.float32)
    return g.standard_normal(shape).astype(np.float32)


def stored16(g, rows, cols, ld, tdt, dist="normal"):
    """A rows x cols 16-bit matrix inside a rows x ld buffer; the extra
    columns hold NaN (must never be read)."""
    buf = torch.full((rows, ld), float("nan"), dtype=tdt)
    buf[:, :cols] = torch.from_numpy(draw(g, (rows, cols), dist)).to(tdt)
    return buf


def ld_for(cols, path):
    if path == "direct":
        return (cols + 1 + 7) // 8 * 8
    ld = cols + 3
    return ld + 1 if ld % 8 == 0 else ld


def run_mixed(code, ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C0, ldc, **cfg):
    a, b, c = A.cuda(), B.cuda(), torch.from_numpy(C0).cuda()
    st = mt.mt_gemm_mixed_general(code, ta, tb, M, N, K, alpha, a.data_ptr(), lda,
                                  b.data_ptr(), ldb, beta, c.data_ptr(), ldc,
                                  torch.cuda.current_stream().cuda_stream,
                                  mt.make_config(**cfg) if cfg else None)
    assert st == mt.MT_OK, mt.mt_status_string(st)
    assert mt.mt_device_status(0) == mt.MT_OK
    return c.cpu().numpy()


def assert_within(got, want, W, what=""):
    err = np.abs(got.astype(np.float64) - want.astype(np.float64))
    ratio = (err / np.maximum(W, 1e-30)).max() if err.size else 0.0
    assert np.all(err <= TOL * W), f"{what}: max err/W {ratio:.3g}"


@pytest.mark.parametrize("dt", sorted(DTYPES))
@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("path", ["direct", "repack"])
@pytest.mark.parametrize("shape", [(133, 97, 71), (260, 300, 200), (31, 17, 300)])
@pytest.mark.parametrize("tile", sorted(TILES))
def test_mixed_matches_oracle(dt, ta, tb, path, shape, tile):
    code, tdt = DTYPES[dt]
    M, N, K = shape
    g = np.random.default_rng(M + 7 * N + 13 * K + 2 * ta + tb + (path == "direct"))
    a_rows, a_cols = (K, M) if ta else (M, K)
    b_rows, b_cols = (N, K) if tb else (K, N)
    lda, ldb, ldc = ld_for(a_cols, path), ld_for(b_cols, path), N + 3
    A = stored16(g, a_rows, a_cols, lda, tdt)
    B = stored16(g, b_rows, b_cols, ldb, tdt)
    C0 = np.full((M, ldc), np.nan, np.float32)
    C0[:, :N] = draw(g, (M, N), "normal")
    alpha, beta = 1.75, -0.5
    cfg = TILES[tile]
    p = mt.plan_mixed(code, M, N, K, ta, tb, lda, ldb, ldc, **cfg)
    assert p["vec_ab"] == (1 if path == "direct" else 0)
    got = run_mixed(code, ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C0, ldc, **cfg)
    want, W = oracle.gemm_mixed_general(code, A, B, C0, M, N, K, lda, ldb, ldc, alpha, beta,
                                        ta, tb, with_w=True)
    want = want.reshape(M, ldc)
    assert_within(got[:, :N], want[:, :N], W, f"{dt} ta={ta} tb={tb} {path}")
    assert np.isnan(got[:, N:]).all()  # C's padding columns untouched


@pytest.mark.parametrize("dt", sorted(DTYPES))
@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 1)])
@pytest.mark.parametrize("tile", sorted(TILES))
def test_mixed_integers_exact(dt, ta, tb, tile):
    code, tdt = DTYPES[dt]
    M, N, K = 300, 264, 1000
    g = np.random.default_rng(11 + ta)
    a_rows, a_cols = (K, M) if ta else (M, K)
    b_rows, b_cols = (N, K) if tb else (K, N)
    A = stored16(g, a_rows, a_cols, a_cols, tdt, "int")
    B = stored16(g, b_rows, b_cols, b_cols, tdt, "int")
    C0 = draw(g, (M, N), "int")
    got = run_mixed(code, ta, tb, M, N, K, 2.0, A, a_cols, B, b_cols, -3.0, C0, N, **TILES[tile])
    want = oracle.gemm_mixed_general(code, A, B, C0, M, N, K, a_cols, b_cols, N, 2.0, -3.0,
                                     ta, tb).reshape(M, N)
    assert np.array_equal(got, want)


def rows_of(A, rows):
    return A[rows].contiguous()


@pytest.mark.parametrize("dt", sorted(DTYPES))
@pytest.mark.parametrize("name", ["masked_100x72x80", "square_1024", "ragged_4097x3001x2053"])
def test_mixed_workloads(dt, name):
    """The packed call (mt_gemm_mixed through gemm_mixed) on the named
    workloads' inputs rounded to 16 bits; full comparison on the small one,
    sampled rows (first, last and random) on the others."""
    code, tdt = DTYPES[dt]
    w = gemm_inputs.WORKLOADS[name]
    A, B = gemm_inputs.make_ab16(w.M, w.N, w.K, w.seed, w.dist, dt)
    got = mt.gemm_mixed(A.cuda(), B.cuda()).cpu().numpy()
    assert mt.mt_device_status(0) == mt.MT_OK
    if w.M * w.N * w.K <= 1 << 24:
        rows = np.arange(w.M)
    else:
        g = np.random.default_rng(w.seed)
        rows = np.unique(np.concatenate([[0, w.M - 1], g.integers(0, w.M, 62)]))
    As = rows_of(A, torch.from_numpy(rows))
    want, W = oracle.gemm_mixed_general(code, As, B, np.zeros(len(rows) * w.N, np.float32),
                                        len(rows), w.N, w.K, w.K, w.N, w.N, with_w=True)
    assert_within(got[rows], want.reshape(len(rows), w.N), W, name)


@pytest.mark.parametrize("dt", sorted(DTYPES))
@pytest.mark.parametrize("tile", ["auto", "single"])
def test_mixed_bench_size_sampled(dt, tile):
    """8192^3 in the launch configuration the benchmark times (packed rows,
    automatic plan with its split tail), checked on sampled rows."""
    code, tdt = DTYPES[dt]
    w = gemm_inputs.WORKLOADS["square_8192"]
    A, B = gemm_inputs.make_ab16(w.M, w.N, w.K, w.seed, w.dist, dt)
    a, b = A.cuda(), B.cuda()
    c = mt.gemm_mixed(a, b, **TILES[tile])
    assert mt.mt_device_status(0) == mt.MT_OK
    p = mt.plan_mixed(code, w.M, w.N, w.K, a=a, b=b, c=c, **TILES[tile])
    assert p["vec_ab"] == 1 and p["split_k"] >= 1
    g = np.random.default_rng(3)
    # Rows of the first tile row, the split tail's last tile row and random ones.
    rows = np.unique(np.concatenate([[0, 127, 128, 255, w.M - 1], g.integers(0, w.M, 13)]))
    got = c.cpu().numpy()[rows]
    As = rows_of(A, torch.from_numpy(rows))
    want, W = oracle.gemm_mixed_general(code, As, B, np.zeros(len(rows) * w.N, np.float32),
                                        len(rows), w.N, w.K, w.K, w.N, w.N, with_w=True)
    assert_within(got, want.reshape(len(rows), w.N), W, "8192^3")


@pytest.mark.parametrize("dt", sorted(DTYPES))
@pytest.mark.parametrize("tile", ["single", "pair"])
def test_mixed_split_tail_deterministic(dt, tile):
    """512 tiles of 128 x 256 leave a partial round that is split along K;
    the slices are added in a fixed order, so repeated calls agree bit for
    bit, and both the split and the unsplit call match the oracle."""
    code, tdt = DTYPES[dt]
    M, N, K = 4096, 4096, 640
    A, B = gemm_inputs.make_ab16(M, N, K, 21, "normal", dt)
    a, b = A.cuda(), B.cuda()
    cfg = TILES[tile]
    p = mt.plan_mixed(code, M, N, K, a=a, b=b, **cfg)
    tiles = (M // p["bm"]) * (N // p["bn"])
    units = p["grid"] // (2 if p["bm"] == 256 else 1)
    if 0 < 2 * (tiles % units) <= units:
        assert p["split_k"] > 1
    c1 = mt.gemm_mixed(a, b, **cfg)
    c2 = mt.gemm_mixed(a, b, **cfg)
    c3 = mt.gemm_mixed(a, b, split_k=1, **cfg)
    assert mt.mt_device_status(0) == mt.MT_OK
    assert torch.equal(c1, c2)
    # 3840.. is the last row of 256-row tiles, 3968.. of 128-row tiles.
    rows = np.array([0, 1, 130, 2047, 3900, 3968, 4000, 4095])
    As = rows_of(A, torch.from_numpy(rows))
    want, W = oracle.gemm_mixed_general(code, As, B, np.zeros(len(rows) * N, np.float32),
                                        len(rows), N, K, K, N, N, with_w=True)
    for c in (c1, c3):
        assert_within(c.cpu().numpy()[rows], want.reshape(len(rows), N), W, "split tail")


@pytest.mark.parametrize("dt", sorted(DTYPES))
def test_mixed_edge_cases(dt):
    code, tdt = DTYPES[dt]
    g = np.random.default_rng(9)
    s = torch.cuda.current_stream().cuda_stream
    # K == 0: C = beta * C; alpha == 0: A and B (NaN here) are not read.
    C0 = draw(g, (5, 7), "normal")
    c = torch.from_numpy(C0).cuda()
    nan = torch.full((64,), float("nan"), dtype=tdt, device="cuda")
    assert mt.mt_gemm_mixed_general(code, 0, 0, 5, 7, 0, 1.0, nan.data_ptr(), 1,
                                    nan.data_ptr(), 7, 2.0, c.data_ptr(), 7, s, None) == mt.MT_OK
    assert np.array_equal(c.cpu().numpy(), (2.0 * C0).astype(np.float32))
    assert mt.mt_gemm_mixed_general(code, 0, 0, 5, 7, 4, 0.0, nan.data_ptr(), 4,
                                    nan.data_ptr(), 7, 0.5, c.data_ptr(), 7, s, None) == mt.MT_OK
    assert np.array_equal(c.cpu().numpy(), (0.5 * (2.0 * C0).astype(np.float32)))
    # Thin shapes: one row, one column, K shorter than one 64-deep stage,
    # K just past one stage.
    for M, N, K in [(1, 300, 130), (300, 1, 130), (129, 257, 1), (64, 64, 65), (200, 8, 63)]:
        A = torch.from_numpy(draw(g, (M, K), "normal")).to(tdt)
        B = torch.from_numpy(draw(g, (K, N), "normal")).to(tdt)
        got = mt.gemm_mixed(A.cuda(), B.cuda()).cpu().numpy()
        want, W = oracle.gemm_mixed_general(code, A, B, np.zeros(M * N, np.float32), M, N, K,
                                            K, N, N, with_w=True)
        assert_within(got, want.reshape(M, N), W, f"{M}x{N}x{K}")
    # A 2-byte-aligned (not 16-byte) base takes the copy path.
    M, N, K = 70, 90, 96
    A = torch.from_numpy(draw(g, (M * K + 1,), "normal")).to(tdt).cuda()
    B = torch.from_numpy(draw(g, (K, N), "normal")).to(tdt).cuda()
    a = A[1:].view(M, K)
    p = mt.plan_mixed(code, M, N, K, a=a, b=B)
    assert p["vec_ab"] == 0
    got = mt.gemm_mixed(a, B).cpu().numpy()
    want, W = oracle.gemm_mixed_general(code, a.cpu(), B.cpu(), np.zeros(M * N, np.float32),
                                        M, N, K, K, N, N, with_w=True)
    assert_within(got, want.reshape(M, N), W, "offset base")
    assert mt.mt_device_status(0) == mt.MT_OK


@pytest.mark.parametrize("tile", ["single", "pair"])
def test_mixed_timeout_path_reports_and_context_survives(tile):
    """The copy threads issue nothing: every bounded wait runs out (about a
    second), the kernel records the timeout and returns; the context stays
    usable for the next call."""
    A, B = gemm_inputs.make_ab16(100, 72, 80, 0, "uniform", "bf16")
    a, b = A.cuda(), B.cuda()
    c = torch.full((100, 72), 7.0, device="cuda")
    mt.gemm_mixed(a, b, c, fault_inject=1, **TILES[tile])
    assert mt.mt_device_status(0) == mt.MT_ERR_TIMEOUT
    assert torch.all(c == 7.0)
    assert mt.mt_device_status(0) == mt.MT_OK
    got = mt.gemm_mixed(a, b, **TILES[tile]).cpu().numpy()
    want, W = oracle.gemm_mixed_general(oracle.BF16, A, B, np.zeros(100 * 72, np.float32),
                                        100, 72, 80, 80, 72, 72, with_w=True)
    assert_within(got, want.reshape(100, 72), W, "after timeout")
    assert mt.mt_device_status(0) == mt.MT_OK


@pytest.mark.parametrize("dt", sorted(DTYPES))
@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 1)])
@pytest.mark.parametrize("tile", sorted(TILES))
def test_mixed_bias_epilogue(dt, ta, tb, tile):
    """The bias row on 16-bit inputs (mt_gemm_mixed_general_bias): integer
    inputs exact; normal inputs within 5e-5 * (W + |bias|), on every tile
    and its split tail."""
    code, tdt = DTYPES[dt]
    M, N, K = 300, 264, 1000
    g = np.random.default_rng(21 + ta)
    a_rows, a_cols = (K, M) if ta else (M, K)
    b_rows, b_cols = (N, K) if tb else (K, N)
    for dist in ("int", "normal"):
        A = stored16(g, a_rows, a_cols, a_cols, tdt, dist)
        B = stored16(g, b_rows, b_cols, b_cols, tdt, dist)
        C0 = draw(g, (M, N), dist)
        bias = draw(g, (N,), dist)
        a, b, c, bd = A.cuda(), B.cuda(), torch.from_numpy(C0).cuda(), torch.from_numpy(bias).cuda()
        st = mt.mt_gemm_mixed_general_bias(code, ta, tb, M, N, K, 2.0, a.data_ptr(), a_cols,
                                           b.data_ptr(), b_cols, -3.0, bd.data_ptr(),
                                           c.data_ptr(), N, torch.cuda.current_stream().cuda_stream,
                                           mt.make_config(**TILES[tile]) if TILES[tile] else None)
        assert st == mt.MT_OK, mt.mt_status_string(st)
        got = c.cpu().numpy()
        want, W = oracle.gemm_mixed_general(code, A, B, C0, M, N, K, a_cols, b_cols, N, 2.0,
                                            -3.0, ta, tb, with_w=True, bias=bias)
        want = want.reshape(M, N)
        if dist == "int":
            assert np.array_equal(got, want)
        else:
            assert_within(got, want, W, f"bias {dt} {tile}")
    # The same through the torch-level call.
    out = mt.gemm_mixed(a, b, trans_a=bool(ta), trans_b=bool(tb), bias=bd, **TILES[tile])
    want0, W0 = oracle.gemm_mixed_general(code, A, B, np.zeros(M * N, np.float32), M, N, K,
                                          a_cols, b_cols, N, 1.0, 0.0, ta, tb, with_w=True,
                                          bias=bias)
    assert_within(out.cpu().numpy(), want0.reshape(M, N), W0, "gemm_mixed bias")


@pytest.mark.parametrize("shape", [(512, 512, 4096), (300, 200, 5000)])
def test_mixed_small_grid_k_slices(shape):
    # Fewer tiles than half the SMs: K cut into slices of at least 1024.
    M, N, K = shape
    p = mt.plan_mixed(mt.MT_DTYPE_BF16, M, N, K)
    assert p["split_k"] > 1
    A16, B16 = gemm_inputs.make_ab16(M, N, K, 25, "uniform", "bf16")
    Cref, W = oracle.gemm_mixed_general(oracle.BF16, A16, B16, np.zeros(M * N, np.float32),
                                        M, N, K, K, N, N, with_w=True)
    a, b = A16.cuda(), B16.cuda()
    got = mt.gemm_mixed(a, b)
    again = mt.gemm_mixed(a, b)
    torch.cuda.synchronize()
    assert_within(got.cpu().numpy(), Cref.reshape(M, N), W.reshape(M, N), f"{shape}")
    assert torch.equal(got, again)
