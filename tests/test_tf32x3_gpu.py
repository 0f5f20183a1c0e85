"""GPU parity of the tcgen05 3xTF32 variant against the CPU oracle.

Tolerance |C - C_ref| <= 5e-5 * W (W = |A|*|B|), elementwise.  Derivation:
each input is split exactly into big (tf32) + small; the dropped
small*small product and the tf32 conversion of the small parts each cost at
most about 2^-21 of |a||b| per product, and fp32 accumulation of random-sign
terms adds a few ulps of W — far inside 5e-5 * W.  Integer inputs in [-8, 8]
are exact in tf32 (small = 0) with integer partial sums below 2^24, so there
the result must be bit-exact.
"""
import numpy as np
import pytest
import torch

import gemm_inputs
import oracle
import tiled_fp32_gemm_gb300 as mt

pytestmark = pytest.mark.gpu

TOL = 5e-5
TF32 = dict(variant="tf32x3")


@pytest.fixture(scope="module", autouse=True)
def library():
    from tiled_fp32_gemm_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    return mt.lib()


def run(A, B, **cfg):
    c = mt.sgemm(A.cuda(), B.cuda(), **cfg)
    torch.cuda.synchronize()
    return c.cpu()


def assert_within(C, Cref, W, tol, what=""):
    C = np.asarray(C, np.float64)
    err = np.abs(C - np.asarray(Cref, np.float64))
    bad = err > tol * np.asarray(W, np.float64)
    if bad.any():
        i, j = np.argwhere(bad)[0]
        pytest.fail(f"{what}: {bad.sum()} outputs outside {tol}*W, first at ({i},{j}): "
                    f"got {C[i, j]!r} want {Cref[i, j]!r} W={W[i, j]!r}, "
                    f"max err/W {(err / np.maximum(W, 1e-300)).max():.3g}")


# Every configuration the kernel is built for: one CTA per 128 x bn tile,
# K depth 16 (64-byte swizzle) or 32 (128-byte swizzle) x tile width 256,
# 128 or 64; and CTA pairs on 256 x 256 tiles with K depth 16 or 32.
DEPTHS = [dict(variant="tf32x3", bm=128, bk=bk, bn=bn, pack_a=1) for bk in (16, 32)
          for bn in (256, 128, 64)]
DEPTH_IDS = [f"bk{c['bk']}-bn{c['bn']}" for c in DEPTHS]
PAIRS = [dict(variant="tf32x3", bm=256, bk=bk) for bk in (16, 32)]
PAIR_IDS = [f"pair-bk{c['bk']}" for c in PAIRS]
# A split inside the GEMM kernel (only B packed); A must be readable by TMA
# in place (K % 4 == 0 for packed rows).
ASPLIT = [dict(variant="tf32x3", bm=128, bk=bk, bn=bn, pack_a=2) for bk in (16, 32)
          for bn in (256, 128, 64)]
ASPLIT_IDS = [f"asplit-bk{c['bk']}-bn{c['bn']}" for c in ASPLIT]
ALL = DEPTHS + PAIRS + ASPLIT
ALL_IDS = DEPTH_IDS + PAIR_IDS + ASPLIT_IDS


def eligible(cfg, K):
    return cfg.get("pack_a") != 2 or K % 4 == 0


@pytest.mark.parametrize("cfg", DEPTHS, ids=DEPTH_IDS)
def test_plan_reports_tile_and_workspace(cfg):
    bk, bn = cfg["bk"], cfg["bn"]
    p = mt.plan(4096, 4096, 4096, **cfg)
    assert (p["bm"], p["bn"], p["bk"], p["threads"]) == (128, bn, bk, 192)
    assert p["stages"] >= 2
    # Packed big and small copies of A (128-row blocks) and B (bn-row
    # blocks), bk k each.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = 32 * (4096 // bn)
    ctas = min(tiles, sms)
    rem = tiles % ctas
    partial = rem * p["split_k"] * 128 * bn * 4 if p["split_k"] > 1 else 0
    assert p["workspace_bytes"] == 4096 * 4096 * 4 * 4 + partial
    units = tiles + (p["split_k"] - 1) * rem if p["split_k"] > 1 else tiles
    assert p["grid"] == min(units, sms)  # persistent: one CTA per SM at most
    auto = mt.plan(4096, 4096, 4096, variant="tf32x3")
    # The automatic choice for large squares: CTA pairs, K depth 16.
    assert (auto["bm"], auto["bn"], auto["bk"]) == (256, 256, 16)


@pytest.mark.parametrize("cfg", PAIRS, ids=PAIR_IDS)
def test_pair_plan_reports_tile_and_workspace(cfg):
    p = mt.plan(4096, 4096, 4096, **cfg)
    assert (p["bm"], p["bn"], p["bk"], p["threads"]) == (256, 256, cfg["bk"], 192)
    # Both operands packed in 128-row blocks (big and small): 2 x 4 bytes
    # per element of A and of B, plus the split tail's 256 x 256 partials.
    tiles = 16 * 16
    clusters = p["grid"] // 2
    rem = tiles % clusters if tiles > clusters else 0
    partial = rem * p["split_k"] * 256 * 256 * 4 if p["split_k"] > 1 else 0
    assert p["workspace_bytes"] == 2 * 2 * 4096 * 4096 * 4 + partial


@pytest.mark.parametrize("cfg", ALL, ids=ALL_IDS)
@pytest.mark.parametrize("name", ["masked_100x72x80", "square_1024", "ragged_4097x3001x2053"])
def test_workloads_full_oracle(name, cfg):
    if not eligible(cfg, gemm_inputs.WORKLOADS[name].K):
        pytest.skip("A's rows are not 16-byte multiples: split-A needs TMA on A")
    A, B = gemm_inputs.make_workload(name)
    Cref, W = oracle.sgemm(A.numpy(), B.numpy(), with_w=True)
    assert_within(run(A, B, **cfg).numpy(), Cref, W, TOL, name)


@pytest.mark.parametrize("split", [0, 1], ids=["auto-split-tail", "no-split"])
@pytest.mark.parametrize("tile", [0, 128], ids=["auto", "single"])
@pytest.mark.parametrize("name", ["square_4096", "square_8192", "skinny_65536x128x4096",
                                  "skinny_65536x128x4096/packed-A"])
def test_full_size_every_element(name, split, tile, full_oracle):
    name, _, how = name.partition("/")
    w = gemm_inputs.WORKLOADS[name]
    A, B = gemm_inputs.make_workload(w)
    pack = dict(pack_a=1) if how == "packed-A" else {}
    c = mt.sgemm(A.cuda(), B.cuda(), split_k=split, bm=tile, **TF32, **pack)
    if name.startswith("skinny"):
        assert mt.plan(w.M, w.N, w.K, bm=tile, **TF32, **pack)["pack_a"] == (1 if pack else 2)
    torch.cuda.synchronize()
    Cref, W = full_oracle(name)
    assert_within(c.cpu().numpy(), Cref, W, TOL, name)


@pytest.mark.parametrize("cfg", ALL, ids=ALL_IDS)
@pytest.mark.parametrize("shape", [(100, 72, 80), (257, 130, 77), (128, 256, 96),
                                   (300, 520, 1000)])
def test_integer_inputs_bit_exact(shape, cfg):
    M, N, K = shape
    if not eligible(cfg, K):
        pytest.skip("split-A needs K % 4 == 0 here")
    A, B = gemm_inputs.make_ab(M, N, K, seed=21, dist="int")
    assert np.array_equal(run(A, B, **cfg).numpy(), oracle.sgemm(A.numpy(), B.numpy()))


TINY = [(1, 1, 1), (1, 7, 3), (5, 1, 9), (3, 5, 7), (17, 15, 33), (31, 33, 1),
        (129, 257, 31), (130, 258, 65), (1, 1, 4), (5, 3, 8), (129, 257, 32), (130, 65, 36)]


@pytest.mark.parametrize("shape", TINY)
def test_tiny_ragged(shape):
    M, N, K = shape
    A, B = gemm_inputs.make_ab(M, N, K, seed=M * 7 + N * 3 + K, dist="normal")
    Cref, W = oracle.sgemm(A.numpy(), B.numpy(), with_w=True)
    for cfg in ALL:
        if eligible(cfg, K):
            assert_within(run(A, B, **cfg).numpy(), Cref, W, TOL, f"{shape} {cfg}")


def test_identity_within_tolerance():
    A = torch.randn(150, 97, generator=torch.Generator().manual_seed(3))
    C = run(A, torch.eye(97), **TF32).numpy()
    assert np.all(np.abs(C - A.numpy()) <= TOL * np.abs(A.numpy()))


@pytest.mark.parametrize("offset", [0, 1])
def test_guard_bands_and_canaries(offset):
    M, N, K = 133, 260, 72
    A, B = gemm_inputs.make_ab(M, N, K, seed=22, dist="uniform")
    guard = 4096
    abuf = torch.full((M * K + 2 * guard,), float("nan"))
    bbuf = torch.full((K * N + 2 * guard,), float("nan"))
    abuf[guard + offset:guard + offset + M * K] = A.reshape(-1)
    bbuf[guard + offset:guard + offset + K * N] = B.reshape(-1)
    sentinel = -12345.0
    cbuf = torch.full((M * N + 2 * guard,), sentinel, device="cuda")
    a_d, b_d = abuf.cuda(), bbuf.cuda()
    off = 4 * (guard + offset)
    st = mt.mt_sgemm_ex(a_d.data_ptr() + off, b_d.data_ptr() + off, cbuf.data_ptr() + off, M, N, K,
                        torch.cuda.current_stream().cuda_stream, mt.make_config(**TF32))
    assert st == mt.MT_OK
    torch.cuda.synchronize()
    out = cbuf.cpu()
    C = out[guard + offset:guard + offset + M * N].reshape(M, N).numpy()
    Cref, W = oracle.sgemm(A.numpy(), B.numpy(), with_w=True)
    assert np.isfinite(C).all()
    assert_within(C, Cref, W, TOL, "guarded")
    assert torch.all(out[:guard + offset] == sentinel)
    assert torch.all(out[guard + offset + M * N:] == sentinel)


def test_nan_propagates():
    A, B = gemm_inputs.make_ab(40, 36, 50, seed=23, dist="uniform")
    A[3, 7] = float("nan")
    C = run(A, B, **TF32).numpy()
    assert np.isnan(C[3]).all()
    assert np.isfinite(np.delete(C, 3, axis=0)).all()


def test_device_status_clean_after_runs():
    A, B = gemm_inputs.make_workload("masked_100x72x80")
    run(A, B, **TF32)
    assert mt.mt_device_status(0) == mt.MT_OK


@pytest.mark.parametrize("tile", [dict(bm=128, pack_a=1), dict(bm=256),
                                  dict(bm=128, bk=16, pack_a=2)], ids=["single", "pair", "asplit"])
def test_timeout_path_reports_and_context_survives(tile):
    """The copy threads issue nothing: every bounded wait runs out (about a
    second), the kernel records the timeout and returns; the context stays
    usable for the next call."""
    A, B = gemm_inputs.make_workload("masked_100x72x80")
    a, b = A.cuda(), B.cuda()
    c = torch.full((100, 72), 7.0, device="cuda")
    mt.sgemm(a, b, out=c, variant="tf32x3", fault_inject=1, **tile)
    assert mt.mt_check_device_status(0) == mt.MT_ERR_TIMEOUT
    assert torch.all(c == 7.0)  # nothing written
    assert mt.mt_check_device_status(0) == mt.MT_OK  # the status word was cleared
    # The earlier name is the same call: a second timeout shows through it.
    mt.sgemm(a, b, out=c, variant="tf32x3", fault_inject=1, **tile)
    assert mt.mt_device_status(0) == mt.MT_ERR_TIMEOUT
    assert mt.mt_check_device_status(0) == mt.MT_OK
    Cref, W = oracle.sgemm(A.numpy(), B.numpy(), with_w=True)
    assert_within(run(A, B, **TF32).numpy(), Cref, W, TOL, "after timeout")
    assert mt.mt_device_status(0) == mt.MT_OK


def test_split_tail_plan_and_parity():
    # 512 tiles of 128 x 256 on one CTA per SM leave a partial last round;
    # its tiles are cut into K slices whose partials a second kernel adds.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = mt.plan(4096, 4096, 4096, variant="tf32x3", bm=128)
    rem = 512 % sms
    if 0 < 2 * rem <= sms:
        assert p["split_k"] == min(sms // rem, 4)
    # 32 x 5 = 160 tiles: 152 in the first round, 8 split into 4 K slices.
    M, N, K = 4096, 1280, 520
    q = mt.plan(M, N, K, variant="tf32x3", bm=128)
    if sms == 152:
        assert (q["bn"], q["split_k"]) == (256, 4)
    A, B = gemm_inputs.make_ab(M, N, K, seed=24, dist="normal")
    rows = np.array([0, 1, 127, 128, 2047, 3968, 4095])
    Cr, Wr = oracle.sgemm_rows(A.numpy(), B.numpy(), rows, with_w=True)
    for cfg in (dict(bm=128), dict(bm=256)):
        got = run(A, B, **TF32, **cfg).numpy()[rows]
        assert_within(got, Cr, Wr, TOL, f"split tail {cfg}")
        assert np.array_equal(run(A, B, **TF32, **cfg).numpy()[rows], got)  # deterministic


@pytest.mark.parametrize("shape", [(512, 512, 4096), (300, 200, 5000)])
def test_small_grid_k_slices(shape):
    # Fewer tiles than half the SMs: K cut into slices of at least 1024,
    # added in slice order by the reduce; within the tolerance,
    # deterministic, and integer inputs exact.
    M, N, K = shape
    p = mt.plan(M, N, K, **TF32)
    assert p["split_k"] > 1
    A, B = gemm_inputs.make_ab(M, N, K, seed=23, dist="uniform")
    Cref, W = oracle.sgemm(A.numpy(), B.numpy(), with_w=True)
    got = run(A, B, **TF32).numpy()
    assert_within(got, Cref, W, TOL, f"{shape} small-grid split")
    assert np.array_equal(run(A, B, **TF32).numpy(), got)
    Ai, Bi = gemm_inputs.make_ab(M, N, K, seed=24, dist="int")
    assert np.array_equal(run(Ai, Bi, **TF32).numpy(), oracle.sgemm(Ai.numpy(), Bi.numpy()))
