"""GPU parity of the stream-K schedule (FFMA and tensor-core kernels) against the CPU oracle.

Stream-K (mt_config.schedule = 2) spreads the K tiles of the tiles past the
last whole wave over one wave of CTAs, each taking a contiguous run across
tile boundaries; a second kernel adds the pieces of every tile that no run
covered whole, in k order.  Each output is then a sum of a few fp32 FMA
chains over consecutive k ranges: within the FFMA tolerance 1e-5 * |A|*|B|
of the oracle, bit-exact on integer inputs (every partial sum is an integer
below 2^24), and the same bits on every run (the order of the additions is
fixed by the plan, not by scheduling).
"""
import numpy as np
import pytest
import torch

import gemm_inputs
import oracle
import tiled_fp32_gemm_gb300 as mt

pytestmark = pytest.mark.gpu

TOL = 1e-5
SK = dict(schedule="stream_k")
# Tiles with every K-major A source and the row-major A tile.
TILES = [
    dict(),                                                   # automatic tile
    dict(bm=128, bn=128, bk=16, stages=4, wm=64, pack_a=5),   # A from a K x M copy
    dict(bm=128, bn=128, bk=16, stages=4, wm=64, pack_a=4),   # A gathered
    dict(bm=64, bn=128, bk=32, stages=2, pack_a=4),
    dict(bm=128, bn=128, bk=32, stages=3, fma=2, pack_a=2),   # row-major A tiles
    dict(bm=64, bn=64, pack_a=5),
]
TILE_IDS = ["-".join(f"{k}{v}" for k, v in c.items()) or "auto" for c in TILES]


@pytest.fixture(scope="module", autouse=True)
def library():
    from tiled_fp32_gemm_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    return mt.lib()


def run(a, b, **cfg):
    c = mt.sgemm(a, b, **cfg)
    torch.cuda.synchronize()
    return c.cpu().numpy()


def assert_within(C, Cref, W, what):
    err = np.abs(np.asarray(C, np.float64) - Cref)
    bad = err > TOL * W
    if bad.any():
        i, j = np.argwhere(bad)[0]
        pytest.fail(f"{what}: {bad.sum()} outputs outside {TOL}*W, first at ({i},{j}): "
                    f"got {C[i, j]!r} want {Cref[i, j]!r} W={W[i, j]!r}")


@pytest.mark.parametrize("cfg", TILES, ids=TILE_IDS)
@pytest.mark.parametrize("name", ["masked_100x72x80", "square_1024", "ragged_4097x3001x2053"])
def test_stream_k_workloads_full_oracle(name, cfg, full_oracle):
    A, B = gemm_inputs.make_workload(name)
    a, b = A.cuda(), B.cuda()
    w = gemm_inputs.WORKLOADS[name]
    p = mt.plan(w.M, w.N, w.K, a=a, b=b, **SK, **cfg)
    assert p["stream_k"] > 0 and p["split_k"] == 1
    got = run(a, b, **SK, **cfg)
    Cref, W = full_oracle(name)
    assert_within(got, Cref, W, f"{name} {cfg}")
    # Deterministic: the same bits again.
    assert np.array_equal(run(a, b, **SK, **cfg), got)


@pytest.mark.parametrize("name", ["square_4096", "skinny_65536x128x4096"])
def test_stream_k_large_workloads_every_element(name, full_oracle):
    A, B = gemm_inputs.make_workload(name)
    got = run(A.cuda(), B.cuda(), **SK)
    Cref, W = full_oracle(name)
    assert_within(got, Cref, W, name)


@pytest.mark.parametrize("cfg", TILES, ids=TILE_IDS)
@pytest.mark.parametrize("shape", [(100, 72, 80), (257, 130, 77), (1024, 1024, 1024),
                                   (1000, 1000, 1200)])
def test_stream_k_integer_inputs_bit_exact(shape, cfg):
    M, N, K = shape
    A, B = gemm_inputs.make_ab(M, N, K, seed=11, dist="int")
    Cref = oracle.sgemm(A.numpy(), B.numpy())
    assert np.array_equal(run(A.cuda(), B.cuda(), **SK, **cfg), Cref)


def test_stream_k_runs_across_tile_boundaries():
    # 1024^3 on 128 x 128 tiles: 64 tiles of 64 K tiles over one wave of
    # CTAs, so every tile is cut into pieces taken by several CTAs and
    # most CTAs start or end inside a tile.
    cfg = dict(bm=128, bn=128, bk=16, stages=4, wm=64, pack_a=5, **SK)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = mt.plan(1024, 1024, 1024, **cfg)
    assert p["stream_k"] == min(2 * sms, 64 * 64 // 2) and p["grid"] == p["stream_k"]
    # Two partial slots per stream-K CTA, after the copy of A.
    assert p["workspace_bytes"] >= 2 * p["stream_k"] * 128 * 128 * 4
    A, B = gemm_inputs.make_ab(1024, 1024, 1024, seed=21, dist="uniform")
    Cref, W = oracle.sgemm(A.numpy(), B.numpy(), with_w=True)
    assert_within(run(A.cuda(), B.cuda(), **cfg), Cref, W, "1024^3 128x128 stream-K")


def test_stream_k_runs_shorter_than_a_tile_and_empty_runs():
    # Few K tiles: fewer iterations than resident CTAs, so the plan uses
    # fewer CTAs (each at least two K tiles); one tile of three K tiles on
    # one CTA that covers it whole (no fix-up work at all).
    for (M, N, K) in [(64, 64, 96), (300, 200, 64), (128, 128, 4)]:
        A, B = gemm_inputs.make_ab(M, N, K, seed=5, dist="uniform")
        Cref, W = oracle.sgemm(A.numpy(), B.numpy(), with_w=True)
        for cfg in TILES:
            assert_within(run(A.cuda(), B.cuda(), **SK, **cfg), Cref, W, f"{(M, N, K)} {cfg}")


def test_stream_k_general_form_alpha_beta_bias():
    # The fix-up applies alpha, beta and the bias row like every epilogue.
    M, N, K = 1000, 520, 700
    A, B = gemm_inputs.make_ab(M, N, K, seed=8, dist="uniform")
    g = torch.Generator().manual_seed(9)
    C0 = torch.rand(M, N, generator=g) * 2 - 1
    bias = torch.rand(N, generator=g) * 2 - 1
    alpha, beta = 0.75, -1.5
    ref, W = oracle.sgemm_general(A.numpy(), B.numpy(), C0.numpy().ravel().copy(), M, N, K,
                                  K, N, N, alpha=alpha, beta=beta, bias=bias.numpy(),
                                  with_w=True)
    c = C0.cuda()
    mt.gemm(A.cuda(), B.cuda(), c, alpha=alpha, beta=beta, bias=bias.cuda(), **SK)
    torch.cuda.synchronize()
    assert_within(c.cpu().numpy(), ref.reshape(M, N), W.reshape(M, N), "general stream-K")


def test_stream_k_choices_refused():
    # Explicit split_k with stream-K, tiles whose warps form K groups, and
    # the one-warp kernel refuse the schedule before any launch.
    with pytest.raises(mt.MtError):
        mt.plan(1024, 1024, 1024, split_k=2, **SK)
    with pytest.raises(mt.MtError):
        mt.plan(1024, 1024, 1024, bm=64, bn=128, stages=3, pack_a=4, **SK)
    # ... but the automatic tile of such a grid is one without K groups.
    assert mt.plan(512, 512, 4096, **SK)["threads"] == 128
    with pytest.raises(mt.MtError):
        mt.plan(1024, 1024, 1024, variant="p18", **SK)
    # split_k = 1 turns stream-K off like the split tail.
    p = mt.plan(1024, 1024, 1024, split_k=1, **SK)
    assert p["stream_k"] == 0 and p["split_k"] == 1


# --- the persistent tensor-core kernels ----------------------------------------
# The same schedule on the tcgen05 kernels: after its whole tiles, each CTA
# (CTA pair) of the persistent grid takes a run of the remaining tiles' K
# tiles; the same fix-up adds the pieces.  Tolerance 5e-5 * W, as for every
# tensor-core path.
TC_TOL = 5e-5
TF32_TILES = [dict(variant="tf32x3"),                                  # automatic
              dict(variant="tf32x3", bm=128, bn=256, bk=16, pack_a=1),  # one CTA per tile
              dict(variant="tf32x3", bm=128, bn=64, bk=32, pack_a=1),
              dict(variant="tf32x3", bm=256, bk=16),                    # CTA pairs
              dict(variant="tf32x3", bm=128, bn=128, bk=32, pack_a=2)]  # A split in the kernel
TF32_IDS = ["-".join(f"{k}{v}" for k, v in c.items()) for c in TF32_TILES]


def assert_tc(C, Cref, W, what):
    err = np.abs(np.asarray(C, np.float64) - Cref)
    bad = err > TC_TOL * W
    if bad.any():
        i, j = np.argwhere(bad)[0]
        pytest.fail(f"{what}: {bad.sum()} outputs outside {TC_TOL}*W, first at ({i},{j})")


@pytest.mark.parametrize("cfg", TF32_TILES, ids=TF32_IDS)
@pytest.mark.parametrize("name", ["masked_100x72x80", "square_1024", "ragged_4097x3001x2053"])
def test_stream_k_tf32x3_workloads(name, cfg, full_oracle):
    w = gemm_inputs.WORKLOADS[name]
    if cfg.get("pack_a") == 2 and w.K % 4:
        pytest.skip("A split in the kernel needs rows of whole float4s")
    A, B = gemm_inputs.make_workload(name)
    a, b = A.cuda(), B.cuda()
    p = mt.plan(w.M, w.N, w.K, a=a, b=b, **SK, **cfg)
    assert p["stream_k"] > 0 and p["split_k"] == 1
    got = run(a, b, **SK, **cfg)
    Cref, W = full_oracle(name)
    assert_tc(got, Cref, W, f"{name} {cfg}")
    assert np.array_equal(run(a, b, **SK, **cfg), got)


@pytest.mark.parametrize("cfg", TF32_TILES, ids=TF32_IDS)
@pytest.mark.parametrize("shape", [(100, 72, 80), (1000, 1000, 1200), (2304, 2304, 256)])
def test_stream_k_tf32x3_integer_inputs_bit_exact(shape, cfg):
    M, N, K = shape
    A, B = gemm_inputs.make_ab(M, N, K, seed=12, dist="int")
    Cref = oracle.sgemm(A.numpy(), B.numpy())
    assert np.array_equal(run(A.cuda(), B.cuda(), **SK, **cfg), Cref)


def test_stream_k_tf32x3_square_4096_every_element(full_oracle):
    A, B = gemm_inputs.make_workload("square_4096")
    p = mt.plan(4096, 4096, 4096, variant="tf32x3", **SK)
    assert p["stream_k"] > 0 and p["bm"] == 256
    got = run(A.cuda(), B.cuda(), variant="tf32x3", **SK)
    Cref, W = full_oracle("square_4096")
    assert_tc(got, Cref, W, "square_4096 tf32x3 stream-K")


_MIXED_REF = {}


@pytest.mark.parametrize("tile", [dict(), dict(bm=128), dict(bm=128, bn=128), dict(bm=256)],
                         ids=["auto", "single", "bn128", "pair"])
@pytest.mark.parametrize("shape", [(100, 72, 80), (1024, 1024, 1024), (4097, 3001, 2053),
                                   (4096, 4096, 4096)])
def test_stream_k_16bit_inputs(shape, tile):
    M, N, K = shape
    A16, B16 = gemm_inputs.make_ab16(M, N, K, 3, "normal", "bf16")
    p = mt.plan_mixed(mt.MT_DTYPE_BF16, M, N, K, **SK, **tile)
    assert p["stream_k"] > 0 and p["split_k"] == 1
    if shape not in _MIXED_REF:  # one oracle run per shape for all tiles
        _MIXED_REF.clear()
        _MIXED_REF[shape] = oracle.gemm_mixed_general(
            oracle.BF16, A16, B16, np.zeros(M * N, np.float32), M, N, K, K, N, N, with_w=True)
    Cref, W = _MIXED_REF[shape]
    a, b = A16.cuda(), B16.cuda()
    got = mt.gemm_mixed(a, b, **SK, **tile)
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    assert_tc(got, Cref.reshape(M, N), W.reshape(M, N), f"bf16 {shape} {tile}")
    again = mt.gemm_mixed(a, b, **SK, **tile)
    torch.cuda.synchronize()
    assert np.array_equal(again.cpu().numpy(), got)
    assert mt.mt_check_device_status(0) == mt.MT_OK


def test_stream_k_16bit_integer_inputs_bit_exact():
    M, N, K = 1000, 1000, 1200
    A16, B16 = gemm_inputs.make_ab16(M, N, K, 4, "int", "bf16")
    Cref = oracle.gemm_mixed_general(oracle.BF16, A16, B16, np.zeros(M * N, np.float32),
                                     M, N, K, K, N, N)
    for tile in (dict(), dict(bm=128), dict(bm=256)):
        got = mt.gemm_mixed(A16.cuda(), B16.cuda(), **SK, **tile)
        torch.cuda.synchronize()
        assert np.array_equal(got.cpu().numpy(), Cref.reshape(M, N)), tile


@pytest.mark.parametrize("variant", ["tf32x3", "bf16"])
def test_stream_k_tensor_cores_general_form(variant):
    # alpha, beta and the bias row through the fix-up on the tensor-core
    # paths, with transposed A (the pieces' sums are the same; only the
    # operand order differs).
    M, N, K = 700, 1300, 900
    g = torch.Generator().manual_seed(19)
    C0 = torch.rand(M, N, generator=g) * 2 - 1
    bias = torch.rand(N, generator=g) * 2 - 1
    alpha, beta = -0.5, 1.25
    c = C0.cuda()
    if variant == "tf32x3":
        A, B = gemm_inputs.make_ab(M, N, K, seed=20, dist="uniform")
        At = A.t().contiguous()  # stored K x M
        ref, W = oracle.sgemm_general(At.numpy(), B.numpy(), C0.numpy().ravel().copy(), M, N,
                                      K, M, N, N, alpha=alpha, beta=beta, trans_a=True,
                                      bias=bias.numpy(), with_w=True)
        mt.gemm(At.cuda(), B.cuda(), c, alpha=alpha, beta=beta, trans_a=True, bias=bias.cuda(),
                variant="tf32x3", **SK)
    else:
        A16, B16 = gemm_inputs.make_ab16(M, N, K, 20, "uniform", "bf16")
        At16 = A16.t().contiguous()
        ref, W = oracle.gemm_mixed_general(oracle.BF16, At16, B16, C0.numpy().ravel().copy(),
                                           M, N, K, M, N, N, alpha, beta, 1, 0, with_w=True,
                                           bias=bias.numpy())
        mt.gemm_mixed(At16.cuda(), B16.cuda(), c, alpha=alpha, beta=beta, trans_a=True,
                      bias=bias.cuda(), **SK)
    torch.cuda.synchronize()
    assert_tc(c.cpu().numpy(), ref.reshape(M, N), W.reshape(M, N), f"{variant} general stream-K")
    assert mt.mt_check_device_status(0) == mt.MT_OK


@pytest.mark.parametrize("shape", [(64, 64, 100000), (1, 4096, 8192), (4096, 1, 8192),
                                   (3, 5, 70000)])
def test_stream_k_one_tile_many_runs(shape):
    """A tile whose K is dealt out to hundreds of CTAs: its pieces exceed
    the fix-up's 256 slots per pass, so the sum runs over several passes,
    still in k order.  Single rows and columns of C."""
    M, N, K = shape
    for cfg in (dict(), dict(bm=128, bn=128, bk=16, stages=4, wm=64, pack_a=5)):
        p = mt.plan(M, N, K, **SK, **cfg)
        assert p["stream_k"] > 0
        A, B = gemm_inputs.make_ab(M, N, K, seed=26, dist="uniform")
        Cref, W = oracle.sgemm(A.numpy(), B.numpy(), with_w=True)
        a, b = A.cuda(), B.cuda()
        got = run(a, b, **SK, **cfg)
        assert_within(got, Cref, W, f"{shape} {cfg}")
        assert np.array_equal(run(a, b, **SK, **cfg), got)
    # The persistent tensor-core kernels on the same shapes.
    got = run(a, b, variant="tf32x3", **SK)
    assert_tc(got, Cref, W, f"{shape} tf32x3")
