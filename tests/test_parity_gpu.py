"""GPU parity: the CUDA kernels, called through the C ABI, against the CPU oracle.

Tolerances (from the arithmetic, written here): every output of the FFMA and
P18 kernels is a chain of K fp32 FMAs in increasing k; for inputs of random
sign its error is a few fp32 ulps of the |A|*|B| scale W, far inside the
bound |C - C_ref| <= 1e-5 * W that is asserted elementwise.  Integer-valued
inputs whose partial sums stay below 2**24 have an exact result, so there
the kernels must match the oracle bit for bit.
"""
import numpy as np
import pytest
import torch

import gemm_inputs
import oracle
import tiled_fp32_gemm_gb300 as mt

pytestmark = pytest.mark.gpu

FFMA_TOL = 1e-5

# Every FFMA tile configuration the library builds (tile choice, micro-kernel).
FFMA_CONFIGS = [
    dict(),                                           # automatic
    dict(bm=128, bn=128, bk=32, stages=3, fma=2),     # 4 warps of 64 x 64
    dict(pack_a=2),                                   # row-major A tiles
    dict(pack_a=4),                                   # K-major A, gathered
    dict(pack_a=5),                                   # K-major A, from a copy
    dict(bm=64, bn=128, pack_a=4),
    dict(bm=64, bn=128, pack_a=5),
    dict(bm=64, bn=64, pack_a=5),
    dict(bm=128, bn=128, bk=32, stages=3, fma=2, wm=32, wn=64),
    dict(bm=128, bn=128, bk=32, stages=3, fma=2, wm=64, wn=32),
    dict(bm=128, bn=128, bk=16, stages=4, fma=2),
    # The same tile with shallower K pipelines: one stage (no double
    # buffering, two barriers per K tile), two and three.
    dict(bm=128, bn=128, bk=16, stages=1),
    dict(bm=128, bn=128, bk=16, stages=1, pack_a=4),
    dict(bm=128, bn=128, bk=16, stages=2),
    dict(bm=128, bn=128, bk=16, stages=3, pack_a=4),
    dict(bm=256, bn=128, fma=2),
    dict(bm=128, bn=128, bk=32, stages=3, fma=1),
    dict(bm=128, bn=128, bk=32, stages=4, fma=2),
    dict(bm=128, bn=256, bk=32, stages=3, fma=2),
    dict(bm=64, bn=64, bk=32, stages=3, fma=2),
    dict(bm=128, bn=128, bk=32, stages=3, fma=2, no_pad=True),
    dict(bm=128, bn=128, bk=32, stages=3, fma=2, wm=32, wn=64, no_pad=True),
]
# Tiles whose warps form two K groups (64 x 128, 3 stages): each output is
# the sum of two partial chains, so they agree with the others within the
# tolerance, not bit for bit.
SLICED_CONFIGS = [dict(bm=64, bn=128, stages=3, pack_a=4), dict(bm=64, bn=128, stages=3, pack_a=5),
                  dict(bm=64, bn=128, stages=3, pack_a=2)]
ALL_VARIANTS = FFMA_CONFIGS + SLICED_CONFIGS + [dict(variant="p18"),
                                                dict(variant="p18", no_pad=True),
                                                dict(variant="p18", stages=1)]


def ids(cfgs):
    return ["-".join(f"{k}{v}" for k, v in c.items()) or "auto" for c in cfgs]


@pytest.fixture(scope="module", autouse=True)
def library():
    from tiled_fp32_gemm_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    return mt.lib()


def run(A, B, **cfg):
    a = A.cuda()
    b = B.cuda()
    c = mt.sgemm(a, b, **cfg)
    torch.cuda.synchronize()
    return c.cpu()


def assert_within(C, Cref, W, tol, what=""):
    C = np.asarray(C, np.float64)
    err = np.abs(C - np.asarray(Cref, np.float64))
    bound = tol * np.asarray(W, np.float64)
    bad = err > bound
    if bad.any():
        i, j = np.argwhere(bad)[0]
        pytest.fail(f"{what}: {bad.sum()} outputs outside {tol}*W, first at ({i},{j}): "
                    f"got {C[i, j]!r} want {Cref[i, j]!r} W={W[i, j]!r}")


# --- the small workloads, every variant, full oracle ---------------------------
@pytest.mark.parametrize("cfg", ALL_VARIANTS, ids=ids(ALL_VARIANTS))
@pytest.mark.parametrize("name", ["masked_100x72x80", "square_1024"])
def test_small_workloads_all_variants(name, cfg):
    if cfg.get("variant") == "p18" and name == "square_1024":
        pytest.skip("the one-warp kernel is only a parity reference at small sizes")
    A, B = gemm_inputs.make_workload(name)
    Cref, W = oracle.sgemm(A.numpy(), B.numpy(), with_w=True)
    assert_within(run(A, B, **cfg).numpy(), Cref, W, FFMA_TOL, f"{name} {cfg}")


def test_ragged_workload_full():
    # 4097 x 3001 x 2053: every tile edge on M, N and K is masked.  Row-major
    # A tiles staged as stored: the odd leading dimensions force 4-byte
    # copies.  Row-major A tiles from copies (pack_a = 1): A and B copied
    # into rows padded to whole float4s, then 16-byte chunks.  Automatically:
    # A staged K-major from a transposed copy, B from a padded copy, on
    # 64 x 128 tiles, the tiles past the last full wave run as stream-K (the
    # split tail of four K slices on request); and A gathered K-major inside
    # the kernel (pack_a = 4).  Without K splits all give the same FMA chain
    # per output; stream-K and the split tail add a few partial sums, within
    # the tolerance.
    A, B = gemm_inputs.make_workload("ragged_4097x3001x2053")
    a, b = A.cuda(), B.cuda()
    assert mt.plan(4097, 3001, 2053, a=a, b=b, pack_a=2)["vec_ab"] == 0
    assert mt.plan(4097, 3001, 2053, a=a, b=b, pack_a=1)["pack_a"] == 1
    p = mt.plan(4097, 3001, 2053, a=a, b=b)
    assert (p["vec_ab"], p["vec_c"], p["pack_a"], p["bm"], p["bn"]) == (1, 0, 5, 64, 128)
    assert p["stream_k"] > 0 and p["split_k"] == 1
    assert mt.plan(4097, 3001, 2053, a=a, b=b, schedule="split_tail")["split_k"] == 4
    Cref, W = oracle.sgemm(A.numpy(), B.numpy(), with_w=True)
    as_stored = run(A, B, pack_a=2).numpy()
    assert_within(as_stored, Cref, W, FFMA_TOL, "ragged, as stored")
    for choice in (dict(pack_a=1), dict(split_k=1), dict(pack_a=4, split_k=1)):
        assert np.array_equal(run(A, B, **choice).numpy(), as_stored), choice
    assert_within(run(A, B).numpy(), Cref, W, FFMA_TOL, "ragged, automatic (stream-K)")
    assert_within(run(A, B, schedule="split_tail").numpy(), Cref, W, FFMA_TOL,
                  "ragged, split tail")


def sampled_rows(M, bm=128, extra=24, seed=0):
    """First and last rows, rows around tile edges and a few random rows."""
    g = np.random.default_rng(seed)
    rows = {0, M - 1}
    for t in (1, M // bm // 2, M // bm - 1):
        for d in (-1, 0):
            r = t * bm + d
            if 0 <= r < M:
                rows.add(r)
    rows |= set(g.integers(0, M, extra).tolist())
    return np.array(sorted(rows), np.int64)


@pytest.mark.parametrize("name", ["square_4096", "square_8192", "skinny_65536x128x4096"])
def test_full_size_every_element(name, full_oracle):
    """The benchmark's workloads in the benchmark's launch configuration,
    every output against the full oracle."""
    A, B = gemm_inputs.make_workload(name)
    c = mt.sgemm(A.cuda(), B.cuda())  # automatic choice, as the benchmark calls it
    torch.cuda.synchronize()
    Cref, W = full_oracle(name)
    assert_within(c.cpu().numpy(), Cref, W, FFMA_TOL, name)


# --- exact cases ----------------------------------------------------------------
@pytest.mark.parametrize("cfg", ALL_VARIANTS, ids=ids(ALL_VARIANTS))
@pytest.mark.parametrize("shape", [(100, 72, 80), (257, 130, 77), (128, 256, 96)])
def test_integer_inputs_bit_exact(shape, cfg):
    M, N, K = shape
    A, B = gemm_inputs.make_ab(M, N, K, seed=11, dist="int")
    Cref = oracle.sgemm(A.numpy(), B.numpy())
    got = run(A, B, **cfg).numpy()
    assert np.array_equal(got, Cref)


@pytest.mark.parametrize("name", ["tf32x3", "p18"])
def test_environment_selects_the_default_variant(name, monkeypatch):
    """mt_sgemm (no configuration) under MT_SGEMM_VARIANT gives the bits of
    the explicitly chosen variant."""
    A, B = gemm_inputs.make_workload("masked_100x72x80")
    a, b = A.cuda(), B.cuda()
    want = mt.sgemm(a, b, variant=name)
    c = torch.full((100, 72), float("nan"), device="cuda")
    monkeypatch.setenv("MT_SGEMM_VARIANT", name)
    st = mt.mt_sgemm(a.data_ptr(), b.data_ptr(), c.data_ptr(), 100, 72, 80,
                     torch.cuda.current_stream().cuda_stream)
    monkeypatch.delenv("MT_SGEMM_VARIANT")
    assert st == mt.MT_OK
    torch.cuda.synchronize()
    assert torch.equal(c, want)


@pytest.mark.parametrize("cfg", [dict(), dict(variant="p18")], ids=["ffma", "p18"])
def test_identity_and_permutation_exact(cfg):
    g = torch.Generator().manual_seed(5)
    A = torch.randn(150, 97, generator=g)
    I = torch.eye(97)
    assert torch.equal(run(A, I, **cfg), A)
    perm = torch.randperm(150, generator=g)
    P = torch.zeros(150, 150)
    P[torch.arange(150), perm] = 1.0
    assert torch.equal(run(P, A, **cfg), A[perm])


def test_all_variants_agree_bitwise():
    # Without K splitting, every FFMA/P18 output is the same chain of fp32
    # FMAs in increasing k, so every variant must produce the same bits.
    A, B = gemm_inputs.make_ab(200, 136, 300, seed=12, dist="normal")
    ref = run(A, B, variant="p18")
    assert torch.equal(run(A, B, variant="p18", stages=1), ref)
    for cfg in FFMA_CONFIGS:
        assert torch.equal(run(A, B, split_k=1, **cfg), ref), cfg


@pytest.mark.parametrize("stages", [1, 2, 3])
def test_pipeline_depths_bit_identical_at_4096(stages):
    """The K pipeline's depth changes when tiles are copied, not what is
    summed: on the 4096^3 workload (the depth measurements' shape, A from
    its transposed copy) every depth gives the 4-stage kernel's bits."""
    A, B = gemm_inputs.make_workload("square_4096")
    a, b = A.cuda(), B.cuda()
    tile = dict(bm=128, bn=128, bk=16, wm=64, split_k=1, pack_a=5)
    p = mt.plan(4096, 4096, 4096, a=a, b=b, stages=stages, **tile)
    assert (p["stages"], p["pack_a"], p["split_k"]) == (stages, 5, 1)
    ref = mt.sgemm(a, b, stages=4, **tile)
    got = mt.sgemm(a, b, stages=stages, **tile)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)
    rows = sampled_rows(4096, extra=8)
    Cr, Wr = oracle.sgemm_rows(A.numpy(), B.numpy(), rows, with_w=True)
    assert_within(got[torch.from_numpy(rows).cuda()].cpu().numpy(), Cr, Wr, FFMA_TOL,
                  f"4096^3, {stages} stages")


@pytest.mark.parametrize("split", [2, 3, 4])
@pytest.mark.parametrize("shape", [(257, 130, 777), (1000, 1000, 1000), (64, 64, 4096)])
def test_split_k_matches_oracle_and_is_deterministic(shape, split):
    M, N, K = shape
    A, B = gemm_inputs.make_ab(M, N, K, seed=16, dist="normal")
    Cref, W = oracle.sgemm(A.numpy(), B.numpy(), with_w=True)
    first = run(A, B, split_k=split)
    assert_within(first.numpy(), Cref, W, FFMA_TOL, f"split {split}")
    assert torch.equal(run(A, B, split_k=split), first)  # slices add in a fixed order


@pytest.mark.parametrize("shape,rows_only", [((512, 512, 4096), False),
                                             ((300, 200, 5000), False),
                                             ((33, 17, 9000), False),
                                             ((2048, 2048, 8192), True),
                                             ((65536, 128, 4096), True)])
def test_automatic_k_slices_match_oracle(shape, rows_only):
    """The automatic plans cut K: 512 x 512 x 4096 and the ragged 300 x 200
    x 5000 and 33 x 17 x 9000 have fewer tiles than SMs (every tile in
    slices, each CTA with two K groups of warps), 2048 x 2048 x 8192 and
    65536 x 128 x 4096 leave a last partial wave (those tiles' K tiles dealt
    out as stream-K runs on 64 x 128 tiles).  Within the tolerance and
    deterministic."""
    M, N, K = shape
    A, B = gemm_inputs.make_ab(M, N, K, seed=18, dist="uniform")
    a, b = A.cuda(), B.cuda()
    p = mt.plan(M, N, K, a=a, b=b)
    assert p["split_k"] > 1 or p["stream_k"] > 0
    first = mt.sgemm(a, b)
    again = mt.sgemm(a, b)
    torch.cuda.synchronize()
    assert torch.equal(first, again)
    if rows_only:
        rows = sampled_rows(M, bm=64, extra=24)
        Cr, Wr = oracle.sgemm_rows(A.numpy(), B.numpy(), rows, with_w=True)
        got = first[torch.from_numpy(rows).cuda()].cpu().numpy()
    else:
        Cr, Wr = oracle.sgemm(A.numpy(), B.numpy(), with_w=True)
        got = first.cpu().numpy()
    assert_within(got, Cr, Wr, FFMA_TOL, f"{shape} automatic split")


def test_split_k_integer_inputs_bit_exact():
    A, B = gemm_inputs.make_ab(300, 200, 1024, seed=17, dist="int")
    Cref = oracle.sgemm(A.numpy(), B.numpy())
    for split in (2, 4):
        assert np.array_equal(run(A, B, split_k=split).numpy(), Cref)





# --- edge cases ---------------------------------------------------------------------
TINY = [(1, 1, 1), (1, 7, 3), (5, 1, 9), (3, 5, 7), (16, 16, 16), (17, 15, 33),
        (31, 33, 1), (33, 31, 32), (63, 65, 31), (129, 127, 64), (130, 258, 33)]
# Plus a seeded sample of {1..9, 15, 16, 17, 31, 32, 33, 63, 65}^3: every axis
# just under, on and just over the staging widths and tile edges.
_AXIS = [1, 2, 3, 4, 5, 6, 7, 8, 9, 15, 16, 17, 31, 32, 33, 63, 65]
_g = np.random.default_rng(77)
while len(TINY) < 35:
    _t = tuple(int(x) for x in _g.choice(_AXIS, 3))
    if _t not in TINY:
        TINY.append(_t)


@pytest.mark.parametrize("shape", TINY)
def test_tiny_ragged_shapes(shape):
    M, N, K = shape
    A, B = gemm_inputs.make_ab(M, N, K, seed=M * 10000 + N * 100 + K, dist="uniform")
    Cref, W = oracle.sgemm(A.numpy(), B.numpy(), with_w=True)
    for cfg in (dict(), dict(bm=128, bn=256, bk=32, stages=3, fma=2), dict(variant="p18")):
        assert_within(run(A, B, **cfg).numpy(), Cref, W, FFMA_TOL, f"{shape} {cfg}")


def test_k_zero_writes_zeros_and_empty_is_noop():
    c = torch.full((7, 5), float("nan"), device="cuda")
    a = torch.empty((7, 0), device="cuda")
    b = torch.empty((0, 5), device="cuda")
    mt.sgemm(a, b, out=c)
    torch.cuda.synchronize()
    assert torch.equal(c.cpu(), torch.zeros(7, 5))
    c = torch.full((0, 5), 1.0, device="cuda")
    assert mt.mt_sgemm(0, 0, c.data_ptr(), 0, 5, 3, 0) == mt.MT_OK
    c = torch.full((4, 4), 3.0, device="cuda")
    assert mt.mt_sgemm(0, 0, c.data_ptr(), 4, 0, 3, 0) == mt.MT_OK
    torch.cuda.synchronize()
    assert torch.all(c == 3.0)


@pytest.mark.parametrize("cfg", [dict(), dict(bm=64, bn=64, bk=32, stages=3, fma=2),
                                 dict(variant="p18")], ids=["auto", "64x64", "p18"])
@pytest.mark.parametrize("offset", [0, 1])
def test_guard_bands_and_canaries(cfg, offset):
    """NaN around A and B catches any unmasked read; sentinels around C catch
    any stray write.  offset=1 misaligns the operands (4-byte staging)."""
    M, N, K = 133, 100, 72
    A, B = gemm_inputs.make_ab(M, N, K, seed=13, dist="uniform")
    guard = 4096
    abuf = torch.full((M * K + 2 * guard,), float("nan"))
    bbuf = torch.full((K * N + 2 * guard,), float("nan"))
    abuf[guard + offset:guard + offset + M * K] = A.reshape(-1)
    bbuf[guard + offset:guard + offset + K * N] = B.reshape(-1)
    sentinel = -12345.0
    cbuf = torch.full((M * N + 2 * guard,), sentinel, device="cuda")
    a_d, b_d = abuf.cuda(), bbuf.cuda()
    pa = a_d.data_ptr() + 4 * (guard + offset)
    pb = b_d.data_ptr() + 4 * (guard + offset)
    pc = cbuf.data_ptr() + 4 * (guard + offset)
    st = mt.mt_sgemm_ex(pa, pb, pc, M, N, K, torch.cuda.current_stream().cuda_stream,
                        mt.make_config(**cfg))
    assert st == mt.MT_OK
    torch.cuda.synchronize()
    out = cbuf.cpu()
    C = out[guard + offset:guard + offset + M * N].reshape(M, N).numpy()
    Cref, W = oracle.sgemm(A.numpy(), B.numpy(), with_w=True)
    assert np.isfinite(C).all()
    assert_within(C, Cref, W, FFMA_TOL, "guarded")
    assert torch.all(out[:guard + offset] == sentinel)
    assert torch.all(out[guard + offset + M * N:] == sentinel)


def test_nan_and_inf_propagate_like_ieee():
    M, N, K = 40, 36, 50
    A, B = gemm_inputs.make_ab(M, N, K, seed=14, dist="uniform")
    A[3, 7] = float("nan")
    B[11, 5] = float("inf")
    C = run(A, B).numpy()
    Cref = oracle.sgemm(A.numpy(), B.numpy())
    same = (C == Cref) | (np.isnan(C) & np.isnan(Cref))
    finite = np.isfinite(Cref)
    assert np.array_equal(np.isnan(C), np.isnan(Cref))
    assert np.array_equal(np.isinf(C), np.isinf(Cref))
    assert same[~finite].all()


def test_host_buffer_entry_point():
    A, B = gemm_inputs.make_workload("masked_100x72x80")
    a = A.numpy()
    b = B.numpy()
    c = np.full((100, 72), np.nan, np.float32)
    st = mt.mt_sgemm_host(a.ctypes.data, b.ctypes.data, c.ctypes.data, 100, 72, 80, 0, None)
    assert st == mt.MT_OK
    Cref, W = oracle.sgemm(a, b, with_w=True)
    assert_within(c, Cref, W, FFMA_TOL, "host")


def test_runs_on_caller_stream():
    A, B = gemm_inputs.make_ab(300, 260, 200, seed=15, dist="normal")
    s = torch.cuda.Stream()
    a, b = A.cuda(), B.cuda()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        c = mt.sgemm(a, b)
    s.synchronize()
    Cref, W = oracle.sgemm(A.numpy(), B.numpy(), with_w=True)
    assert_within(c.cpu().numpy(), Cref, W, FFMA_TOL, "stream")


def test_alias_rejected_without_launch():
    a = torch.ones(64, 64, device="cuda")
    b = torch.ones(64, 64, device="cuda")
    st = mt.mt_sgemm(a.data_ptr(), b.data_ptr(), a.data_ptr(), 64, 64, 64, 0)
    assert st == mt.MT_ERR_ALIAS
    torch.cuda.synchronize()
    assert torch.all(a == 1.0)
    assert mt.mt_device_status(0) == mt.MT_OK


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_entry_point_pipelined_blocks(pinned):
    """8192 x 8192 x 512 from host buffers: four row blocks, each copied in,
    multiplied and copied out on its own stream while its neighbours move.
    Without K slices the FFMA result is bit-identical to the device entry
    point (the same FMA chain per output); the automatic plans split the
    last partial wave of each call (different tiles for a block than for the
    whole product) and stay within tolerance, as does 3xTF32."""
    M, N, K = 8192, 8192, 512
    A, B = gemm_inputs.make_ab(M, N, K, seed=17, dist="normal")
    if pinned:
        A, B = A.pin_memory(), B.pin_memory()
        c = torch.full((M, N), float("nan")).pin_memory()
    else:
        c = torch.full((M, N), float("nan"))
    unsplit = mt.make_config(split_k=1)
    st = mt.mt_sgemm_host(A.data_ptr(), B.data_ptr(), c.data_ptr(), M, N, K, 0, unsplit)
    assert st == mt.MT_OK
    dev = mt.sgemm(A.cuda(), B.cuda(), split_k=1).cpu()
    assert torch.equal(c, dev)
    rows = np.array([0, 2047, 2048, 4095, 4096, 6143, 6144, 8191])
    Cr, Wr = oracle.sgemm_rows(A.numpy(), B.numpy(), rows, with_w=True)
    assert_within(c.numpy()[rows], Cr, Wr, FFMA_TOL, "host pipelined")
    c.fill_(float("nan"))
    st = mt.mt_sgemm_host(A.data_ptr(), B.data_ptr(), c.data_ptr(), M, N, K, 0, None)
    assert st == mt.MT_OK
    assert not torch.isnan(c).any()
    assert_within(c.numpy()[rows], Cr, Wr, FFMA_TOL, "host pipelined, automatic")
    c.fill_(float("nan"))
    st = mt.mt_sgemm_host(A.data_ptr(), B.data_ptr(), c.data_ptr(), M, N, K, 0,
                          mt.make_config(variant="tf32x3"))
    assert st == mt.MT_OK
    assert_within(c.numpy()[rows], Cr, Wr, 5e-5, "host pipelined tf32x3")
    assert mt.mt_device_status(0) == mt.MT_OK


def test_host_entry_point_async_calls_overlap_and_match():
    """Two mt_sgemm_host_async calls back to back on one stream (pinned
    buffers), then one synchronisation: each result equals the synchronous
    entry point's bit for bit."""
    shapes = [(4096, 2048, 1024), (2048, 4096, 2048)]
    bufs = []
    for i, (M, N, K) in enumerate(shapes):
        A, B = gemm_inputs.make_ab(M, N, K, seed=60 + i, dist="normal")
        bufs.append((M, N, K, A.pin_memory(), B.pin_memory(),
                     torch.full((M, N), float("nan")).pin_memory(),
                     torch.full((M, N), float("nan")).pin_memory()))
    s = torch.cuda.Stream()
    for (M, N, K, A, B, c_async, _c) in bufs:
        assert mt.mt_sgemm_host_async(A.data_ptr(), B.data_ptr(), c_async.data_ptr(), M, N, K,
                                      s.cuda_stream, None) == mt.MT_OK
    s.synchronize()
    for (M, N, K, A, B, c_async, c_sync) in bufs:
        assert mt.mt_sgemm_host(A.data_ptr(), B.data_ptr(), c_sync.data_ptr(), M, N, K, 0,
                                None) == mt.MT_OK
        assert torch.equal(c_async, c_sync)
        rows = np.array([0, M // 2, M - 1])
        Cr, Wr = oracle.sgemm_rows(A.numpy(), B.numpy(), rows, with_w=True)
        assert_within(c_async.numpy()[rows], Cr, Wr, FFMA_TOL, "host async")
    assert mt.mt_device_status(0) == mt.MT_OK
