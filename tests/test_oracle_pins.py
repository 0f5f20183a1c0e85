"""Pins the CPU oracle to facts that do not come from the oracle itself.

Each check is chosen so that a plausible slip in the oracle (a dropped term,
a wrong sign, a wrong index or leading dimension, a transposed operand,
fp32 instead of fp64 accumulation) fails at least one of them;
``test_oracle_mutants.py`` plants such slips and confirms it.

Setting MT_ORACLE_LIB runs these pins against another build of the oracle,
and MT_ORACLE_RULES against another copy of ``oracle/smem_rules.py`` (the
mutant test uses both).
"""
import importlib.util
import json
import math
import os
import sys
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import smem_rules as R

if os.environ.get("MT_ORACLE_RULES"):
    _spec = importlib.util.spec_from_file_location("mt_rules_under_test",
                                                   os.environ["MT_ORACLE_RULES"])
    R = importlib.util.module_from_spec(_spec)
    sys.modules[_spec.name] = R  # dataclasses resolve the module by name
    _spec.loader.exec_module(R)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
LIB = oracle.load(os.environ.get("MT_ORACLE_LIB") or None)


def gemm(A, B, **kw):
    return oracle.sgemm(A, B, lib=LIB, **kw)


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def rng(seed):
    return np.random.default_rng(seed)


# --- exact special cases ------------------------------------------------------
@pytest.mark.parametrize("M,K", [(37, 29), (5, 64), (64, 3)])
def test_identity_right_and_left(M, K):
    A = rng(1).standard_normal((M, K)).astype(np.float32)
    assert np.array_equal(gemm(A, np.eye(K, dtype=np.float32)), A)
    assert np.array_equal(gemm(np.eye(M, dtype=np.float32), A), A)


@pytest.mark.parametrize("M,N,K", [(23, 17, 11), (8, 40, 8)])
def test_permutation_rows_and_columns(M, N, K):
    g = rng(2)
    B = g.standard_normal((K, N)).astype(np.float32)
    perm = g.permutation(K)
    P = np.zeros((K, K), np.float32)
    P[np.arange(K), perm] = 1.0          # (P @ B)[r] = B[perm[r]]
    assert np.array_equal(gemm(P, B), B[perm])
    A = g.standard_normal((M, K)).astype(np.float32)
    Q = np.zeros((K, K), np.float32)
    Q[perm, np.arange(K)] = 1.0          # (A @ Q)[:, c] = A[:, perm[c]]
    assert np.array_equal(gemm(A, Q), A[:, perm])


@pytest.mark.parametrize("M,N,K", [(13, 7, 5), (33, 65, 17), (64, 48, 200),
                                   (1, 9, 31), (9, 1, 2)])
def test_small_integers_exact(M, N, K):
    # Entries in [-8, 8]: every partial sum is an integer far below 2**24,
    # so the exact integer product (numpy int64 matmul) is the answer.
    g = rng(3)
    Ai = g.integers(-8, 9, (M, K))
    Bi = g.integers(-8, 9, (K, N))
    C = gemm(Ai.astype(np.float32), Bi.astype(np.float32))
    assert np.array_equal(C.astype(np.int64), Ai @ Bi)


def test_rank_one_closed_form():
    # A[i,k] = x_i, B[k,j] = y_j  ->  C[i,j] = K * x_i * y_j exactly.
    M, N, K = 6, 5, 12
    x = np.array([1, -2, 3, 0.5, -0.25, 7], np.float32)
    y = np.array([2, -1, 0.5, 4, -8], np.float32)
    A = np.repeat(x[:, None], K, axis=1)
    B = np.repeat(y[None, :], K, axis=0)
    assert np.array_equal(gemm(A, B), (K * x[:, None] * y[None, :]).astype(np.float32))


def test_k_zero_gives_zeros():
    # The accumulator starts at zero (tl.zeros) and the K loop runs no trip.
    C = gemm(np.zeros((4, 0), np.float32), np.zeros((0, 3), np.float32))
    assert C.shape == (4, 3) and np.all(C == 0) and not np.signbit(C).any()


def test_w_is_abs_product():
    # W = |A|*|B| with |entries| = 1 and random signs -> W = K everywhere,
    # while C is the signed sum.
    g = rng(4)
    M, N, K = 9, 10, 21
    A = g.choice([-1.0, 1.0], (M, K)).astype(np.float32)
    B = g.choice([-1.0, 1.0], (K, N)).astype(np.float32)
    C, W = gemm(A, B, with_w=True)
    assert np.all(W == K)
    assert np.array_equal(C.astype(np.int64),
                          A.astype(np.int64) @ B.astype(np.int64))


def test_fp64_accumulation():
    # 2**24 + 1 - 2**24 summed left to right: fp32 accumulation gives 0,
    # the double accumulation the oracle uses gives 1.
    A = np.array([[2.0 ** 24, 1.0, -(2.0 ** 24)]], np.float32)
    B = np.ones((3, 1), np.float32)
    assert gemm(A, B)[0, 0] == 1.0


# --- brute force on tiny ragged shapes -----------------------------------------
SHAPES = [(1, 1, 1), (3, 5, 7), (9, 2, 16), (15, 17, 16), (16, 16, 17),
          (17, 15, 33), (31, 33, 9), (33, 31, 32), (2, 65, 5), (63, 3, 8)]


def _grid_sample(count=24, seed=2024, max_macs=40000):
    """A seeded sample of (M, N, K) from {1..9, 15, 16, 17, 31, 32, 33, 63,
    65}^3 (each axis on both sides of the tile edges the kernels use), kept
    small enough for exact rational sums."""
    axis = [1, 2, 3, 4, 5, 6, 7, 8, 9, 15, 16, 17, 31, 32, 33, 63, 65]
    g = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        t = tuple(int(x) for x in g.choice(axis, 3))
        if t not in out and t not in SHAPES and t[0] * t[1] * t[2] <= max_macs:
            out.append(t)
    return out


SHAPES = SHAPES + _grid_sample()


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_brute_force_tiny(M, N, K):
    """Exact rational sum, rounded once, versus the oracle.

    The oracle's double sum differs from the exact sum by at most
    K * 2**-53 * W; after one rounding to fp32 the result is within one
    fp32 half-ulp of the exact value plus that amount.
    """
    g = rng(5 + M * 1000 + N * 10 + K)
    A = g.uniform(-1, 1, (M, K)).astype(np.float32)
    B = g.uniform(-1, 1, (K, N)).astype(np.float32)
    C, W = gemm(A, B, with_w=True)
    for i in range(M):
        for j in range(N):
            exact = sum((Fraction(float(A[i, k])) * Fraction(float(B[k, j]))
                         for k in range(K)), Fraction(0))
            e = float(exact)
            bound = (abs(e) * 2.0 ** -24 + K * 2.0 ** -52 * W[i, j]
                     + 2.0 ** -149)
            assert abs(float(C[i, j]) - e) <= bound, (i, j)
            assert math.isclose(W[i, j], sum(abs(float(A[i, k])) *
                                             abs(float(B[k, j]))
                                             for k in range(K)),
                                rel_tol=1e-12, abs_tol=0.0)


def test_second_opinion_float64_library_matmul():
    # A library routine as a second opinion: float64 matmul then one rounding.
    g = rng(6)
    A = g.standard_normal((70, 130)).astype(np.float32)
    B = g.standard_normal((130, 90)).astype(np.float32)
    C, W = gemm(A, B, with_w=True)
    ref = (A.astype(np.float64) @ B.astype(np.float64))
    assert np.all(np.abs(C - ref) <= np.abs(ref) * 2.0 ** -24 + 1e-12 * W)


# --- zero-fill invariant ("Matching the safety mask") ------------------------
def test_zero_padding_changes_nothing():
    # Padding K (and M, N) with zeros up to tile multiples leaves every real
    # output bit-identical: the zero-filled elements contribute nothing.
    g = rng(7)
    M, N, K = 13, 10, 21
    A = g.standard_normal((M, K)).astype(np.float32)
    B = g.standard_normal((K, N)).astype(np.float32)
    Ap = np.zeros((16, 32), np.float32)
    Ap[:M, :K] = A
    Bp = np.zeros((32, 16), np.float32)
    Bp[:K, :N] = B
    Cp = gemm(Ap, Bp)
    assert np.array_equal(Cp[:M, :N], gemm(A, B))
    assert np.all(Cp[M:, :] == 0) and np.all(Cp[:, N:] == 0)


def test_rows_and_elements_agree_with_full():
    g = rng(8)
    A = g.standard_normal((40, 33)).astype(np.float32)
    B = g.standard_normal((33, 27)).astype(np.float32)
    C, W = gemm(A, B, with_w=True)
    rows = [39, 0, 17]
    Cr, Wr = oracle.sgemm_rows(A, B, rows, with_w=True, lib=LIB)
    assert np.array_equal(Cr, C[rows]) and np.array_equal(Wr, W[rows])
    ii, jj = np.array([0, 39, 5]), np.array([26, 0, 13])
    e, w = oracle.sgemm_elements(A, B, ii, jj, lib=LIB)
    assert np.array_equal(e, C[ii, jj]) and np.allclose(w, W[ii, jj], rtol=1e-15)


# --- the pages' rules (smem_rules) -------------------------------------------
def test_padding_rule_worked_examples():
    data = golden("padding_rule_examples.json")
    for c in data["cases"]:
        assert R.row_padding(c["columns"], c["simultaneous_rows"]) == c["padding"], c


def test_bank_mapping_example():
    data = golden("bank_mapping.json")
    for key in ("unpadded", "padded"):
        got = R.column_banks(data[key]["row_stride"], data["rows"], data["column"])
        assert list(got) == data[key]["banks"]


def test_bank_simulator_matches_example_and_textbook_cases():
    data = golden("bank_mapping.json")
    # Four rows read column 0; lanes 8r..8r+7 share row r (a broadcast).
    for key, expect in (("unpadded", 2), ("padded", 1)):
        stride = data[key]["row_stride"]
        addrs = [4 * ((lane // 8) * stride) for lane in range(32)]
        assert R.conflict_degree(addrs, 4) == expect
    # 32 lanes down one column of a 32-wide row-major tile: 32-way conflict;
    # one padding word per row removes it (skills page, step 4).
    assert R.conflict_degree([4 * 32 * t for t in range(32)], 4) == 32
    assert R.conflict_degree([4 * 33 * t for t in range(32)], 4) == 1
    # All lanes on one word: broadcast, one transaction.
    assert R.wavefronts([128] * 32, 4) == 1
    # Consecutive float4 per lane: 4 phases of 8 lanes, none conflicted.
    addrs = [16 * t for t in range(32)]
    assert R.wavefronts(addrs, 16) == R.ideal_wavefronts(addrs, 16) == 4


def test_layout_examples():
    data = golden("layout_examples.json")
    sm = data["stage_mapping"]
    assert [R.dot_stage(k, sm["bk"]) for k in sm["k_base"]] == sm["stage"]
    for b in data["buffers"]:
        buf = R.SharedBuffer(b["rows"], b["columns"])
        assert buf.size == b["floats"]
        counts = [len(R.cooperative_indices(t, b["rows"], b["columns"], b["threads"]))
                  for t in range(b["threads"])]
        assert set(counts) == {b["per_thread"]}
        seen = sorted(p for t in range(b["threads"])
                      for p in R.cooperative_indices(t, b["rows"], b["columns"],
                                                     b["threads"]))
        assert seen == [(r, c) for r in range(b["rows"]) for c in range(b["columns"])]
    pa = data["padded_a"]
    buf = R.SharedBuffer(pa["rows"], pa["columns"], pa["row_padding"], 2)
    assert buf.row_stride == pa["row_stride"]
    assert buf.stage_size == pa["rows"] * pa["row_stride"]
    assert buf.size == 2 * buf.stage_size and buf.nbytes == 4 * buf.size
    assert buf.element(1, 2, 3) == buf.stage_size + 2 * pa["row_stride"] + 3


def test_layout_rejects_invalid():
    for bad in [(0, 4), (4, 0), (-1, 4)]:
        with pytest.raises(ValueError):
            R.SharedBuffer(*bad)
    with pytest.raises(ValueError):
        R.SharedBuffer(4, 16, row_padding=-1)
    with pytest.raises(ValueError):
        R.SharedBuffer(4, 16, stage_count=0)
    buf = R.SharedBuffer(4, 16, 1, 2)
    for coord in [(2, 0, 0), (0, 4, 0), (0, 0, 16), (-1, 0, 0)]:
        with pytest.raises(ValueError):
            buf.element(*coord)


def test_budget_formula():
    limit = golden("layout_examples.json")["budget_limit_bytes"]
    # The pages' own example tile (BM=4, BK=16, BN=8, one padding word).
    assert R.two_stage_pair_bytes(4, 16, 8, 1) == 2 * (4 * 17 + 16 * 8) * 4
    assert R.fits_budget(R.two_stage_pair_bytes(4, 16, 8, 1), limit)
    # A 128x128 tile with BK=32 does not fit 48 KiB with two stages.
    assert not R.fits_budget(R.two_stage_pair_bytes(128, 32, 128, 1), limit)
    # Equality is allowed: the check is required <= limit.
    assert R.fits_budget(limit, limit) and not R.fits_budget(limit + 1, limit)


def _column_read(row_stride_words, rows, lanes_per_phase, column=0):
    """Byte addresses of one warp reading word `column` of `rows` distinct rows.

    Lane l of each phase reads row l % rows; lanes that share a row read the
    same address (a broadcast).  Every phase repeats the pattern."""
    return [4 * ((lane % lanes_per_phase % rows) * row_stride_words + column)
            for lane in range(32)]


def test_scalar_rule_agrees_with_the_simulator():
    # The Part 18 rule against first principles: for every row width and
    # count of rows read at once, the padded layout serves a column read in
    # one transaction per phase, and whenever the rule asks for padding the
    # unpadded layout does not.
    for cols in range(1, 129):
        for rows in range(1, 33):
            pad = R.row_padding(cols, rows)
            assert R.conflict_degree(_column_read(cols + pad, rows, 32), 4) == 1, \
                (cols, rows)
            if pad:
                assert R.conflict_degree(_column_read(cols, rows, 32), 4) > 1
            else:
                # No padding where none is needed: the rule is not just "always pad".
                assert R.conflict_degree(_column_read(cols, rows, 32), 4) == 1


def test_vector_rule_agrees_with_the_simulator():
    # Our float4 reading of the rule, checked the same way: float4 reads are
    # served 8 lanes at a time, so up to 8 distinct rows share a phase.  The
    # column is any 16-byte aligned one; padding keeps every row 16-byte aligned.
    for cols in range(4, 257, 4):
        for rows in range(1, 9):
            pad = R.vector_row_padding(cols, rows)
            assert pad in (0, 4) and (cols + pad) % 4 == 0
            for column in (0, 4, cols - 4):
                padded = _column_read(cols + pad, rows, 8, column)
                assert R.conflict_degree(padded, 16) == 1, (cols, rows, column)
                plain = _column_read(cols, rows, 8, column)
                if pad:
                    assert R.conflict_degree(plain, 16) > 1, (cols, rows)
                else:
                    assert R.conflict_degree(plain, 16) == 1, (cols, rows)
    with pytest.raises(ValueError):
        R.vector_row_padding(6, 2)


def test_simulator_wide_access_phases():
    # Skills page, bank-analysis steps, with the phase sizes this oracle
    # reads for wide accesses: 8-byte accesses in two phases of 16 lanes,
    # 16-byte accesses in four phases of 8 lanes (each phase moves at most
    # 128 bytes through the 32 four-byte banks).
    # Consecutive 8-byte words: each half-warp covers the 32 banks once.
    consecutive8 = [8 * t for t in range(32)]
    assert R.wavefronts(consecutive8, 8) == R.ideal_wavefronts(consecutive8, 8) == 2
    assert R.conflict_degree(consecutive8, 8) == 1
    # A stride of 32 words: the 16 lanes of a phase all land in banks 0 and 1.
    stride32 = [128 * t for t in range(32)]
    assert R.conflict_degree(stride32, 8) == 16
    assert R.wavefronts(stride32, 8) == 32
    # A stride of 32 words read as float4: 8 lanes per phase in banks 0..3.
    assert R.conflict_degree(stride32, 16) == 8
    assert R.wavefronts(stride32, 16) == 32
    # Both half-warps on the same 128 bytes: each phase is served on its own,
    # so the repeat is a second transaction, not a broadcast.
    repeat8 = [8 * (t % 16) for t in range(32)]
    assert R.wavefronts(repeat8, 8) == 2
    # First half-warp strided (16 words in bank 0), second consecutive: the
    # phases cost 16 and 1; served as one they would cost 16.
    mixed8 = [128 * t for t in range(16)] + [8 * t for t in range(16)]
    assert R.wavefronts(mixed8, 8) == 17
    # Inactive lanes cost nothing; a phase with no active lane costs nothing.
    assert R.wavefronts([None] * 16 + [8 * t for t in range(16)], 8) == 1
    assert R.wavefronts([None] * 32, 16) == 0
    # Misaligned wide addresses are refused.
    with pytest.raises(ValueError):
        R.wavefronts([4] + [0] * 31, 8)


# --- the general form: leading dimensions, transposes, alpha and beta --------
def general(A, B, C0, M, N, K, lda, ldb, ldc, **kw):
    return oracle.sgemm_general(A, B, C0, M, N, K, lda, ldb, ldc, lib=LIB, **kw)


def test_general_reduces_to_plain_product():
    g = rng(30)
    M, N, K = 37, 29, 41
    A = g.standard_normal((M, K)).astype(np.float32)
    B = g.standard_normal((K, N)).astype(np.float32)
    C = general(A, B, np.full(M * N, np.nan, np.float32), M, N, K, K, N, N)
    assert np.array_equal(C.reshape(M, N), gemm(A, B))  # beta = 0 never reads C


def test_general_leading_dimensions_and_transposes():
    g = rng(31)
    M, N, K = 13, 11, 17
    A = g.standard_normal((M, K)).astype(np.float32)
    B = g.standard_normal((K, N)).astype(np.float32)
    ref = gemm(A, B)
    lda, ldb, ldc = K + 5, N + 3, N + 7
    Ab = np.full((M, lda), np.nan, np.float32)
    Ab[:, :K] = A
    Bb = np.full((K, ldb), np.nan, np.float32)
    Bb[:, :N] = B
    C = general(Ab, Bb, np.zeros(M * ldc, np.float32), M, N, K, lda, ldb, ldc)
    assert np.array_equal(C.reshape(M, ldc)[:, :N], ref)
    assert np.all(C.reshape(M, ldc)[:, N:] == 0)  # columns past N untouched
    # Transposed storage: A as K x M (lda >= M), B as N x K (ldb >= K).
    At = np.full((K, M + 2), np.nan, np.float32)
    At[:, :M] = A.T
    Bt = np.full((N, K + 1), np.nan, np.float32)
    Bt[:, :K] = B.T
    C = general(At, Bt, np.zeros(M * N, np.float32), M, N, K, M + 2, K + 1, N,
                trans_a=True, trans_b=True)
    assert np.array_equal(C.reshape(M, N), ref)


def test_general_alpha_beta_exact_on_integers():
    g = rng(32)
    M, N, K = 9, 14, 23
    Ai = g.integers(-8, 9, (M, K))
    Bi = g.integers(-8, 9, (K, N))
    Ci = g.integers(-50, 51, (M, N))
    C, W = general(Ai.astype(np.float32), Bi.astype(np.float32), Ci.astype(np.float32),
                   M, N, K, K, N, N, alpha=2.0, beta=-3.0, with_w=True)
    assert np.array_equal(C.reshape(M, N).astype(np.int64), 2 * (Ai @ Bi) - 3 * Ci)
    assert np.array_equal(W, 2 * (np.abs(Ai) @ np.abs(Bi)) + 3 * np.abs(Ci))
    # alpha = 0: A and B are not read (NaN there does not propagate).
    C = general(np.full(M * K, np.nan, np.float32), np.full(K * N, np.nan, np.float32),
                Ci.astype(np.float32), M, N, K, K, N, N, alpha=0.0, beta=0.5)
    assert np.array_equal(C.reshape(M, N), (0.5 * Ci).astype(np.float32))


def test_general_bias_closed_forms():
    """The bias row (one value per output column, added to every row): with
    alpha = beta = 0 the result is the bias repeated on every row; with
    integer inputs the whole update is exact against integer arithmetic; W
    grows by |bias[j]|; no bias is the plain general form."""
    g = rng(33)
    M, N, K = 7, 11, 5            # M != N, so a row/column slip shows
    bias = g.integers(-9, 10, N)
    C = general(np.full(M * K, np.nan, np.float32), np.full(K * N, np.nan, np.float32),
                np.full(M * N, np.nan, np.float32), M, N, K, K, N, N, alpha=0.0, beta=0.0,
                bias=bias.astype(np.float32))
    assert np.array_equal(C.reshape(M, N), np.tile(bias, (M, 1)).astype(np.float32))
    Ai = g.integers(-8, 9, (M, K))
    Bi = g.integers(-8, 9, (K, N))
    Ci = g.integers(-50, 51, (M, N))
    C, W = general(Ai.astype(np.float32), Bi.astype(np.float32), Ci.astype(np.float32),
                   M, N, K, K, N, N, alpha=3.0, beta=-2.0, with_w=True,
                   bias=bias.astype(np.float32))
    assert np.array_equal(C.reshape(M, N).astype(np.int64), 3 * (Ai @ Bi) - 2 * Ci + bias)
    assert np.array_equal(W, 3 * (np.abs(Ai) @ np.abs(Bi)) + 2 * np.abs(Ci) + np.abs(bias))
    plain = general(Ai.astype(np.float32), Bi.astype(np.float32), Ci.astype(np.float32),
                    M, N, K, K, N, N, alpha=3.0, beta=-2.0)
    zero_bias = general(Ai.astype(np.float32), Bi.astype(np.float32), Ci.astype(np.float32),
                        M, N, K, K, N, N, alpha=3.0, beta=-2.0, bias=np.zeros(N, np.float32))
    assert np.array_equal(plain, zero_bias)


# --- 16-bit inputs (fp16 / bf16 patterns, fp32 result) ------------------------
ALL16 = np.arange(1 << 16, dtype=np.uint16)


def same_or_both_nan(x, y):
    x, y = np.asarray(x, np.float64), np.asarray(y, np.float64)
    return np.array_equal(np.isnan(x), np.isnan(y)) and \
        np.array_equal(x[~np.isnan(x)], y[~np.isnan(y)])


def test_f16_decode_every_pattern_matches_numpy():
    # numpy's float16 is an independent implementation of IEEE binary16.
    assert same_or_both_nan(oracle.value16(oracle.F16, ALL16),
                            ALL16.view(np.float16).astype(np.float64))


def test_bf16_decode_every_pattern_matches_torch():
    torch = pytest.importorskip("torch")
    ref = torch.from_numpy(ALL16.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64)
    assert same_or_both_nan(oracle.value16(oracle.BF16, ALL16), ref.numpy())


@pytest.mark.parametrize("dtype,pattern,value", [
    # binary16: one, smallest normal 2^-14, smallest subnormal 2^-24, largest
    # finite (2 - 2^-10) * 2^15 = 65504, minus two.
    (1, 0x3C00, Fraction(1)), (1, 0x0400, Fraction(1, 2 ** 14)),
    (1, 0x0001, Fraction(1, 2 ** 24)), (1, 0x7BFF, Fraction(65504)), (1, 0xC000, Fraction(-2)),
    # bfloat16: one, smallest normal 2^-126, smallest subnormal 2^-133,
    # largest finite (2 - 2^-7) * 2^127, 0x4049 = 1.5703125 * 2.
    (2, 0x3F80, Fraction(1)), (2, 0x0080, Fraction(1, 2 ** 126)),
    (2, 0x0001, Fraction(1, 2 ** 133)), (2, 0x7F7F, (2 - Fraction(1, 2 ** 7)) * 2 ** 127),
    (2, 0x4049, Fraction(201, 64)),
])
def test_16bit_closed_form_values(dtype, pattern, value):
    assert Fraction(float(oracle.value16(dtype, [pattern])[0])) == value


def _int16_operands(dtype, Ai, Bi):
    """Integer matrices as 16-bit patterns (integers up to 8 are exact)."""
    if dtype == oracle.F16:
        return Ai.astype(np.float16).view(np.uint16), Bi.astype(np.float16).view(np.uint16)
    torch = pytest.importorskip("torch")
    cv = lambda x: torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)
    return cv(Ai), cv(Bi)


@pytest.mark.parametrize("dtype", [1, 2])
@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_mixed_exact_on_integers_every_form(dtype, ta, tb):
    g = rng(40 + 2 * ta + tb)
    M, N, K = 11, 13, 19
    Ai = g.integers(-8, 9, (M, K))
    Bi = g.integers(-8, 9, (K, N))
    Ci = g.integers(-50, 51, (M, N))
    A16, B16 = _int16_operands(dtype, Ai, Bi)
    # Stored with padded leading dimensions, transposed where asked.
    As = A16.T if ta else A16
    Bs = B16.T if tb else B16
    lda, ldb, ldc = As.shape[1] + 3, Bs.shape[1] + 5, N + 2
    Ab = np.zeros((As.shape[0], lda), np.uint16)
    Ab[:, :As.shape[1]] = As
    Bb = np.zeros((Bs.shape[0], ldb), np.uint16)
    Bb[:, :Bs.shape[1]] = Bs
    C0 = np.full((M, ldc), 7, np.float32)
    C0[:, :N] = Ci
    C, W = oracle.gemm_mixed_general(dtype, Ab, Bb, C0, M, N, K, lda, ldb, ldc, alpha=2.0,
                                     beta=-3.0, trans_a=ta, trans_b=tb, with_w=True, lib=LIB)
    C = C.reshape(M, ldc)
    assert np.array_equal(C[:, :N].astype(np.int64), 2 * (Ai @ Bi) - 3 * Ci)
    assert np.all(C[:, N:] == 7)
    assert np.array_equal(W, 2 * (np.abs(Ai) @ np.abs(Bi)) + 3 * np.abs(Ci))


@pytest.mark.parametrize("dtype", [1, 2])
def test_mixed_reduces_to_fp32_oracle_on_widened_inputs(dtype):
    # Widening a 16-bit value to fp32 is exact, so the fp32 oracle on the
    # widened operands forms the same exact products in the same order.
    torch = pytest.importorskip("torch")
    M, N, K = 23, 17, 45
    g = torch.Generator().manual_seed(50 + dtype)
    tdt = torch.float16 if dtype == oracle.F16 else torch.bfloat16
    A = (torch.randn((M, K), generator=g) * 3).to(tdt)
    B = (torch.randn((K, N), generator=g) * 3).to(tdt)
    C = oracle.gemm_mixed_general(dtype, A, B, np.zeros(M * N, np.float32), M, N, K, K, N, N,
                                  lib=LIB)
    ref = gemm(A.float().numpy(), B.float().numpy())
    assert np.array_equal(C.reshape(M, N), ref)


@pytest.mark.parametrize("dtype", [1, 2])
def test_mixed_bias_closed_forms(dtype):
    """16-bit inputs with a bias row: integer inputs give the exact integer
    update plus the bias on every column j (M != N, so a row/column slip
    shows); the bias alone with alpha = beta = 0."""
    g = rng(60 + dtype)
    M, N, K = 9, 14, 7
    Ai = g.integers(-8, 9, (M, K))
    Bi = g.integers(-8, 9, (K, N))
    Ci = g.integers(-50, 51, (M, N))
    bias = g.integers(-9, 10, N)
    A16, B16 = _int16_operands(dtype, Ai, Bi)
    C, W = oracle.gemm_mixed_general(dtype, A16, B16, Ci.astype(np.float32), M, N, K, K, N, N,
                                     alpha=2.0, beta=-3.0, with_w=True, lib=LIB,
                                     bias=bias.astype(np.float32))
    assert np.array_equal(C.reshape(M, N).astype(np.int64), 2 * (Ai @ Bi) - 3 * Ci + bias)
    assert np.array_equal(W, 2 * (np.abs(Ai) @ np.abs(Bi)) + 3 * np.abs(Ci) + np.abs(bias))
    C = oracle.gemm_mixed_general(dtype, A16, B16, np.full(M * N, np.nan, np.float32), M, N, K,
                                  K, N, N, alpha=0.0, beta=0.0, lib=LIB,
                                  bias=bias.astype(np.float32))
    assert np.array_equal(C.reshape(M, N), np.tile(bias, (M, 1)).astype(np.float32))


def test_mixed_rejects_unknown_dtype():
    with pytest.raises(RuntimeError):
        oracle.gemm_mixed_general(3, np.zeros(4, np.uint16), np.zeros(4, np.uint16),
                                  np.zeros(4, np.float32), 2, 2, 2, 2, 2, 2, lib=LIB)


def test_fp16_bank_formula_and_simulator():
    data = golden("fp16_banks.json")
    got = [R.element_bank(i, data["element_bytes"]) for i in data["indices"]]
    assert got == data["banks"]
    assert all(R.element_bank(i, 2) == i // 2 % 32 for i in range(4096))
    assert all(R.element_bank(i, 4) == R.bank(i) for i in range(4096))
    # 32 lanes reading consecutive fp16 elements touch 16 words, two lanes
    # per word: one transaction with the same-word broadcast (the two-way
    # conflict the page warns of does not arise); reading them as half2
    # (4 bytes per lane) is one transaction too.
    assert R.wavefronts([2 * t for t in range(32)], 2) == 1
    assert R.wavefronts([4 * t for t in range(32)], 4) == 1
    # A column of a [rows][64] fp16 tile (128-byte rows): every lane in one
    # bank, 32 distinct words, 32-way; a row pitch of 66 halves (33 words,
    # the padding rule on the word count) makes it conflict-free.
    assert R.conflict_degree([128 * t for t in range(32)], 2) == 32
    assert R.conflict_degree([132 * t for t in range(32)], 2) == 1
    assert R.row_padding(64 // 2, 32) == 1 and R.row_padding(66 // 2, 32) == 0
