"""The seeded input recipe both sides read (gemm_inputs), on CPU.

A CPU torch.Generator seeded with the workload's seed draws A (M x K) and
then B (K x N) in float32; "uniform" is rand*2-1 in [-1, 1), "normal" is
randn, "int" integers in [-8, 8]; every shape reseeds (so the two seed-4
shapes of the last configuration both start from seed 4); 16-bit inputs are
the same draws rounded by torch's conversion.
"""
import pytest
import torch

import gemm_inputs as gi


def test_same_seed_same_bytes():
    a1, b1 = gi.make_ab(33, 17, 9, 7, "normal")
    a2, b2 = gi.make_ab(33, 17, 9, 7, "normal")
    assert torch.equal(a1, a2) and torch.equal(b1, b2)
    a3, _ = gi.make_ab(33, 17, 9, 8, "normal")
    assert not torch.equal(a1, a3)


def test_a_is_drawn_before_b_from_one_generator():
    M, N, K = 5, 6, 7
    A, B = gi.make_ab(M, N, K, 3, "uniform")
    g = torch.Generator().manual_seed(3)
    flat = torch.rand(M * K + K * N, generator=g) * 2 - 1
    assert torch.equal(A.reshape(-1), flat[:M * K])
    assert torch.equal(B.reshape(-1), flat[M * K:])


def test_every_shape_reseeds():
    # The square and the skinny seed-4 workloads both start from seed 4: the
    # first draws of A are the same for any shape.
    sq, sk = gi.WORKLOADS["square_8192"], gi.WORKLOADS["skinny_65536x128x4096"]
    assert sq.seed == sk.seed == 4 and sq.dist == sk.dist == "uniform"
    a_small, _ = gi.make_ab(2, 3, 8, 4, "uniform")
    a_wide, _ = gi.make_ab(1, 5, 16, 4, "uniform")
    assert torch.equal(a_small.reshape(-1), a_wide.reshape(-1))


@pytest.mark.parametrize("dist", ["uniform", "normal", "int"])
def test_value_ranges(dist):
    A, B = gi.make_ab(300, 200, 100, 11, dist)
    v = torch.cat([A.reshape(-1), B.reshape(-1)])
    assert v.dtype == torch.float32 and A.is_contiguous() and B.is_contiguous()
    if dist == "uniform":
        assert v.min() >= -1.0 and v.max() < 1.0 and abs(v.mean()) < 0.02
    elif dist == "normal":
        assert abs(v.mean()) < 0.02 and abs(v.var() - 1.0) < 0.03
    else:
        assert torch.equal(v, v.round()) and v.min() == -8 and v.max() == 8


def test_workload_table_matches_the_configurations():
    want = {"masked_100x72x80": (100, 72, 80, 0, "uniform"),
            "square_1024": (1024, 1024, 1024, 1, "normal"),
            "square_4096": (4096, 4096, 4096, 2, "uniform"),
            "ragged_4097x3001x2053": (4097, 3001, 2053, 3, "normal"),
            "square_8192": (8192, 8192, 8192, 4, "uniform"),
            "skinny_65536x128x4096": (65536, 128, 4096, 4, "uniform")}
    got = {n: (w.M, w.N, w.K, w.seed, w.dist) for n, w in gi.WORKLOADS.items()}
    assert got == want
    assert gi.WORKLOADS["square_4096"].flops == 2 * 4096 ** 3


@pytest.mark.parametrize("dtype,tdt", [("bf16", torch.bfloat16), ("f16", torch.float16)])
def test_16bit_inputs_are_the_rounded_draws(dtype, tdt):
    A, B = gi.make_ab(40, 30, 20, 5, "normal")
    A16, B16 = gi.make_ab16(40, 30, 20, 5, "normal", dtype)
    assert A16.dtype == tdt and torch.equal(A16, A.to(tdt)) and torch.equal(B16, B.to(tdt))
