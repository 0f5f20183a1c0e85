"""The benchmark's multi-rank bookkeeping on CPU: two gloo ranks.

The GEMM does not shard (every rank runs its own replica), so the only
cross-rank steps are the barrier and the max-over-ranks timing; `value`
counts the work of all ranks over the slowest rank's time.  The reference
arm prints from rank 0 only.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # Rank r "measured" 10 + r milliseconds; every rank must see the max.
    slowest = bench.reduce_max(10.0 + rank, "cpu")
    value = bench.job_tflops(world, 2.0 * 4096 ** 3, 5, slowest * 5 / 1e3)
    dist.barrier()
    # The reference arm: only rank 0 runs and prints; the others exit 0.
    buf = io.StringIO()
    rc = None
    if rank != 0:
        class A:  # the parsed arguments run_reference reads
            gpus, steps, warmup = world, 1, 0
        with redirect_stdout(buf):
            rc = bench.run_reference(A())
    out[rank] = (slowest, value, rc, buf.getvalue())
    dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 11.0
    # 2 ranks x 5 steps x 2*4096^3 flops in 5 x 11 ms.
    want = 2 * 2.0 * 4096 ** 3 * 5 / (5 * 11e-3) / 1e12
    assert res[0][1] == pytest.approx(want) and res[1][1] == pytest.approx(want)
    assert res[1][2] == 0 and res[1][3] == ""


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5, "cpu") == 3.5
    assert bench.job_tflops(1, 1e12, 2, 2.0) == pytest.approx(1.0)
