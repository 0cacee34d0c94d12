"""The N > 1 path of bench.py on CPU: two gloo ranks (replicas, no collective
on the data path).  The whole-job value is the bytes of all replicas over the
slowest replica's step time, and only rank 0 runs the reference arm."""
from __future__ import annotations

import os
import socket
import sys
from pathlib import Path

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = Path(__file__).resolve().parents[1]


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    sys.path.insert(0, str(ROOT))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        assert bench.dist_setup() == (world, rank, rank)
        ms = bench.max_over_ranks(1.0 + rank)  # rank r took (1 + r) ms per step
        gbs = bench.whole_job_gbs(1_000_000_000, world, ms)

        class Args:
            steps, warmup, config, layout, ref_budget = 1, 0, "tiny", "split", 1.0
        ref = bench.run_reference(Args, world, rank) if rank != 0 else "rank0"
        out.put((rank, ms, gbs, ref))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_and_sum_the_bytes():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms, gbs, ref in res:
        assert ms == 2.0                                  # max over ranks
        assert abs(gbs - 2 * 1e9 / 2e-3 / 1e9) < 1e-9     # 2 GB over 2 ms
    assert res[1][3] is None                              # rank 1: no reference work
