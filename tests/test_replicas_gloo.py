"""The N > 1 path of bench.py on CPU: two gloo ranks (replicas, no collective
on the data path).  The whole-job value is the bytes of all replicas over the
slowest replica's step time, and only rank 0 runs the reference arm.  The CLI
case runs `bench.py --gpus 2` itself, which launches the two ranks."""
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
        if rank == 0:
            dist.barrier()  # the barrier rank 1 takes inside run_reference
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


def test_cli_gpus_2_launches_two_ranks_and_prints_one_line():
    """`bench.py --gpus 2` with no launcher around it starts two ranks (torch's
    launcher over 127.0.0.1), each joins the process group, and rank 0 alone
    prints one JSON line for the whole job."""
    import json
    import subprocess
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--gpus", "2", "--impl", "reference",
                        "--config", "tiny", "--steps", "1", "--warmup", "3", "--ref-budget", "2"],
                       cwd=str(ROOT), env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["config"]["name"] == "tiny" and d["value"] > 0
    for rank in range(2):
        assert f"rank {rank} of 2 joined" in r.stderr


def test_cli_rejects_a_world_size_that_differs_from_gpus():
    import subprocess
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--gpus", "2", "--impl", "reference",
                        "--config", "tiny"], cwd=str(ROOT), env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode != 0 and "WORLD_SIZE" in r.stderr
