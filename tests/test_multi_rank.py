"""Replicas path of bench.py on CPU ranks (gloo, world size 2).

The MoE path does not shard, so several GPUs run independent replicas; the
only multi-rank logic is the timing contract: a barrier around the timed
region, the max of the per-rank times, and the sum of the units every rank
processed.  These tests run that logic as two gloo processes on the CPU.
"""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, w = bench.dist_env()
        bench.barrier(w)
        # rank r took (r + 1) seconds for 10 * (r + 1) tokens
        sec, units = bench.aggregate(float(r + 1), 10.0 * (r + 1), w)
        q.put((r, lr, w, sec, units))
    finally:
        dist.destroy_process_group()


def test_aggregate_is_max_time_and_sum_of_units_over_two_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=5) for _ in range(2))
    for r, (rank, local_rank, world, sec, units) in enumerate(got):
        assert (rank, local_rank, world) == (r, r, 2)
        assert sec == 2.0          # the slowest rank's time
        assert units == 30.0       # 10 + 20 tokens over both ranks


def test_aggregate_is_identity_on_one_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(1.5, 7.0, 1) == (1.5, 7.0)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--workload", "tiny", "--steps", "3", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2
    assert rec["value"] > 0 and rec["unit"] == "tok/s"
    assert rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0


if __name__ == "__main__":
    sys.exit(pytest.main([__file__, "-q"]))
