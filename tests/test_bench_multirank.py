"""The benchmark's multi-process logic on the CPU: world size 2 over gloo.

Each rank runs its own copy of the workload (weak scaling, no collective on the data path); the
job's time is the slowest rank's, and the whole-job value counts every rank's work. The reference
arm runs on rank 0 only and prints one JSON line; other ranks exit 0 without output.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        elapsed = 100.0 + 10.0 * rank          # the ranks' own timings
        slowest = bench.max_over_ranks(elapsed, world)
        value = bench.aggregate_value(2.0e12, 4, elapsed, world)
        out[rank] = (slowest, value)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_over_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    for rank in range(world):
        slowest, value = res[rank]
        assert slowest == 110.0                 # max over ranks, the same on every rank
        # 2 ranks x 4 steps x 2e12 FLOP in 110 ms
        assert value == pytest.approx(2 * 4 * 2.0e12 / 0.110 / 1e12)


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_runs_on_rank_zero_only(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                          "--steps", "1", "--warmup", "0"], capture_output=True, text=True, env=env, timeout=600)
    assert res.returncode == 0, res.stderr
    lines = [l for l in res.stdout.splitlines() if l.strip()]
    if rank != 0:
        assert lines == []
    else:
        assert len(lines) == 1
        d = json.loads(lines[0])
        assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["n_gpus"] == 2
        assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
        assert d["warmup"] >= 3 and d["steps"] == 1
