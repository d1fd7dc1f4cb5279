"""Multi-rank host logic of bench.py, on CPU with the gloo backend (world size 2).

The layer does not shard: with N GPUs each rank runs an independent replica of the forward on
its own tokens, and only the timing is reduced (MAX over ranks). These tests check that
reduction, the per-rank inputs and the whole-job rate, and that under torchrun the reference
arm prints exactly one line (rank 0's) while the other ranks exit 0.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synthetic  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (r + 1) * 10 ms in total: the job is as slow as the slowest rank
        total_ms = bench.max_over_ranks(10.0 * (rank + 1), world)
        spec = synthetic.CONFIGS[1]
        seeds = [bench.batch_seed(spec, rank, b, 8) for b in range(8)]
        q.put((rank, total_ms, seeds))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_per_rank_inputs_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got.sort()
    assert [g[1] for g in got] == [20.0, 20.0]  # both ranks see the slowest rank's time
    s0, s1 = set(got[0][2]), set(got[1][2])
    assert len(s0) == 8 and len(s1) == 8 and not (s0 & s1)  # no rank repeats another's tokens


def test_whole_job_rate_counts_every_rank():
    assert bench.whole_job_rate(1, 4096, 5, 1.0) == 4096 * 5
    assert bench.whole_job_rate(8, 1, 50, 0.5) == 8 * 50 / 0.5
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--config", "0", "--steps", "2", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 2
    assert line["value"] > 0 and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle"
