"""The one-process-per-GPU launch (replicas, weak scaling) without a GPU: the
host logic of bench.py's N > 1 path on world_size-2 gloo ranks (rank layout from
the launcher's environment, the slowest rank's time on every rank, the
whole-job aggregate), and a torchrun launch of the reference arm, where rank 0
alone runs and prints and the other rank exits 0 without work."""
from __future__ import annotations

import json
import multiprocessing as mp
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


def _rank_main(rank: int, world: int, port: int, out) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.rank_env()
        elapsed = 10.0 + 5.0 * rank            # the second rank is the slow one
        slowest = bench.max_over_ranks(elapsed, dist, device="cpu")
        value = bench.job_throughput(1000, w, slowest)
        dist.barrier()
        out.put((rank, r, w, local, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_total():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (r, r_env, w, local, slowest, value) in enumerate(got):
        assert (r, r_env, w, local) == (rank, rank, world, rank)
        assert slowest == 15.0                      # max over ranks, seen by every rank
        assert value == pytest.approx(2 * 1000 / 0.015)   # both replicas' tokens / slowest


def test_single_process_defaults():
    sys.path.insert(0, ROOT)
    import bench
    env = {k: os.environ.pop(k) for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK") if k in os.environ}
    try:
        assert bench.rank_env() == (0, 1, 0)
        assert bench.max_over_ranks(3.5) == 3.5
        assert bench.job_throughput(500, 1, 2.0) == pytest.approx(250000.0)
    finally:
        os.environ.update(env)


def test_torchrun_reference_arm_prints_once_from_rank_zero(tmp_path):
    """Two processes under torch.distributed.run: one JSON line (rank 0, the CPU
    oracle on a tiny sample), rank 1 exits 0."""
    env = dict(os.environ, KATA_REF_STEP_SECONDS="0.2", OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--workload", "small_fp32", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
