"""The N > 1 host logic of bench.py, run as two gloo ranks on the CPU.

On several GPUs every rank denoises its own segment (independent problems, no data-path
collective); the only exchange is the max over ranks of the timed region.  These tests run
that reduction, the whole-job throughput formula and the reference arm's rank gating with
world_size 2 over gloo.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [120.0, 150.0][rank]                 # rank 1 is the slowest
        slowest = bench.max_over_ranks(local_ms, world)
        value = bench.job_throughput(4.0e12, 10, world, slowest)
        q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo_world_2():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get() for _ in range(2))
    for rank, slowest, value in got:
        assert slowest == 150.0                          # every rank sees the slowest rank's time
        # 2 ranks x 10 steps x 4 TFLOP in 150 ms
        assert value == pytest.approx(2 * 10 * 4.0e12 / 0.150 / 1e12)


def test_job_throughput_single_rank_is_plain_ratio():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_throughput(1e12, 4, 1, 2000.0) == pytest.approx(2.0)


def test_reference_arm_non_zero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_reference_arm_rank0_prints_one_json_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--workload", "sweep:0:4"], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
