"""Host-side logic of bench.py: the multi-rank aggregation (max time over
ranks, whole-job rate) on two gloo ranks, the reference arm's rank handling,
and the peak / traffic bookkeeping. No GPU."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from conftest import ROOT

sys.path.insert(0, ROOT)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import bench

    dist = bench.init_dist(world, "gloo")
    t = bench.reduce_max(1.0 + rank, dist)          # rank 1 is the slowest
    rate = bench.aggregate_rate(1_000_000_000, 10, world, t)
    q.put((rank, t, rate))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_time_and_whole_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, rate in got:
        assert t == 2.0                               # max over ranks
        assert rate == pytest.approx(1e9 * 10 * 2 / 2.0 / 1e9)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_peak_and_traffic_bookkeeping():
    import bench

    peak, src = bench.hbm_peak()
    assert peak > 1000 and src in ("measured", "fallback")
    assert len(bench.gemm_source_hash()) == 16
    t = bench.recorded_traffic()
    assert t is None or t > 0
    assert bench.aggregate_rate(10, 4, 1, 2.0) == pytest.approx(20 / 1e9)


def test_warmup_floor():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "1"],
                       capture_output=True, text=True, timeout=60)
    assert r.returncode != 0


def test_quantiles_interpolate():
    import bench

    assert bench.quantiles([3.0, 1.0, 2.0], (0.0, 0.5, 1.0)) == [1.0, 2.0, 3.0]
    assert bench.quantiles([0.0, 10.0], (0.1, 0.9)) == pytest.approx([1.0, 9.0])
    assert bench.quantiles([5.0]) == [5.0, 5.0, 5.0]
