"""Host-side logic of bench.py without a GPU: the multi-rank aggregation (world size 2 over gloo,
one process per rank, as torchrun would launch them), the reference arm (the fp64 oracle on the
host cores) and its behaviour on ranks other than 0."""

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


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [3.0, 5.0][rank]
        worst = bench.max_over_ranks(ms, world)
        q.put((rank, worst, bench.job_tflops(1e12, 10, world, worst)))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_job_throughput():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    # Both ranks see the slowest rank's time; the value counts both ranks' work.
    assert [r[1] for r in res] == [5.0, 5.0]
    assert res[0][2] == pytest.approx(1e12 * 10 * 2 / 5e-3 / 1e12)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.job_tflops(2e12, 4, 1, 1000.0) == pytest.approx(8.0)


def _run_bench(env_extra, *args):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          env=env, timeout=600)


def test_reference_arm_prints_one_line():
    r = _run_bench({}, "--impl", "reference", "--steps", "3", "--warmup", "3")
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["metric"] == bench.METRIC and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["B"] == 2 and line["config"]["N"] == 4096


def test_reference_arm_other_ranks_exit_quietly():
    r = _run_bench({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, "--impl", "reference", "--steps", "3",
                   "--warmup", "3")
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_warmup_floor_enforced():
    r = _run_bench({}, "--impl", "reference", "--steps", "3", "--warmup", "2")
    assert r.returncode != 0
