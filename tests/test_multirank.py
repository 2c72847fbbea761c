"""The N > 1 path of bench.py on CPU: two gloo ranks (127.0.0.1).  The hot path shards with no
exchange (every rank runs an independent replica), so the only collective is the timing
reduction: the whole-job time is the slowest rank's and the throughput counts every rank's
units.  The reference arm runs on rank 0 only; the other ranks exit at once without work."""
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


def _rank_main(rank, world, port, local_ms, units, results):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, value = bench.aggregate(local_ms[rank], units, world)
        results[rank] = (ms, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_all_units():
    world, units = 2, 6.0e8  # bytes each replica moves per step
    local_ms = [0.125, 0.25]
    ctx = mp.get_context("spawn")
    port = _free_port()
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, local_ms, units, results))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        got = dict(results)
    for r in range(world):
        ms, value = got[r]
        assert ms == pytest.approx(0.25)
        assert value == pytest.approx(units * world / 0.25e-3)


def test_single_rank_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench

    ms, value = bench.aggregate(0.5, 1.0e9, 1)
    assert ms == 0.5 and value == pytest.approx(2.0e12)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "3", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_reference_arm_line_echoes_steps_and_warmup():
    # the oracle arm runs --warmup untimed and --steps timed steps, each over a bounded sample
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "1", "--reference-seconds", "2"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 3 and line["warmup"] == 1
    assert line["value"] > 0 and line["unit"] == "GB/s"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
