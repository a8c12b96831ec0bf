"""The N>1 path of bench.py, on CPU with two gloo ranks.  The decode path
shards as replicas (one independent batch per GPU, no collective on the data
path); what spans ranks is the timing: the job's step takes the slowest
rank's time and the whole-job rate counts every rank's bytes.  The reference
arm prints from rank 0 only."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, per_rank_ms, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sys.path.insert(0, ROOT)
        import bench
        ms = bench.max_over_ranks(per_rank_ms[rank], world, "cpu")
        rate = bench.whole_job_gbs(2.0e8, ms, world)
        torch.distributed.barrier()
        out.put((rank, ms, rate))
    finally:
        torch.distributed.destroy_process_group()


def test_two_ranks_take_the_slowest_rank_time():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    per_rank_ms = [0.25, 0.40]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, per_rank_ms, out))
             for r in range(2)]
    for p in procs:
        p.start()
    results = [out.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sorted(r for r, _, _ in results) == [0, 1]
    for _, ms, rate in results:
        assert ms == pytest.approx(0.40)  # every rank sees the slowest time
        # two ranks x 200 MB per step in 0.40 ms
        assert rate == pytest.approx(2 * 2.0e8 / 0.40e-3 / 1e9)


def test_one_rank_is_its_own_time():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.5, 1, "cpu") == 1.5
    assert bench.whole_job_gbs(1.0e9, 1.0, 1) == pytest.approx(1000.0)


def test_reference_arm_prints_from_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "3", "--warmup", "3"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [line for line in r.stdout.splitlines() if line.strip().startswith("{")]


def test_bench_line_contract_keys():
    """The JSON keys the driver reads, as bench.py builds its line (checked on
    the source, since the line itself needs a GPU)."""
    src = open(os.path.join(ROOT, "bench.py")).read()
    for key in ('"metric"', '"value"', '"unit"', '"n_gpus"', '"steps"', '"warmup"',
                '"ms_per_step"', '"higher_is_better"', '"scaling"', '"vs_baseline"', '"dtype"',
                '"data"', '"config"', '"roofline"', '"cpu_baseline"', '"e2e"', '"gpu_launches"',
                '"clocks"'):
        assert key in src, key
    json.dumps({})  # the line is plain JSON
