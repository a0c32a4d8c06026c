"""The N > 1 host logic of bench.py on CPU: world-size-2 gloo ranks on
127.0.0.1 (the replicas path has no data-path collective; only the timing
reduction and the rank-0 report are multi-rank)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, local_ms, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(dist, local_ms[rank], torch.device("cpu"))
        out[rank] = (slowest, bench.whole_job_rate(1e9, 10, world, slowest))
    finally:
        dist.destroy_process_group()


def test_timing_reduction_takes_the_slowest_rank():
    world, local_ms = 2, [12.5, 20.0]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), local_ms, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        slowest, rate = res[r]
        assert slowest == 20.0                              # every rank sees the max
        assert rate == pytest.approx(1e9 * 10 * 2 / 20e-3)  # all ranks' units over the slowest time


def test_reference_arm_reports_on_rank_zero_only():
    env = dict(os.environ, WORLD_SIZE="2", MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    outs = []
    for rank in (0, 1):
        e = dict(env, RANK=str(rank), LOCAL_RANK=str(rank))
        p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                            "tail_130x70x65_b_rowmajor", "--steps", "3", "--warmup", "3", "--gpus", "2"],
                           env=e, capture_output=True, text=True, timeout=600)
        assert p.returncode == 0, p.stderr[-2000:]
        outs.append(p.stdout.strip())
    assert outs[1] == ""
    line = json.loads(outs[0].splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
