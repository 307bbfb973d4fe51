"""Host logic of the multi-GPU bench path on CPU: world size 2 over gloo.

Each rank runs a full replica of the workload (the path shards by batch and
heads with no data exchange); the bench takes the slowest rank's time
(all-reduce MAX) and reports the whole job's units over that time.  These tests
run that reduction and aggregation on two gloo ranks, and check that the
reference arm's rank 1 exits without work.
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


def _rank_main(rank, ws, port, values, out):
    import torch
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        m = bench.reduce_max(values[rank], torch.device("cpu"), ws)
        rate = bench.whole_job_rate(ws, 1000.0, m)
        dist.barrier()
        out.put((rank, m, rate))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate():
    ws, port = 2, _free_port()
    values = [3.25, 7.5]  # per-rank milliseconds
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, values, out)) for r in range(ws)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, rate in res:
        assert m == max(values)                          # every rank sees the slowest time
        assert rate == pytest.approx(ws * 1000.0 / (max(values) * 1e-3))


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.reduce_max(4.0, None, 1) == 4.0
    assert bench.whole_job_rate(1, 10.0, 2.0) == pytest.approx(5000.0)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""  # only rank 0 prints the line
