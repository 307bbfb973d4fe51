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


def test_reference_arm_line_on_rank0():
    """Rank 0 of the reference arm times the oracle on the host cores on the CUDA arm's
    workload (decode + layer-shaped prefill) and prints one JSON line with the same metric,
    unit and workload name as the CUDA arm."""
    sys.path.insert(0, ROOT)
    import bench
    from softmax_covariance_correction_pass_b300 import configs

    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "1"], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference"
    assert j["metric"] == bench.METRIC and j["unit"] == "GB/s" and j["higher_is_better"] is True
    assert j["config"]["workload"] == (configs.DECODE_UNIFORM["name"] + " + "
                                       + configs.LAYER_PREFILL["name"])
    assert j["steps"] == 2 and j["warmup"] == 1 and j["value"] > 0
    assert j["decode"]["value"] == j["value"] and j["prefill"]["value"] > 0
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["value"] == j["value"]
    assert j["cpu_baseline"]["cores"] >= 1
    assert j["e2e"] == {"value": j["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert j["gpu_launches"] == 0


def test_clock_sampler_summary():
    """The clock record that decides whether a timed run stands: median SM clock under load,
    the maximum clock, and every throttle reason seen Active (nvidia-smi csv, no units)."""
    sys.path.insert(0, ROOT)
    import bench

    s = bench.ClockSampler("0")
    s.out = "\n".join([
        "0, 1920, 2032, 150.2, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2032, 540.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 1935, 2032, 610.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 1950, 2032, [N/A], 0x0, Not Active, Not Active, Not Active, Not Active",  # skipped
        "garbage line",
    ])
    r = s.summary()
    assert r["samples"] == 3
    assert r["sm_mhz"] == 1957.5             # median of the two samples above 250 W
    assert r["sm_max_mhz"] == 2032.0
    assert r["reasons"] == ["sw_power_cap"]
    assert r["power_w_max"] == 610.5
    s.out = "0, 1200, 2032, 500, 0x8, Active, Not Active, Active, Not Active"
    assert s.summary()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    s.out = ""
    assert s.summary(max_mhz_hint=2032) == {"sm_mhz": None, "sm_max_mhz": 2032, "reasons": [],
                                            "samples": 0}
