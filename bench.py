#!/usr/bin/env python3
"""Benchmark of the Parallax attention forward hot path (one JSON line on stdout).

A step is one pass of the whole hot path over synthetic inputs resident in HBM:
  * single-token decode, bf16 KV cache, B=64, H=16, d=128, 8192 keys per head
    (split-KV decode kernel + log-sum-exp combine), and
  * causal prefill, bf16, B=8, H=16, L=4096, d=128, with q, k, v, rho produced
    by random projections of x (width 2048) (tcgen05 tensor-core kernel).
`value` is the decode KV-stream bandwidth (GB/s); the prefill throughput
(TFLOP/s) is reported in the `prefill` object.  Both kernels also get a
roofline entry against the measured B300 peaks.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the only reference this method
has) on the host cores, on bounded samples of the same decode workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode KV-stream GB/s (% B300 HBM peak); causal prefill TFLOP/s (% TC peak)"

# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) comes from the ncu
# captures listed in profiles/dram_traffic.md, one table row per kernel: the captured case, its
# bytes, the factor that scales it to the bench's launch (units processed), and a hash of the
# kernel's source file and the csrc headers it includes at capture time.  A figure whose hash no
# longer matches the source is reported as null: the kernel has changed since the counters were
# taken.
TRAFFIC_TABLE = os.path.join(ROOT, "profiles", "dram_traffic.md")
CSRC = os.path.join(ROOT, "softmax_covariance_correction_pass_b300", "csrc")


def source_hash(cu_name: str) -> str:
    """sha256 (first 16 hex digits) of csrc/<cu_name> followed by the csrc headers (.cuh) it
    includes, transitively, in include order."""
    import hashlib
    import re

    seen, order = set(), []

    def walk(name):
        if name in seen:
            return
        seen.add(name)
        order.append(name)
        with open(os.path.join(CSRC, name), "rb") as f:
            text = f.read().decode()
        for inc in re.findall(r'#include\s+"([^"/]+\.cuh)"', text):
            walk(inc)

    walk(cu_name)
    h = hashlib.sha256()
    for name in order:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic(path: str = TRAFFIC_TABLE) -> dict:
    """kernel -> {"bytes": scaled read+write bytes per bench launch or None, ...} from the
    table in profiles/dram_traffic.md (rows whose first cell is a kernel name)."""
    out = {}
    try:
        with open(path) as f:
            lines = f.read().splitlines()
    except OSError:
        return out
    for line in lines:
        cells = [c.strip().strip("`") for c in line.strip().strip("|").split("|")]
        if len(cells) < 7 or not cells[0].endswith("_kernel"):
            continue
        try:
            kernel, src, case = cells[0], cells[1], cells[2]
            rd, wr, scale = float(cells[3]), float(cells[4]), float(cells[5])
            sha = cells[6]
        except ValueError:
            continue
        try:
            fresh = source_hash(src) == sha
        except OSError:
            fresh = False
        out[kernel] = {"bytes": (rd + wr) * scale if fresh else None,
                       "captured": case, "scale": scale, "source": src,
                       "note": "profiles/dram_traffic.md" if fresh else
                       f"stale: {src} changed since the capture (profiles/dram_traffic.md)"}
    return out


def traffic_of(table: dict, *kernels: str):
    """Summed traffic of the kernels of one call, or None if any of them has no fresh figure."""
    vals = [table.get(k, {}).get("bytes") for k in kernels]
    return None if any(v is None for v in vals) else sum(vals)


def traffic_notes(table: dict, *kernels: str) -> dict:
    return {k: table.get(k, {"note": "not captured"}) for k in kernels}


TRAFFIC = load_traffic()


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--only", choices=["decode", "prefill", "projection", "backward", "gqa", "lla",
                                       "chunk"],
                    default=None,
                    help="time one kernel alone (profiling runs); the default times both")
    ap.add_argument("--decode-batch", type=int, default=None,
                    help="override the decode batch (profiling runs on smaller cases)")
    ap.add_argument("--prefill-batch", type=int, default=None,
                    help="override the prefill batch (profiling runs on smaller cases)")
    ap.add_argument("--no-projection", action="store_true",
                    help="skip the q/k/v/probe projection leg")
    ap.add_argument("--no-backward", action="store_true", help="skip the prefill backward leg")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the decode sweep grid reported beside the step")
    ap.add_argument("--wr-zero", action="store_true",
                    help="time the W_R = 0 path (rho = NULL) in the step instead of the "
                         "correction path (profiling runs)")
    ap.add_argument("--serving", action="store_true",
                    help="instead of the step: time the serving variants (grouped-query decode, "
                         "paged ragged decode, chunked prefill), one JSON line each")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the step: time the decode sweep cells and the ragged-batch "
                         "decode, one JSON line per case (plus a markdown table on stderr)")
    return ap.parse_args(argv)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
                "source": "fallback"}


# ----------------------------------------------------------------------------- workloads
def decode_bytes(B, H, n, d, elem=2):
    kv = 2 * B * H * n * d * elem                 # K and V rows streamed once
    io = 2 * B * H * d * elem + B * H * d * 4 + B * 4  # q, rho in; o out; seqlens
    return kv, kv + io


def prefill_flops(B, H, L, d):
    # four causal contractions (S, R, U, W), each 2*d flop per (query, visible key)
    return 8.0 * d * (L * (L + 1) / 2) * B * H


def reduce_max(x: float, dev, ws: int) -> float:
    """The largest of the ranks' values (each rank passes its own); ws == 1: x itself."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], device=dev, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(ws: int, units_per_rank: float, max_ms: float) -> float:
    """Units per second of the whole job: every replica processes units_per_rank, the job
    takes as long as its slowest rank (weak scaling, no exchange between replicas)."""
    return ws * units_per_rank / (max_ms * 1e-3)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi samples of SM clock / throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", self.gpu_id], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self, max_mhz_hint=None):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": max_mhz_hint, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v == "Active"})
        busy = [r for r in rows if r[2] > 250.0] or rows
        return {"sm_mhz": statistics.median(r[0] for r in busy), "sm_max_mhz": rows[0][1],
                "reasons": reasons, "samples": len(rows), "power_w_max": max(r[2] for r in rows)}


# ----------------------------------------------------------------------------- CPU oracle
def cpu_oracle_decode_sample(inp, target_s: float, max_batches: int = 64):
    """Time the fp64 oracle (explicit covariance form, OpenMP over heads) on the first
    b sequences of the decode workload; b grows until about target_s of CPU work."""
    import numpy as np

    import oracle

    B, H, Lmax, d = inp.k_cache.shape
    n = int(inp.seqlens[0])

    def host(b):
        return [np.ascontiguousarray(t[:b].to("cpu").double().numpy()) for t in
                (inp.q, inp.rho, inp.k_cache, inp.v_cache)] + [inp.seqlens[:b].cpu().numpy()]

    b = 1
    while True:
        q, rho, kc, vc, sl = host(b)
        t0 = time.perf_counter()
        oracle.decode(q, rho, kc, vc, sl, form="explicit")
        dt = time.perf_counter() - t0
        if dt >= 0.25 * target_s or b >= max_batches:
            break
        b = min(max_batches, max(b + 1, int(b * min(8.0, 0.6 * target_s / max(dt, 1e-3)))))
    _, total = decode_bytes(b, H, n, d)
    return {"value": total / dt / 1e9, "unit": "GB/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{b * H} of {B * H} heads x {n} keys (explicit d x d covariance, fp64), "
                      f"{dt:.2f} s"}


# ----------------------------------------------------------------------------- reference arm
def run_reference(args):
    """The oracle timed on the host cores, on the same step as the CUDA arm: per step a bounded
    sample of the decode workload (the H heads of one sequence) and of the layer-shaped causal
    prefill (query rows of one head spread over the causal range), both with the explicit d x d
    covariance in fp64.  `value` is the decode part's KV-stream GB/s, as in the CUDA arm; the
    prefill part's TFLOP/s (8 d flop per visible (query, key) pair) is reported beside it."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np
    import torch

    import oracle
    from softmax_covariance_correction_pass_b300 import configs

    c = configs.DECODE_UNIFORM
    B, H, d, n = c["B"], c["H"], c["d"], c["ctx"]
    # the same seeded recipes, drawn on the host
    inp = configs.decode_inputs(B, H, d, n, n, c["seed"], c["rho_std"], device="cpu")
    q = inp.q.double().numpy()
    rho = inp.rho.double().numpy()
    pc = configs.LAYER_PREFILL
    pin = configs.layer_prefill_inputs(device="cpu", B=1)
    PH, PL, Pd = pc["H"], pc["L"], pc["d"]
    pq, pr = pin.q[0].double().numpy(), pin.rho[0].double().numpy()
    pk, pv = pin.k[0].double().numpy(), pin.v[0].double().numpy()
    # about two minutes for the whole run, half for each part
    budget = 60.0 / max(1, args.steps + args.warmup)
    t0 = time.perf_counter()
    oracle.decode(q[:1], rho[:1], inp.k_cache[:1].double().numpy(),
                  inp.v_cache[:1].double().numpy(), inp.seqlens[:1].numpy(), form="explicit")
    t_one = time.perf_counter() - t0
    keys = n if t_one <= budget else max(256, int(n * budget / t_one) // 256 * 256)
    kh = [inp.k_cache[b:b + 1, :, :keys].double().numpy() for b in range(min(B, 8))]
    vh = [inp.v_cache[b:b + 1, :, :keys].double().numpy() for b in range(min(B, 8))]
    sl = np.full(1, keys, dtype=np.int32)

    def prefill_rows(step, R):
        h = step % PH
        idx = (np.arange(R, dtype=np.int64) * PL // R + 7 * step) % PL
        return h, idx

    h, idx = prefill_rows(0, 16)
    t0 = time.perf_counter()
    oracle.rows(pq[h, idx], pr[h, idx], pk[h], pv[h], idx + 1, pin.scale, form="explicit")
    t16 = time.perf_counter() - t0
    R = int(min(1024, max(8, 16 * budget / max(t16, 1e-4))) // 8 * 8)

    dec_t, pre_t, pre_flops = [], [], 0.0
    for s in range(args.warmup + args.steps):
        b = s % len(kh)
        t0 = time.perf_counter()
        oracle.decode(q[b:b + 1], rho[b:b + 1], kh[b], vh[b], sl, form="explicit")
        t1 = time.perf_counter()
        h, idx = prefill_rows(s, R)
        oracle.rows(pq[h, idx], pr[h, idx], pk[h], pv[h], idx + 1, pin.scale, form="explicit")
        t2 = time.perf_counter()
        if s >= args.warmup:
            dec_t.append(t1 - t0)
            pre_t.append(t2 - t1)
            pre_flops += 8.0 * Pd * float((idx + 1).sum())
    _, per_step = decode_bytes(1, H, keys, d)
    value = per_step * len(dec_t) / sum(dec_t) / 1e9
    pre_tflops = pre_flops / sum(pre_t) / 1e12
    sample = (f"per step: decode {H} heads x {keys} keys of one sequence of the B={B} decode "
              f"workload; prefill {R} query rows (keys 0..row) of one head of a B=1 draw of the "
              f"layer-shaped causal prefill; explicit d x d covariance, fp64")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * (sum(dec_t) + sum(pre_t)) / len(dec_t), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": c["name"] + " + " + pc["name"], "sample": sample},
        "decode": {"metric": "decode KV-stream GB/s", "value": value, "unit": "GB/s",
                   "ms_per_call": 1e3 * sum(dec_t) / len(dec_t)},
        "prefill": {"metric": "causal prefill TFLOP/s", "value": pre_tflops, "unit": "TFLOP/s",
                    "rows_per_step": R, "ms_per_step": 1e3 * sum(pre_t) / len(pre_t)},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def time_projection(args, dev, peaks, max_over_ranks, n_rep=20):
    """The layer-shaped projection x [B, L, 2048] -> q, k, v, rho [B, H, L, d] (one tcgen05
    GEMM, 4*H*d output features), `n_rep` launches back to back after 3 warm-ups."""
    import torch

    import softmax_covariance_correction_pass_b300 as px
    from softmax_covariance_correction_pass_b300 import configs

    pc = configs.LAYER_PREFILL
    PB, PH, PL, Pd = args.prefill_batch or pc["B"], pc["H"], pc["L"], pc["d"]
    stream = torch.cuda.current_stream()
    x, w = configs.layer_projection_inputs(dev, B=PB)
    pq = [torch.empty((PB, PH, PL, Pd), dtype=torch.bfloat16, device=dev) for _ in range(4)]
    width = x.shape[-1]
    proj_flops = 2.0 * PB * PL * width * 4 * PH * Pd

    def project():
        px.parallax_attn_qkvr_projection(x, w, PH, Pd, *pq)

    for _ in range(max(args.warmup, 3)):
        project()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(n_rep):
        project()
    b.record(stream)
    torch.cuda.synchronize()
    proj_ms = max_over_ranks(a.elapsed_time(b) / n_rep)
    if px.parallax_check_device_error() != 0:
        raise RuntimeError("device error in the projection")
    proj_tf = proj_flops / (proj_ms * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": proj_tf, "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": proj_tf / peaks["bf16_tflops"],
            "traffic": traffic_of(TRAFFIC, "proj_kernel"),
            "traffic_source": traffic_notes(TRAFFIC, "proj_kernel"), "kernel": "proj_kernel",
            "algorithmic_flops_per_launch": proj_flops, "avg_launch_ms": proj_ms,
            "launches": n_rep,
            "shape": f"x [{PB},{PL},{width}] x W^T [{width},{4 * PH * Pd}] -> q,k,v,rho "
                     f"[{PB},{PH},{PL},{Pd}] bf16",
            "peak_source": peaks["source"] + f" (burst: timed alone, {n_rep} launches)"}


def time_backward(args, dev, peaks, max_over_ranks, n_rep=10):
    """Backward pass of the layer-shaped causal prefill (B=8, H=16, L=4096, d=128): the
    training forward once (for lse, rbar, mu_v), then `n_rep` backward calls back to back
    after warm-ups.  Algorithmic work: 8 causal contractions (S, R recomputed, D = dout V^T,
    dV, the two dK terms, dQ, drho) = 16 d flop per (query, visible key)."""
    import torch

    import softmax_covariance_correction_pass_b300 as px
    from softmax_covariance_correction_pass_b300 import configs

    pc = configs.LAYER_PREFILL
    PB = args.prefill_batch or pc["B"]
    inp = configs.layer_prefill_inputs(dev, B=PB)
    B, H, L, d = inp.q.shape
    g = torch.Generator(device=dev).manual_seed(44)
    dout = torch.randn(inp.q.shape, generator=g, device=dev).to(torch.bfloat16)
    o, lse, rbar, mu = px.parallax_attn_prefill_train(inp.q, inp.rho, inp.k, inp.v, causal=True,
                                                      scale=inp.scale)
    stream = torch.cuda.current_stream()
    flops = 16.0 * d * (L * (L + 1) / 2) * B * H

    def backward():
        return px.parallax_attn_prefill_backward(inp.q, inp.rho, inp.k, inp.v, o, mu, lse, rbar,
                                                 dout, causal=True, scale=inp.scale)

    for _ in range(max(args.warmup, 3)):
        backward()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(n_rep):
        backward()
    b.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b) / n_rep)
    if px.parallax_check_device_error() != 0:
        raise RuntimeError("device error in the backward pass")
    tf = flops / (ms * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": tf / peaks["bf16_tflops"],
            "traffic": traffic_of(TRAFFIC, "bwd_pre_kernel", "bwd_kv_kernel", "bwd_q_kernel"),
            "traffic_source": traffic_notes(TRAFFIC, "bwd_pre_kernel", "bwd_kv_kernel",
                                            "bwd_q_kernel"),
            "kernel": "bwd_pre_kernel + bwd_kv_kernel + bwd_q_kernel",
            "algorithmic_flops_per_launch": flops, "avg_launch_ms": ms, "launches": n_rep,
            "shape": f"causal prefill backward B={B} H={H} L={L} d={d}, bf16 in, fp32 grads",
            "tokens_per_s": B * L / (ms * 1e-3),
            "peak_source": peaks["source"] + f" (burst: timed alone, {n_rep} calls)"}


def run_projection_only(args):
    """--only projection: the projection leg alone (profiling runs), one JSON line."""
    import torch

    dev = torch.device("cuda", torch.cuda.current_device())
    import softmax_covariance_correction_pass_b300 as px

    px.load_library()
    r = time_projection(args, dev, load_peaks(), lambda x: x, n_rep=args.steps)
    print(json.dumps({"metric": "projection TFLOP/s", "value": r["achieved"], "unit": "TFLOP/s",
                      "steps": args.steps, "warmup": args.warmup, "roofline": r}), flush=True)
    return 0


# ----------------------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    import torch.distributed as dist

    import softmax_covariance_correction_pass_b300 as px
    from softmax_covariance_correction_pass_b300 import configs

    ws, rank, local = dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if ws > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    px.load_library()
    peaks = load_peaks()

    def barrier():
        if ws > 1:
            dist.barrier()

    def max_over_ranks(x: float) -> float:
        return reduce_max(x, dev, ws)

    # ---- inputs resident in HBM
    dc = configs.DECODE_UNIFORM
    B, H, d, n = args.decode_batch or dc["B"], dc["H"], dc["d"], dc["ctx"]
    dinp = configs.decode_uniform_inputs(dev, B=B)
    do = torch.empty((B, H, d), dtype=torch.float32, device=dev)
    pc = configs.LAYER_PREFILL
    PB, PH, PL, Pd = args.prefill_batch or pc["B"], pc["H"], pc["L"], pc["d"]
    pinp = configs.layer_prefill_inputs(dev, B=PB)
    po = torch.empty((PB, PH, PL, Pd), dtype=torch.float32, device=dev)
    kv_bytes, dec_bytes = decode_bytes(B, H, n, d)
    pre_flops = prefill_flops(PB, PH, PL, Pd)
    if args.wr_zero:  # S and U only: two of the four contractions
        pre_flops /= 2
    chunk = px.parallax_attn_decode_chunk_keys(B, H, n, d, 2)
    dec_launches = 2 if chunk < n else 1
    dec_kernel = px.parallax_attn_decode_plan_kernel(B, H, H, n, d)
    dec_kernels = (dec_kernel, "combine_kernel") if chunk < n else (dec_kernel,)

    run_decode = args.only in (None, "decode")
    run_prefill = args.only in (None, "prefill")

    drho = None if args.wr_zero else dinp.rho
    prho = None if args.wr_zero else pinp.rho

    def decode():
        if run_decode:
            px.parallax_attn_decode(dinp.q, drho, dinp.k_cache, dinp.v_cache, dinp.seqlens, do)

    def prefill():
        if run_prefill:
            px.parallax_attn_prefill(pinp.q, prho, pinp.k, pinp.v, po, causal=True,
                                     scale=pinp.scale)

    for _ in range(max(args.warmup, 3)):
        decode()
        prefill()
    torch.cuda.synchronize()
    if px.parallax_check_device_error() != 0:
        raise RuntimeError("device error during warm-up")

    # ---- timed region: K steps, per-kernel events on the launching stream
    K = args.steps
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    props = torch.cuda.get_device_properties(dev)
    gpu_id = f"GPU-{props.uuid}" if getattr(props, "uuid", None) else str(dev.index)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(gpu_id) as clocks:
        t_start.record(stream)
        for k in range(K):
            ev[k][0].record(stream)
            decode()
            ev[k][1].record(stream)
            ev[k][2].record(stream)
            prefill()
            ev[k][3].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier()
    total_ms = t_start.elapsed_time(t_end)
    dec_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    pre_ms = sum(e[2].elapsed_time(e[3]) for e in ev) / K
    total_ms = max_over_ranks(total_ms)
    dec_ms = max_over_ranks(dec_ms)
    pre_ms = max_over_ranks(pre_ms)
    if px.parallax_check_device_error() != 0:
        raise RuntimeError("device error in the timed region")

    dec_ms = max(dec_ms, 1e-9)
    pre_ms = max(pre_ms, 1e-9)
    dec_gbs = dec_bytes / (dec_ms * 1e-3) / 1e9
    pre_tflops = pre_flops / (pre_ms * 1e-3) / 1e12
    value = whole_job_rate(ws, dec_bytes, dec_ms) / 1e9  # all replicas' bytes / slowest time

    roof_dec = {"bound": "hbm", "achieved": dec_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": dec_gbs / peaks["hbm_gbs"],
                "traffic": traffic_of(TRAFFIC, *dec_kernels),
                "traffic_source": traffic_notes(TRAFFIC, *dec_kernels),
                "kernel": " + ".join(dec_kernels),
                "algorithmic_bytes_per_launch": dec_bytes, "avg_launch_ms": dec_ms,
                "peak_source": peaks["source"]}
    # the prefill launches take about a millisecond each inside a timed region of tens of
    # milliseconds: the burst peak is the denominator (the sustained one is reported beside it)
    roof_pre = {"bound": "tensor", "achieved": pre_tflops, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": pre_tflops / peaks["bf16_tflops"],
                "traffic": traffic_of(TRAFFIC, "prefill_pair_kernel"),
                "traffic_source": traffic_notes(TRAFFIC, "prefill_pair_kernel"),
                "kernel": "prefill_pair_kernel",
                "algorithmic_flops_per_launch": pre_flops, "avg_launch_ms": pre_ms,
                "peak_sustained": peaks["bf16_tflops_sustained"],
                "frac_sustained": pre_tflops / peaks["bf16_tflops_sustained"],
                "peak_source": peaks["source"] + " (burst)"}
    if not run_decode:
        roof_dec = None
    if not run_prefill:
        roof_pre = None
    dominant = roof_pre if (run_prefill and (not run_decode or pre_ms >= dec_ms)) else roof_dec

    # ---- W_R = 0 fast paths (rho = NULL), for context
    f0 = {}
    for name, fn, units in () if args.only else (
            ("decode_gbs", lambda: px.parallax_attn_decode(dinp.q, None, dinp.k_cache,
                                                           dinp.v_cache, dinp.seqlens, do),
             dec_bytes / 1e9),
            ("prefill_tflops_softmax_only", lambda: px.parallax_attn_prefill(
                pinp.q, None, pinp.k, pinp.v, po, causal=True, scale=pinp.scale),
             pre_flops / 2 / 1e12)):
        fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(20):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        f0[name] = units / (a.elapsed_time(b) / 20 * 1e-3)

    # ---- torch's scaled_dot_product_attention (a library kernel, not this path) on the same
    # decode and prefill tensors, softmax attention only, for context beside the W_R = 0 paths
    sdpa = {}
    if not args.only:
        try:
            attn = torch.nn.functional.scaled_dot_product_attention
            qd = dinp.q.unsqueeze(2)
            for name, fn, units in (
                    ("decode_gbs", lambda: attn(qd, dinp.k_cache, dinp.v_cache), dec_bytes / 1e9),
                    ("prefill_tflops_softmax_only", lambda: attn(
                        pinp.q, pinp.k, pinp.v, is_causal=True, scale=pinp.scale),
                     pre_flops / 2 / 1e12)):
                fn()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(20):
                    fn()
                b.record(stream)
                torch.cuda.synchronize()
                sdpa[name] = units / (a.elapsed_time(b) / 20 * 1e-3)
        except Exception as e:  # context only: never fail the bench on it
            sdpa = {"error": f"{type(e).__name__}: {e}"[:300]}

    # ---- q/k/v/probe projection of the layer-shaped workload (one tcgen05 GEMM), timed alone
    proj = None
    if not args.only and not args.no_projection:
        proj = time_projection(args, dev, peaks, max_over_ranks)
    bwd = None
    if not args.only and not args.no_backward:
        bwd = time_backward(args, dev, peaks, max_over_ranks)
        torch.cuda.empty_cache()

    # ---- end to end through the public call, host buffers (pinned), copies timed
    e2e = None
    e2e_prefill = None
    if not args.no_e2e and not args.only:
        hq = [t.to("cpu").pin_memory() for t in (dinp.q, dinp.rho, dinp.k_cache, dinp.v_cache,
                                                  dinp.seqlens)]
        ho = torch.empty((B, H, d), dtype=torch.float32).pin_memory()
        dq = [torch.empty_like(t, device=dev) for t in hq]
        h2d = sum(t.numel() * t.element_size() for t in hq)
        d2h = ho.numel() * ho.element_size()

        def e2e_step():
            for src, dst in zip(hq, dq):
                dst.copy_(src, non_blocking=True)
            px.parallax_attn_decode(dq[0], dq[1], dq[2], dq[3], dq[4], do)
            ho.copy_(do, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(a.elapsed_time(b) / args.e2e_steps)
        e2e = {"value": ws * dec_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}
        del hq, dq

        hp = [t.to("cpu").pin_memory() for t in (pinp.q, pinp.rho, pinp.k, pinp.v)]
        hpo = torch.empty_like(po, device="cpu").pin_memory()
        dp = [torch.empty_like(t, device=dev) for t in hp]

        def e2e_prefill_step():
            for src, dst in zip(hp, dp):
                dst.copy_(src, non_blocking=True)
            px.parallax_attn_prefill(dp[0], dp[1], dp[2], dp[3], po, causal=True,
                                     scale=pinp.scale)
            hpo.copy_(po, non_blocking=True)

        e2e_prefill_step()
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(args.e2e_steps):
            e2e_prefill_step()
        b.record(stream)
        torch.cuda.synchronize()
        ep_ms = max_over_ranks(a.elapsed_time(b) / args.e2e_steps)
        e2e_prefill = {"value": ws * pre_flops / (ep_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                       "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in hp),
                       "d2h_bytes_per_step": hpo.numel() * hpo.element_size(),
                       "ms_per_step": ep_ms}
        del hp, dp

    # ---- the decode sweep grid (17 cells, batch 1-2048 x context 128-32768) and the ragged
    # batch, each timed alone; reported beside the step, not part of it
    sweep = None
    if not args.only and not args.no_sweep:
        sweep = [{"B": r["B"], "context": r["context"], "GB/s": round(r["GB/s"], 1),
                  "frac_of_hbm_peak": round(r["frac_of_hbm_peak"], 4), "ms": round(r["ms"], 5),
                  "chunk_keys": r["chunk_keys"], "l2": r["l2"]}
                 for r in sweep_rows(dev, peaks, include_boundary=False, include_ragged=True,
                                     quiet=True)]

    # ---- CPU oracle baseline (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_decode_sample(dinp, args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": K,
            "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {
                "workload": configs.DECODE_UNIFORM["name"] + " + " + configs.LAYER_PREFILL["name"],
                "decode": {"B": B, "H": H, "d": d, "context": n, "chunk_keys": chunk,
                           "kv_bytes": kv_bytes, "tokens_per_s": ws * B / (dec_ms * 1e-3)},
                "prefill": {"B": PB, "H": PH, "L": PL, "d": Pd, "causal": True,
                            "tokens_per_s": ws * PB * PL / (pre_ms * 1e-3)},
                "l2": "inputs larger than L2 (4.3 GB KV cache; 1.07 GB of prefill tensors)",
                "only": args.only,
                "w_r_zero": bool(args.wr_zero),
                "parallelism": f"replicas x{ws} (no collectives)"},
            "roofline": dominant,
            "roofline_decode": roof_dec,
            "roofline_prefill": roof_pre,
            "prefill": None if roof_pre is None else {
                "metric": "causal prefill TFLOP/s", "value": ws * pre_tflops, "unit": "TFLOP/s",
                "frac_of_peak": roof_pre["frac"], "ms_per_launch": pre_ms, "e2e": e2e_prefill},
            "decode": None if roof_dec is None else {
                "metric": "decode KV-stream GB/s", "value": value, "unit": "GB/s",
                "frac_of_peak": roof_dec["frac"], "ms_per_call": dec_ms},
            "w_r_zero_fast_path": f0,
            "torch_sdpa_w_r_zero": sdpa,
            "roofline_projection": proj,
            "roofline_backward": bwd,
            "decode_sweep": sweep,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "clocks": clocks.summary(),
            "gpu_launches": K * ((dec_launches if run_decode else 0) + (1 if run_prefill else 0)),
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


# ----------------------------------------------------------------------------- decode sweep
def sweep_rows(dev, peaks, include_boundary=True, include_ragged=True, quiet=False):
    """Decode over the sweep grid (batch x context, caches up to 64e9 bytes; optionally the
    64 GiB boundary cell, flagged) and the ragged batch.  Each case is timed with CUDA events
    per call; caches smaller than twice the L2 are evicted before every call by writing a
    512 MB buffer (not timed), larger ones are timed back to back."""
    import torch

    import softmax_covariance_correction_pass_b300 as px
    from softmax_covariance_correction_pass_b300 import configs

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    sw = configs.DECODE_SWEEP
    cases = [("sweep", B, L, False) for B, L in configs.decode_sweep_cells()]
    if include_boundary:
        cases += [("sweep", B, L, True) for B, L in configs.decode_sweep_cells(include_boundary=True)
                  if (B, L) not in configs.decode_sweep_cells()]
    if include_ragged:
        cases.append(("ragged", configs.DECODE_RAGGED["B"], configs.DECODE_RAGGED["hi"], False))
    rows = []
    for kind, B, L, boundary in cases:
        if kind == "sweep":
            inp = configs.decode_sweep_inputs(B, L, dev)
        else:
            inp = configs.decode_ragged_inputs(dev)
        H, d = sw["H"], sw["d"]
        keys = int(inp.seqlens.sum().item())
        kv = keys * H * d * 2 * 2
        total = kv + 2 * B * H * d * 2 + B * H * d * 4 + B * 4
        o = torch.empty((B, H, d), dtype=torch.float32, device=dev)
        call = lambda: px.parallax_attn_decode(inp.q, inp.rho, inp.k_cache, inp.v_cache,
                                               inp.seqlens, o)
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        cold = kv < 2 * l2
        reps = 20 if cold else max(5, min(50, int(2e10 / max(total, 1))))
        times = []
        for _ in range(reps):
            if cold:
                flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            torch.cuda.synchronize() if cold else None
            times.append((a, b))
        torch.cuda.synchronize()
        if px.parallax_check_device_error() != 0:
            raise RuntimeError(f"device error in decode case {kind} B={B} L={L}")
        ms = statistics.median(a.elapsed_time(b) for a, b in times)
        gbs = total / (ms * 1e-3) / 1e9
        chunk = px.parallax_attn_decode_chunk_keys(B, H, int(inp.k_cache.shape[2]), d, 2)
        row = {"case": kind, "B": B, "context": L if kind == "sweep" else f"U[128,{L}]",
               "keys": keys, "kv_bytes": kv, "ms": ms, "GB/s": gbs,
               "frac_of_hbm_peak": gbs / peaks["hbm_gbs"], "tokens_per_s": B / (ms * 1e-3),
               "chunk_keys": chunk, "l2": "evicted before each call" if cold else "larger than L2",
               "boundary_cell_64GiB": boundary}
        rows.append(row)
        if not quiet:
            print(json.dumps(row), flush=True)
        del inp, o
        torch.cuda.empty_cache()
    del flush
    torch.cuda.empty_cache()
    return rows


def run_sweep(args):
    """--sweep: every decode sweep cell (plus the 64 GiB boundary cell) and the ragged batch,
    one JSON line per case, and a markdown table on stderr."""
    import torch

    import softmax_covariance_correction_pass_b300 as px

    dev = torch.device("cuda", torch.cuda.current_device())
    px.load_library()
    rows = sweep_rows(dev, load_peaks())
    print("| case | B | context | KV bytes | ms | GB/s | % of HBM peak | tokens/s | chunk |",
          file=sys.stderr)
    print("|---|---|---|---|---|---|---|---|---|", file=sys.stderr)
    for r in rows:
        tag = " (64 GiB, flagged)" if r["boundary_cell_64GiB"] else ""
        print(f"| {r['case']}{tag} | {r['B']} | {r['context']} | {r['kv_bytes'] / 1e9:.3f} GB | "
              f"{r['ms']:.4f} | {r['GB/s']:.0f} | {100 * r['frac_of_hbm_peak']:.1f}% | "
              f"{r['tokens_per_s']:.0f} | {r['chunk_keys']} |", file=sys.stderr)
    return 0


# ----------------------------------------------------------------------------- serving variants
def run_serving_one(args):
    """--only gqa / --only lla (profiling runs): the grouped-query decode at B=64, H=16 over
    H_kv=2, 8192 keys, or the exact LLA decode at the uniform decode shape; `--steps` timed
    calls after `--warmup` warm-ups, one JSON line."""
    import torch

    import softmax_covariance_correction_pass_b300 as px
    from softmax_covariance_correction_pass_b300 import configs

    dev = torch.device("cuda", torch.cuda.current_device())
    px.load_library()
    B = args.decode_batch or 64
    if args.only == "gqa":
        inp = configs.decode_gqa_inputs(B, 16, 2, 128, 8192, 8192, seed=1, device=dev)
        call = lambda: px.parallax_attn_decode_gqa(inp.q, inp.rho, inp.k_cache, inp.v_cache,
                                                   inp.seqlens)
    else:
        inp = configs.decode_uniform_inputs(dev, B=B)
        call = lambda: px.parallax_lla_decode(inp.q, inp.k_cache, inp.v_cache, inp.seqlens)
    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        call()
    b.record(stream)
    torch.cuda.synchronize()
    if px.parallax_check_device_error() != 0:
        raise RuntimeError("device error")
    print(json.dumps({"case": args.only, "B": B, "ms": a.elapsed_time(b) / args.steps}),
          flush=True)
    return 0


def time_chunk(args, dev, peaks, timed, reps):
    """Chunked prefill of the layer-shaped workload: 3072 tokens cached, the last 1024 of each
    sequence appended (append_kernel) and attended (prefill_pair_kernel with offsets)."""
    import torch

    import softmax_covariance_correction_pass_b300 as px
    from softmax_covariance_correction_pass_b300 import configs

    full = configs.layer_prefill_inputs(dev, B=args.prefill_batch)
    B, H, L, d = full.q.shape
    off, Lq = 3072, 1024
    kc, vc = full.k.clone(), full.v.clone()
    cl = torch.full((B,), off, dtype=torch.int32, device=dev)
    sl_ = slice(off, L)
    qn, rn, kn, vn = (t[:, :, sl_].contiguous() for t in (full.q, full.rho, full.k, full.v))
    o = torch.empty((B, H, Lq, d), dtype=torch.float32, device=dev)
    ms = timed(lambda: px.parallax_attn_prefill_chunk(qn, rn, kn, vn, kc, vc, cl, o), reps)
    pairs = B * H * sum(off + i + 1 for i in range(Lq))
    flops = 8.0 * d * pairs
    return {"case": f"chunked prefill B={B} H={H} cached={off} chunk={Lq}", "ms": ms,
            "TFLOP/s": flops / ms / 1e9, "frac_of_tensor_peak_burst":
                flops / ms / 1e9 / peaks["bf16_tflops"], "tokens_per_s": B * Lq / (ms * 1e-3)}


def run_serving(args):
    """Grouped-query decode (B=64, H=16 over H_kv in {8, 4, 2}, 8192 keys), paged decode of
    the ragged batch (B=512, U[128,16384] keys, 256-key pages, H_kv in {16, 4}) and the
    layer-shaped chunked prefill (3072 cached + 1024 new tokens).  Each case: 3 warm-ups,
    then `reps` calls timed with CUDA events (inputs larger than L2, back to back)."""
    import torch

    import softmax_covariance_correction_pass_b300 as px
    from softmax_covariance_correction_pass_b300 import configs

    dev = torch.device("cuda", torch.cuda.current_device())
    px.load_library()
    peaks = load_peaks()
    stream = torch.cuda.current_stream()

    def timed(call, reps):
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            call()
        b.record(stream)
        torch.cuda.synchronize()
        if px.parallax_check_device_error() != 0:
            raise RuntimeError("device error")
        return a.elapsed_time(b) / reps

    rows = []
    d = 128
    for Hkv in (8, 4, 2):
        B, H, n = 64, 16, 8192
        inp = configs.decode_gqa_inputs(B, H, Hkv, d, n, n, seed=1, device=dev)
        o = torch.empty((B, H, d), dtype=torch.float32, device=dev)
        ms = timed(lambda: px.parallax_attn_decode_gqa(inp.q, inp.rho, inp.k_cache, inp.v_cache,
                                                        inp.seqlens, o), 20)
        byts = 2 * B * Hkv * n * d * 2 + 2 * B * H * d * 2 + B * H * d * 4
        rows.append({"case": f"gqa decode B={B} H={H} H_kv={Hkv} ctx={n}", "ms": ms,
                     "GB/s": byts / ms / 1e6, "frac_of_hbm_peak": byts / ms / 1e6 / peaks["hbm_gbs"],
                     "kv_bytes": 2 * B * Hkv * n * d * 2, "tokens_per_s": B / (ms * 1e-3)})
        del inp, o
    c = configs.DECODE_RAGGED
    sl = configs.ragged_seqlens()
    for Hkv in (16, 4):
        B, H, P = c["B"], c["H"], 256
        inp, bt = configs.paged_decode_inputs(B, H, Hkv, d, sl, P, seed=c["seed"], device=dev)
        o = torch.empty((B, H, d), dtype=torch.float32, device=dev)
        ms = timed(lambda: px.parallax_attn_decode_paged(inp.q, inp.rho, inp.k_cache, inp.v_cache,
                                                          bt, inp.seqlens, o), 10)
        keys = int(sl.sum())
        byts = 2 * keys * Hkv * d * 2 + 2 * B * H * d * 2 + B * H * d * 4
        rows.append({"case": f"paged decode ragged B={B} H={H} H_kv={Hkv} page={P}", "ms": ms,
                     "GB/s": byts / ms / 1e6, "frac_of_hbm_peak": byts / ms / 1e6 / peaks["hbm_gbs"],
                     "kv_bytes": 2 * keys * Hkv * d * 2, "tokens_per_s": B / (ms * 1e-3)})
        del inp, o, bt
        torch.cuda.empty_cache()
    rows.append(time_chunk(args, dev, peaks, timed, 20))
    torch.cuda.empty_cache()
    # exact local linear attention decode (comparison workload) at the uniform decode shape
    dc = configs.DECODE_UNIFORM
    inp = configs.decode_uniform_inputs(dev)
    B, H, n = dc["B"], dc["H"], dc["ctx"]
    ms = timed(lambda: px.parallax_lla_decode(inp.q, inp.k_cache, inp.v_cache, inp.seqlens), 5)
    gram = 2.0 * d * d * n * B * H        # p-weighted second moment of the keys
    kv_bytes = 2.0 * B * H * n * d * 2    # K and V, read once
    rows.append({"case": f"exact LLA decode B={B} H={H} ctx={n} (one pass: second moments, CG probe, output)",
                 "ms": ms, "bound": "hbm", "GB/s": kv_bytes / ms / 1e6,
                 "frac_of_hbm_peak": kv_bytes / ms / 1e6 / peaks["hbm_gbs"],
                 "gram_TFLOP/s": gram / ms / 1e9,
                 "tokens_per_s": B / (ms * 1e-3),
                 "vs_parallax_decode": "see the decode line of the step"})
    for r in rows:
        print(json.dumps(r), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    if args.serving:
        return run_serving(args)
    if args.only == "projection":
        return run_projection_only(args)
    if args.only in ("gqa", "lla"):
        return run_serving_one(args)
    if args.only == "chunk":
        import torch

        import softmax_covariance_correction_pass_b300 as px

        px.load_library()
        dev = torch.device("cuda", torch.cuda.current_device())
        stream = torch.cuda.current_stream()

        def timed(call, reps):
            for _ in range(max(args.warmup, 3)):
                call()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                call()
            b.record(stream)
            torch.cuda.synchronize()
            if px.parallax_check_device_error() != 0:
                raise RuntimeError("device error")
            return a.elapsed_time(b) / reps

        print(json.dumps(time_chunk(args, dev, load_peaks(), timed, args.steps)), flush=True)
        return 0
    if args.only == "backward":
        import torch

        r = time_backward(args, torch.device("cuda", torch.cuda.current_device()), load_peaks(),
                          lambda x: x, n_rep=args.steps)
        print(json.dumps({"metric": "prefill backward TFLOP/s", "value": r["achieved"],
                          "unit": "TFLOP/s", "steps": args.steps, "warmup": args.warmup,
                          "roofline": r}), flush=True)
        return 0
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
