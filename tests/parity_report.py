"""Parity report: rel-L2 and max-abs of the CUDA path against the fp64 oracle on
every workload (GPU needed).  Not collected by pytest; run it directly:

    python tests/parity_report.py > parity.md

Prints a markdown table, one line per workload / variant.  Full-size workloads
are compared on sampled heads or rows (named in the line); the small ones in
full.
"""
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import oracle  # noqa: E402
import softmax_covariance_correction_pass_b300 as px  # noqa: E402
from softmax_covariance_correction_pass_b300 import configs  # noqa: E402
from parity_util import errors  # noqa: E402

DEV = "cuda"
ROWS = []


def row(workload, what, got, ref):
    rel, mx = errors(got, ref)
    scale = float(np.abs(np.asarray(ref)).max())
    ROWS.append((workload, what, rel, mx, scale))


def main():
    px.load_library()
    # 1. causal prefill fp32 [1,2,128,64] and its two variants
    for variant in ("base", "rho0", "same_k"):
        inp = configs.causal_f32_inputs(DEV, variant)
        o = px.parallax_attn_prefill(inp.q, inp.rho, inp.k, inp.v, causal=True, scale=inp.scale)
        ref = oracle.prefill(inp.q, inp.rho, inp.k, inp.v, causal=True, scale=inp.scale)
        row("causal prefill fp32 [1,2,128,64]", variant, o, ref)
    # 2. uniform decode B=64 H=16 d=128 ctx=8192, every head
    inp = configs.decode_uniform_inputs(DEV)
    o = px.parallax_attn_decode(inp.q, inp.rho, inp.k_cache, inp.v_cache, inp.seqlens)
    row("bf16 decode B=64 H=16 d=128 ctx=8192", "all 1024 heads",
        o, oracle.decode(inp.q, inp.rho, inp.k_cache, inp.v_cache, inp.seqlens, form="contracted"))
    del inp
    # 3. decode sweep: 2 sampled sequences of every cell
    rng = np.random.default_rng(0)
    for B, L in configs.decode_sweep_cells():
        inp = configs.decode_sweep_inputs(B, L, DEV)
        o = px.parallax_attn_decode(inp.q, inp.rho, inp.k_cache, inp.v_cache, inp.seqlens)
        bs = sorted(set(int(b) for b in rng.choice(B, min(2, B), replace=False)))
        idx = torch.as_tensor(bs, device=DEV)
        ref = oracle.decode(inp.q.index_select(0, idx), inp.rho.index_select(0, idx),
                            inp.k_cache.index_select(0, idx), inp.v_cache.index_select(0, idx),
                            inp.seqlens.index_select(0, idx), form="contracted")
        row("bf16 decode sweep", f"B={B} ctx={L}, sequences {bs}", o.index_select(0, idx), ref)
        del inp, o
        torch.cuda.empty_cache()
    # 4. ragged decode B=512: 16 sampled sequences
    inp = configs.decode_ragged_inputs(DEV)
    o = px.parallax_attn_decode(inp.q, inp.rho, inp.k_cache, inp.v_cache, inp.seqlens)
    idx = torch.as_tensor(sorted(rng.choice(512, 16, replace=False)), device=DEV)
    ref = oracle.decode(inp.q.index_select(0, idx), inp.rho.index_select(0, idx),
                        inp.k_cache.index_select(0, idx), inp.v_cache.index_select(0, idx),
                        inp.seqlens.index_select(0, idx), form="contracted")
    row("bf16 ragged decode B=512", "16 sampled sequences", o.index_select(0, idx), ref)
    del inp, o
    torch.cuda.empty_cache()
    # 5. layer-shaped causal prefill: 4 heads in full
    inp = configs.layer_prefill_inputs(DEV)
    o = px.parallax_attn_prefill(inp.q, inp.rho, inp.k, inp.v, causal=True, scale=inp.scale)
    for b, h in ((0, 0), (2, 5), (5, 10), (7, 15)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = oracle.prefill(inp.q[sl], inp.rho[sl], inp.k[sl], inp.v[sl], causal=True,
                             scale=inp.scale, form="contracted")
        row("bf16 causal prefill B=8 H=16 L=4096 d=128", f"head b={b} h={h}", o[sl], ref)
    # projection of the same layer: 64 sampled tokens
    x, w = configs.layer_projection_inputs(DEV)
    outs = px.parallax_attn_qkvr_projection(x, w, 16, 128)
    ls = torch.as_tensor(sorted(rng.choice(4096, 64, replace=False)), device=DEV)
    refs = oracle.qkvr_projection(x.index_select(1, ls), w, 16, 128)
    for name, g, r in zip(("q", "k", "v", "rho"), outs, refs):
        row("q/k/v/probe projection [8,4096,2048] -> [8,16,4096,128]", f"{name}, 64 tokens",
            g.index_select(2, ls), r)
    del outs, x, w
    # backward of the layer: 2 heads
    g = torch.Generator(device=DEV).manual_seed(44)
    dout = torch.randn(inp.q.shape, generator=g, device=DEV).to(torch.bfloat16)
    o2, lse, rbar, mu = px.parallax_attn_prefill_train(inp.q, inp.rho, inp.k, inp.v, causal=True,
                                                       scale=inp.scale)
    grads = px.parallax_attn_prefill_backward(inp.q, inp.rho, inp.k, inp.v, o2, mu, lse, rbar,
                                              dout, causal=True, scale=inp.scale)
    for b, h in ((0, 0), (6, 13)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        refs = oracle.prefill_backward(inp.q[sl], inp.rho[sl], inp.k[sl], inp.v[sl], dout[sl],
                                       causal=True, scale=inp.scale)
        for name, gg, r in zip(("dq", "drho", "dk", "dv"), grads, refs):
            row("prefill backward B=8 H=16 L=4096 d=128", f"{name}, head b={b} h={h}", gg[sl], r)
    # chunked prefill: 3072 cached + 1024 new, 2 heads against the oracle
    kc, vc = inp.k.clone(), inp.v.clone()
    cl = torch.full((8,), 3072, dtype=torch.int32, device=DEV)
    s = slice(3072, 4096)
    oc = px.parallax_attn_prefill_chunk(*(t[:, :, s].contiguous() for t in
                                          (inp.q, inp.rho, inp.k, inp.v)), kc, vc, cl)
    for b, h in ((1, 3), (6, 14)):
        rows = np.arange(1024)
        ref = oracle.rows(inp.q[b, h, 3072:], inp.rho[b, h, 3072:], inp.k[b, h], inp.v[b, h],
                          3072 + rows + 1, inp.scale, form="contracted")
        row("chunked prefill B=8 H=16 (3072 cached + 1024)", f"head b={b} h={h}", oc[b, h], ref)
    del inp, kc, vc, o, o2, mu, grads
    torch.cuda.empty_cache()
    # serving decode variants
    gi = configs.decode_gqa_inputs(64, 16, 2, 128, 8192, 8192, seed=11, device=DEV)
    og = px.parallax_attn_decode_gqa(gi.q, gi.rho, gi.k_cache, gi.v_cache, gi.seqlens)
    row("GQA decode B=64 H=16 H_kv=2 ctx=8192", "all heads", og,
        oracle.decode_gqa(gi.q, gi.rho, gi.k_cache, gi.v_cache, gi.seqlens, form="contracted"))
    # exact LLA decode: 8 sampled heads of the uniform decode workload
    inp = configs.decode_uniform_inputs(DEV)
    ol, rl = px.parallax_lla_decode(inp.q, inp.k_cache, inp.v_cache, inp.seqlens)
    for b, h in ((0, 0), (13, 7), (40, 2), (63, 15)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        ro, rr = oracle.lla_decode(inp.q[sl], inp.k_cache[sl], inp.v_cache[sl],
                                   inp.seqlens[b:b + 1])
        row("exact LLA decode B=64 H=16 ctx=8192", f"o, head b={b} h={h}", ol[sl], ro)
        row("exact LLA decode B=64 H=16 ctx=8192", f"rho, head b={b} h={h}", rl[sl], rr)
    assert px.parallax_check_device_error() == 0

    print("| workload | compared | rel-L2 | max-abs | max abs of the reference |")
    print("|---|---|---|---|---|")
    for w, what, rel, mx, sc in ROWS:
        print(f"| {w} | {what} | {rel:.2e} | {mx:.2e} | {sc:.3g} |")


if __name__ == "__main__":
    main()
