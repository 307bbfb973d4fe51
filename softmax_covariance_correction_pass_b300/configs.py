"""Seeded synthetic inputs for the Parallax workloads.

This module only draws random tensors (and, for the layer-shaped prefill
workload, multiplies them by random projection matrices the way a layer would
produce q, k, v and the probe rho = W_R x).  It contains none of the attention
arithmetic and is the one module that the CUDA path and the oracle both use:
the same tensors are handed to both.

Draw order is fixed: q, k, v, then rho (then scaled), from one torch
generator seeded per workload and living on the target device (Philox on CUDA,
MT19937 on the CPU).  Values are drawn in fp32 and then cast.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

# ----------------------------------------------------------------------------- workloads
CAUSAL_F32 = dict(name="causal prefill fp32 [1,2,128,64]", B=1, H=2, L=128, d=64, seed=0,
                  rho_scale=0.1)
DECODE_UNIFORM = dict(name="bf16 decode B=64 H=16 d=128 ctx=8192", B=64, H=16, d=128, ctx=8192,
                      seed=1, rho_std=0.1)
DECODE_SWEEP = dict(name="bf16 decode sweep H=16 d=128", H=16, d=128, seed=2, rho_std=0.1,
                    batches=(1, 8, 64, 256, 2048), contexts=(128, 1024, 8192, 32768),
                    max_kv_bytes=64e9)
DECODE_RAGGED = dict(name="bf16 ragged decode B=512 H=16 d=128 ctx~U[128,16384]", B=512, H=16,
                     d=128, lo=128, hi=16384, seed=3, rho_std=0.1)
LAYER_PREFILL = dict(name="bf16 causal prefill B=8 H=16 L=4096 d=128 (width 2048)", B=8, H=16,
                     L=4096, d=128, width=2048, seed=4, wr_std=0.02)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(seed)
    return g


def _randn(shape, g, device, dtype):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(dtype)


@dataclass
class PrefillInputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    rho: torch.Tensor | None
    scale: float


@dataclass
class DecodeInputs:
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    rho: torch.Tensor | None
    seqlens: torch.Tensor


def prefill_inputs(B, H, L, d, seed, rho_scale=0.1, device="cpu", dtype=torch.float32,
                   variant="base") -> PrefillInputs:
    """q, k, v, rho ~ N(0, 1) (rho then scaled by rho_scale), in that draw order.

    variant: "base"; "rho0" (rho = 0); "same_k" (every k_j equal to k_0 of its head).
    """
    g = _gen(seed, device)
    q = _randn((B, H, L, d), g, device, dtype)
    k = _randn((B, H, L, d), g, device, dtype)
    v = _randn((B, H, L, d), g, device, dtype)
    rho = (_randn((B, H, L, d), g, device, torch.float32) * rho_scale).to(dtype)
    if variant == "rho0":
        rho = torch.zeros_like(rho)
    elif variant == "same_k":
        k = k[:, :, :1].expand(B, H, L, d).contiguous()
    elif variant != "base":
        raise ValueError(variant)
    return PrefillInputs(q, k, v, rho, 1.0 / math.sqrt(d))


def causal_f32_inputs(device="cpu", variant="base") -> PrefillInputs:
    c = CAUSAL_F32
    return prefill_inputs(c["B"], c["H"], c["L"], c["d"], c["seed"], c["rho_scale"], device,
                          torch.float32, variant)


def decode_inputs(B, H, d, seqlens, Lmax, seed, rho_std=0.1, device="cpu",
                  dtype=torch.bfloat16) -> DecodeInputs:
    """q [B,H,d], caches [B,H,Lmax,d] ~ N(0,1), rho ~ N(0, rho_std^2); draw order q, k, v, rho."""
    g = _gen(seed, device)
    q = _randn((B, H, d), g, device, dtype)
    k = _randn((B, H, Lmax, d), g, device, dtype)
    v = _randn((B, H, Lmax, d), g, device, dtype)
    rho = (_randn((B, H, d), g, device, torch.float32) * rho_std).to(dtype)
    sl = torch.as_tensor(seqlens, dtype=torch.int32)
    if sl.ndim == 0:
        sl = sl.repeat(B)
    return DecodeInputs(q, k, v, rho, sl.to(device))


def decode_gqa_inputs(B, H, Hkv, d, seqlens, Lmax, seed, rho_std=0.1, device="cpu"):
    """q, rho [B, H, d]; caches [B, Hkv, Lmax, d] bf16 (draw order q, k, v, rho)."""
    g = _gen(seed, device)
    bf = torch.bfloat16
    q = _randn((B, H, d), g, device, bf)
    k = _randn((B, Hkv, Lmax, d), g, device, bf)
    v = _randn((B, Hkv, Lmax, d), g, device, bf)
    rho = (_randn((B, H, d), g, device, torch.float32) * rho_std).to(bf)
    sl = torch.as_tensor(seqlens, dtype=torch.int32)
    if sl.ndim == 0:
        sl = sl.repeat(B)
    return DecodeInputs(q, k, v, rho, sl.to(device))


def page_cache(k_cache, v_cache, page_size, seed, spare_pages=3):
    """Cut contiguous caches [B, Hkv, Lmax, d] (Lmax a multiple of page_size) into a shuffled
    page pool [num_pages, Hkv, page_size, d] plus a block table [B, Lmax // page_size] that
    maps every sequence's pages back; `spare_pages` unused pages are added to the pool.
    Pure data movement (the permutation comes from a CPU generator)."""
    B, Hkv, Lmax, d = k_cache.shape
    assert Lmax % page_size == 0
    mp = Lmax // page_size
    n = B * mp + spare_pages
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(seed))
    bt = perm[:B * mp].view(B, mp).to(torch.int32)

    def pool(c):
        pages = c.view(B, Hkv, mp, page_size, d).permute(0, 2, 1, 3, 4).reshape(B * mp, Hkv,
                                                                                 page_size, d)
        out = torch.zeros((n, Hkv, page_size, d), dtype=c.dtype, device=c.device)
        out[perm[:B * mp].to(c.device)] = pages
        return out

    return pool(k_cache), pool(v_cache), bt.to(k_cache.device)


def paged_decode_inputs(B, H, Hkv, d, seqlens, page_size, seed, rho_std=0.1, device="cpu",
                        spare_pages=3):
    """A paged cache drawn directly: q, rho [B, H, d]; a pool of exactly the pages the
    sequences need (plus `spare_pages`) [num_pages, Hkv, page_size, d] ~ N(0,1) bf16; a
    block table [B, max_pages] giving each sequence distinct pages in shuffled order
    (entries past a sequence's last page are -1).  Draw order q, k pool, v pool, rho; the
    shuffle comes from a CPU generator seeded with `seed`.
    Returns (DecodeInputs with k_cache / v_cache holding the pools, block_table)."""
    sl = torch.as_tensor(seqlens, dtype=torch.int32)
    if sl.ndim == 0:
        sl = sl.repeat(B)
    npg = [(int(n) + page_size - 1) // page_size for n in sl]
    max_pages = max(1, max(npg))
    num_pages = sum(npg) + spare_pages
    g = _gen(seed, device)
    bf = torch.bfloat16
    q = _randn((B, H, d), g, device, bf)
    k = _randn((num_pages, Hkv, page_size, d), g, device, bf)
    v = _randn((num_pages, Hkv, page_size, d), g, device, bf)
    rho = (_randn((B, H, d), g, device, torch.float32) * rho_std).to(bf)
    perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(seed))
    bt = torch.full((B, max_pages), -1, dtype=torch.int32)
    pos = 0
    for b, n in enumerate(npg):
        bt[b, :n] = perm[pos:pos + n].to(torch.int32)
        pos += n
    return DecodeInputs(q, k, v, rho, sl.to(device)), bt.to(device)


def decode_uniform_inputs(device="cuda", B=None, ctx=None) -> DecodeInputs:
    c = DECODE_UNIFORM
    B = B or c["B"]
    ctx = ctx or c["ctx"]
    return decode_inputs(B, c["H"], c["d"], ctx, ctx, c["seed"], c["rho_std"], device)


def decode_sweep_cells(include_boundary: bool = False):
    """(batch, context) cells whose K+V cache (B*L*H*d*2 bytes*2) does not exceed 64e9 bytes.

    include_boundary also returns the (256, 32768) cell, whose cache is exactly
    64 GiB (68.7e9 bytes): over the limit read in decimal gigabytes.
    """
    c = DECODE_SWEEP
    cells = []
    for B in c["batches"]:
        for L in c["contexts"]:
            kv = B * L * c["H"] * c["d"] * 2 * 2
            if kv <= c["max_kv_bytes"] or (include_boundary and kv == 2 ** 36):
                cells.append((B, L))
    return cells


def decode_sweep_inputs(B, L, device="cuda") -> DecodeInputs:
    c = DECODE_SWEEP
    return decode_inputs(B, c["H"], c["d"], L, L, c["seed"], c["rho_std"], device)


def ragged_seqlens(B=None, lo=None, hi=None, seed=None) -> torch.Tensor:
    """Per-sequence lengths ~ U{lo..hi} (inclusive), drawn on the CPU so every device agrees."""
    c = DECODE_RAGGED
    g = torch.Generator().manual_seed(seed if seed is not None else c["seed"])
    return torch.randint(lo or c["lo"], (hi or c["hi"]) + 1, (B or c["B"],), generator=g,
                         dtype=torch.int64).to(torch.int32)


def decode_ragged_inputs(device="cuda", B=None, hi=None) -> DecodeInputs:
    c = DECODE_RAGGED
    B = B or c["B"]
    hi = hi or c["hi"]
    sl = ragged_seqlens(B, c["lo"], hi)
    return decode_inputs(B, c["H"], c["d"], sl, hi, c["seed"], c["rho_std"], device)


def _layer_draws(device, B, L):
    """x ~ N(0,1) [B, L, width]; W_q, W_k, W_v ~ N(0, 1/width), W_R ~ N(0, wr_std^2), each
    [width, H*d] (bf16).  Draw order: x, W_q, W_k, W_v, W_R."""
    c = LAYER_PREFILL
    H, d, width = c["H"], c["d"], c["width"]
    g = _gen(c["seed"], device)
    bf = torch.bfloat16
    x = _randn((B, L, width), g, device, bf)
    ws = [(_randn((width, H * d), g, device, torch.float32) / math.sqrt(width)).to(bf)
          for _ in range(3)]
    wr = (_randn((width, H * d), g, device, torch.float32) * c["wr_std"]).to(bf)
    return x, ws + [wr]


def layer_prefill_inputs(device="cuda", B=None, L=None) -> PrefillInputs:
    """Layer-shaped bf16 prefill: x ~ N(0,1) [B, L, width]; W_q, W_k, W_v ~ N(0, 1/width);
    W_R ~ N(0, wr_std^2); q, k, v, rho = x W (bf16 matmuls on the device), viewed as
    [B, L, H, d] and made [B, H, L, d].  Draw order: x, W_q, W_k, W_v, W_R."""
    c = LAYER_PREFILL
    B = B or c["B"]
    L = L or c["L"]
    H, d = c["H"], c["d"]
    x, ws = _layer_draws(device, B, L)

    def proj(w):
        return (x @ w).view(B, L, H, d).permute(0, 2, 1, 3).contiguous()

    q, k, v, rho = (proj(w) for w in ws)
    return PrefillInputs(q, k, v, rho, 1.0 / math.sqrt(d))


def layer_projection_inputs(device="cuda", B=None, L=None):
    """The same draws as layer_prefill_inputs, as the projection's inputs: x [B, L, width]
    and the stacked weight [W_q; W_k; W_v; W_R] of shape [4*H*d, width] (rows = output
    features), both bf16."""
    c = LAYER_PREFILL
    x, ws = _layer_draws(device, B or c["B"], L or c["L"])
    return x, torch.cat([w.t() for w in ws], dim=0).contiguous()


def projection_inputs(B, L, width, H, d, n_out, seed, device="cpu"):
    """x ~ N(0,1) [B, L, width] and a stacked weight ~ N(0, 1/width) [n_out*H*d, width],
    bf16, for projection tests at arbitrary shapes (draw order x, w)."""
    g = _gen(seed, device)
    x = _randn((B, L, width), g, device, torch.bfloat16)
    w = (_randn((n_out * H * d, width), g, device, torch.float32) / math.sqrt(width)).to(
        torch.bfloat16)
    return x, w
