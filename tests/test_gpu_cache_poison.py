"""Decode-side kernels must not read the KV cache past each sequence's length into a
result.  Rows at and after seqlens[b] (and pool pages no block table references) are
set to NaN before the call; the outputs must still match the fp64 oracle, which only
sees the rows below seqlens[b].  A kernel that multiplies a zero weight into such a
row (0 * NaN = NaN) or lets one into a max fails here.

Covered: split-KV decode (bf16 and fp32, automatic plan and forced 256-key chunks),
grouped-query decode on the warp-level MMA kernel, paged decode (SIMT and MMA
kernels), exact LLA decode.  Tolerances as in the parity tests of each path.
"""
import pytest
import torch

import oracle
import softmax_covariance_correction_pass_b300 as px
from softmax_covariance_correction_pass_b300 import configs
from parity_util import assert_bf16, errors

pytestmark = pytest.mark.gpu
DEV = "cuda"


def poison_tail(cache, seqlens):
    """NaN into rows n.. of every (b, h) of a [B, H, Lmax, d] cache."""
    for b, n in enumerate(seqlens.tolist()):
        cache[b, :, n:] = float("nan")


@pytest.fixture(params=[0, 256], ids=["auto-chunk", "chunk256"])
def chunk(request):
    px.parallax_attn_set_decode_chunk_keys(request.param)
    yield request.param
    px.parallax_attn_set_decode_chunk_keys(0)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
def test_decode_ignores_rows_past_seqlen(dtype, chunk):
    sl = [1000, 517, 3, 0]
    inp = configs.decode_inputs(4, 4, 128, sl, 1000, seed=71, device=DEV, dtype=dtype)
    ref = oracle.decode(inp.q, inp.rho, inp.k_cache, inp.v_cache, inp.seqlens)
    poison_tail(inp.k_cache, inp.seqlens)
    poison_tail(inp.v_cache, inp.seqlens)
    # (the binding calls parallax_attn_decode or parallax_attn_decode_f32 by dtype)
    o = px.parallax_attn_decode(inp.q, inp.rho, inp.k_cache, inp.v_cache, inp.seqlens)
    torch.cuda.synchronize()
    assert px.parallax_check_device_error() == 0
    assert torch.isfinite(o).all()
    if dtype == torch.bfloat16:
        assert_bf16(o, ref, "decode, poisoned tail")
    else:
        rel, _ = errors(o, ref)
        assert rel <= 1e-5, f"fp32 decode, poisoned tail: rel-L2 {rel:.3e}"


@pytest.mark.parametrize("H,Hkv", [(8, 2), (16, 2), (8, 4)])
def test_gqa_ignores_rows_past_seqlen(H, Hkv, chunk):
    sl = [2048, 1300, 77]
    inp = configs.decode_gqa_inputs(3, H, Hkv, 128, sl, 2048, seed=72 + H, device=DEV)
    ref = oracle.decode_gqa(inp.q, inp.rho, inp.k_cache, inp.v_cache, inp.seqlens)
    poison_tail(inp.k_cache, inp.seqlens)
    poison_tail(inp.v_cache, inp.seqlens)
    o = px.parallax_attn_decode_gqa(inp.q, inp.rho, inp.k_cache, inp.v_cache, inp.seqlens)
    torch.cuda.synchronize()
    assert px.parallax_check_device_error() == 0
    assert torch.isfinite(o).all()
    assert_bf16(o, ref, f"gqa H={H} Hkv={Hkv}, poisoned tail")


@pytest.mark.parametrize("P,H,Hkv", [(256, 8, 2), (64, 4, 4)])
def test_paged_ignores_unused_rows_and_pages(P, H, Hkv):
    sl = [1000, 300, 5]
    inp, bt = configs.paged_decode_inputs(3, H, Hkv, 128, sl, P, seed=73 + P, device=DEV)
    ref = oracle.decode_paged(inp.q, inp.rho, inp.k_cache, inp.v_cache, bt, inp.seqlens, P)
    used = set()
    for b, n in enumerate(sl):
        npg = (n + P - 1) // P
        pages = bt[b, :npg].tolist()
        used.update(pages)
        if n % P:
            inp.k_cache[pages[-1], :, n % P:] = float("nan")
            inp.v_cache[pages[-1], :, n % P:] = float("nan")
    for pg in range(inp.k_cache.shape[0]):
        if pg not in used:
            inp.k_cache[pg] = float("nan")
            inp.v_cache[pg] = float("nan")
    o = px.parallax_attn_decode_paged(inp.q, inp.rho, inp.k_cache, inp.v_cache, bt, inp.seqlens)
    torch.cuda.synchronize()
    assert px.parallax_check_device_error() == 0
    assert torch.isfinite(o).all()
    assert_bf16(o, ref, f"paged P={P} H={H} Hkv={Hkv}, poisoned rows and pages")


@pytest.mark.parametrize("d", [64, 128])
def test_lla_ignores_rows_past_seqlen(d):
    sl = [1000, 517, 0]
    inp = configs.decode_inputs(3, 4, d, sl, 1000, seed=74 + d, device=DEV)
    ro, rr = oracle.lla_decode(inp.q, inp.k_cache, inp.v_cache, inp.seqlens)
    poison_tail(inp.k_cache, inp.seqlens)
    poison_tail(inp.v_cache, inp.seqlens)
    o, rho = px.parallax_lla_decode(inp.q, inp.k_cache, inp.v_cache, inp.seqlens)
    torch.cuda.synchronize()
    assert px.parallax_check_device_error() == 0
    assert torch.isfinite(o).all() and torch.isfinite(rho).all()
    rel, _ = errors(rho, rr)
    assert rel <= 1e-3, f"LLA probe, poisoned tail: rel-L2 {rel:.3e}"
    assert_bf16(o, ro, f"LLA d={d}, poisoned tail")
    assert torch.all(o[2] == 0) and torch.all(rho[2] == 0)
