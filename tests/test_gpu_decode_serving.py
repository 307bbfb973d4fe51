"""GPU parity of the serving variants of decode against the fp64 oracle:
shared key/value heads (grouped-query attention) and a paged key/value cache.

Tolerance: bf16 inputs with fp32 accumulation, rel-L2 <= 1e-2 and max-abs <=
2e-2 over the whole output (the oracle gets the exact bf16 values the kernel
read).  Every case runs with the automatic split plan and with a forced
256-key chunk, so both the single-pass and the split-KV + combine paths are
covered.
"""
import numpy as np
import pytest
import torch

import oracle
import softmax_covariance_correction_pass_b300 as px
from softmax_covariance_correction_pass_b300 import configs
from parity_util import assert_bf16

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(params=[0, 256], ids=["auto-chunk", "chunk256"])
def chunk(request):
    px.parallax_attn_set_decode_chunk_keys(request.param)
    yield request.param
    px.parallax_attn_set_decode_chunk_keys(0)


@pytest.mark.parametrize("H,Hkv", [(8, 8), (8, 4), (8, 2), (8, 1), (16, 2)])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("with_rho", [True, False])
def test_gqa_matches_oracle(H, Hkv, d, with_rho, chunk):
    sl = [1000, 37, 0, 513]
    inp = configs.decode_gqa_inputs(4, H, Hkv, d, sl, 1000, seed=H * 10 + Hkv + d, device=DEV)
    rho = inp.rho if with_rho else None
    o = px.parallax_attn_decode_gqa(inp.q, rho, inp.k_cache, inp.v_cache, inp.seqlens)
    torch.cuda.synchronize()
    assert px.parallax_check_device_error() == 0
    ref = oracle.decode_gqa(inp.q, rho, inp.k_cache, inp.v_cache, inp.seqlens)
    assert_bf16(o, ref, f"gqa H={H} Hkv={Hkv} d={d} rho={with_rho}")
    assert torch.all(o[2] == 0)  # empty sequence


def test_gqa_one_group_equals_plain_decode():
    """H_kv = H runs the same kernel instance and plan as parallax_attn_decode:
    the outputs are identical bit for bit."""
    inp = configs.decode_gqa_inputs(3, 8, 8, 128, [700, 1, 256], 700, seed=5, device=DEV)
    a = px.parallax_attn_decode_gqa(inp.q, inp.rho, inp.k_cache, inp.v_cache, inp.seqlens)
    b = px.parallax_attn_decode(inp.q, inp.rho, inp.k_cache, inp.v_cache, inp.seqlens)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("P", [16, 64, 256])
@pytest.mark.parametrize("H,Hkv,d", [(8, 2, 128), (4, 4, 64)])
def test_paged_matches_oracle(P, H, Hkv, d, chunk):
    Lmax = 1024
    sl = [1000, 33, 0, 1024]
    inp = configs.decode_gqa_inputs(4, H, Hkv, d, sl, Lmax, seed=P + d, device=DEV)
    kp, vp, bt = configs.page_cache(inp.k_cache, inp.v_cache, P, seed=P)
    # table entries past a sequence's last page are never read: poison them
    for b, n in enumerate(sl):
        bt[b, -(-n // P):] = -1
    o = px.parallax_attn_decode_paged(inp.q, inp.rho, kp, vp, bt, inp.seqlens)
    torch.cuda.synchronize()
    assert px.parallax_check_device_error() == 0
    ref = oracle.decode_paged(inp.q, inp.rho, kp, vp, bt.clamp(min=0), inp.seqlens, P)
    assert_bf16(o, ref, f"paged P={P} H={H} Hkv={Hkv} d={d}")


def test_paged_identity_table_equals_contiguous():
    """Pages laid out in order with block_table[b, i] = b * max_pages + i hold
    the contiguous cache; the same split plan then gives identical bits."""
    B, H, Hkv, d, P, Lmax = 3, 8, 2, 128, 64, 2048
    inp = configs.decode_gqa_inputs(B, H, Hkv, d, [2048, 999, 64], Lmax, seed=8, device=DEV)
    mp = Lmax // P

    def pool(c):
        return c.view(B, Hkv, mp, P, d).permute(0, 2, 1, 3, 4).reshape(B * mp, Hkv, P, d) \
            .contiguous()

    bt = torch.arange(B * mp, dtype=torch.int32, device=DEV).view(B, mp)
    a = px.parallax_attn_decode_paged(inp.q, inp.rho, pool(inp.k_cache), pool(inp.v_cache), bt,
                                      inp.seqlens)
    b = px.parallax_attn_decode_gqa(inp.q, inp.rho, inp.k_cache, inp.v_cache, inp.seqlens)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_paged_out_of_range_page_is_flagged():
    """A table entry outside the pool is read as page 0 and raises the
    out-of-range bit; nothing outside the pool is touched."""
    B, H, Hkv, d, P = 2, 4, 4, 128, 16
    inp = configs.decode_gqa_inputs(B, H, Hkv, d, [64, 40], 64, seed=9, device=DEV)
    kp, vp, bt = configs.page_cache(inp.k_cache, inp.v_cache, P, seed=1)
    bt[1, 1] = kp.shape[0] + 1000
    px.parallax_attn_decode_paged(inp.q, inp.rho, kp, vp, bt, inp.seqlens)
    bits = px.parallax_check_device_error()
    assert bits == px.DEVERR_PAGE_OUT_OF_RANGE


def test_gqa_decode_layer_size():
    """Serving shape: B=64, H=16 query heads over H_kv=2 key/value heads, d=128,
    8192 keys per sequence, against the oracle on every head."""
    inp = configs.decode_gqa_inputs(64, 16, 2, 128, 8192, 8192, seed=11, device=DEV)
    o = px.parallax_attn_decode_gqa(inp.q, inp.rho, inp.k_cache, inp.v_cache, inp.seqlens)
    torch.cuda.synchronize()
    assert px.parallax_check_device_error() == 0
    ref = oracle.decode_gqa(inp.q, inp.rho, inp.k_cache, inp.v_cache, inp.seqlens,
                            form="contracted")
    assert_bf16(o, ref, "gqa B=64 H=16 Hkv=2 ctx=8192")


def test_paged_ragged_layer_size():
    """The ragged-batch workload's lengths (B=512, U[128, 16384]) in a pool of
    256-key pages with H=16 query heads over H_kv=4, d=128; 8 sampled sequences
    (the longest among them) checked against the oracle."""
    c = configs.DECODE_RAGGED
    B, H, Hkv, d, P = c["B"], c["H"], 4, c["d"], 256
    sl = configs.ragged_seqlens()
    inp, bt = configs.paged_decode_inputs(B, H, Hkv, d, sl, P, seed=c["seed"], device=DEV)
    o = px.parallax_attn_decode_paged(inp.q, inp.rho, inp.k_cache, inp.v_cache, bt, inp.seqlens)
    torch.cuda.synchronize()
    assert px.parallax_check_device_error() == 0
    rows = np.random.default_rng(0).choice(B, 8, replace=False)
    rows[0] = int(torch.argmax(sl))
    idx = torch.as_tensor(rows, device=DEV)
    # only the pages the sampled sequences use go to the host
    sub_bt = bt.index_select(0, idx)
    used = torch.unique(sub_bt[sub_bt >= 0])
    remap = torch.full((inp.k_cache.shape[0] + 1,), -1, dtype=torch.int64, device=DEV)
    remap[used.long()] = torch.arange(used.numel(), device=DEV)
    sub_bt = torch.where(sub_bt >= 0, remap[sub_bt.long().clamp(min=0)], 0).int()
    ref = oracle.decode_paged(inp.q.index_select(0, idx), inp.rho.index_select(0, idx),
                              inp.k_cache.index_select(0, used), inp.v_cache.index_select(0, used),
                              sub_bt, inp.seqlens.index_select(0, idx), P, form="contracted")
    assert_bf16(o.index_select(0, idx), ref, "paged ragged B=512 sample")
