"""The no-allocation decode entry point against the regular one.

parallax_attn_decode_noalloc serves callers that cannot let the library call
cudaMalloc (engines that pre-reserve device memory for their own KV-cache pool,
and decode loops that cannot afford an allocation's device synchronisation).
It keeps the split-KV partial states in a fixed array inside the library, so
these tests check, through the C ABI, that two calls in a row give the same
output as parallax_attn_decode (and as the oracle), that a call leaves the
device's free memory unchanged, and that a shape needing more scratch than the
array holds is refused before anything is launched.  This file is collected
last on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
import softmax_covariance_correction_pass_b300 as px
from softmax_covariance_correction_pass_b300 import configs
from parity_util import assert_bf16, errors

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _both(inp, rho=True):
    B, H, d = inp.q.shape
    r = inp.rho if rho else None
    ref = torch.full((B, H, d), float("nan"), dtype=torch.float32, device=DEV)
    px.parallax_attn_decode(inp.q, r, inp.k_cache, inp.v_cache, inp.seqlens, ref)
    got = torch.full((B, H, d), float("nan"), dtype=torch.float32, device=DEV)
    px.parallax_attn_decode_noalloc(inp.q, r, inp.k_cache, inp.v_cache, inp.seqlens, got)
    assert px.parallax_check_device_error() == 0
    return got, ref


def test_two_calls_in_a_row_match_regular_decode():
    px.parallax_attn_set_decode_chunk_keys(0)
    try:
        # call 1: 64 heads x 8192 keys -> the automatic plan splits each head into chunks
        a = configs.decode_inputs(4, 16, 128, 8192, 8192, seed=41, device=DEV)
        assert px.parallax_attn_decode_chunk_keys(4, 16, 8192, 128, 2) < 8192
        got, ref = _both(a)
        assert_bf16(got, ref, "no-alloc call 1")
        assert errors(got, ref)[1] <= 1e-6
        # and directly against the oracle on a few heads
        heads = [(0, 0), (1, 7), (3, 15)]
        want = np.stack([oracle.rows(a.q[b, h][None], a.rho[b, h][None], a.k_cache[b, h],
                                     a.v_cache[b, h], [8192], 1.0 / np.sqrt(128), "contracted")[0]
                         for b, h in heads])
        assert_bf16(np.stack([got[b, h].double().cpu().numpy() for b, h in heads]), want,
                    "no-alloc call 1 against the oracle")
        # call 2: other inputs, ragged lengths (one empty), forced small chunks,
        # so it reuses the scratch the first call left behind
        px.parallax_attn_set_decode_chunk_keys(512)
        b = configs.decode_inputs(3, 8, 128, [3000, 0, 1777], 3000, seed=42, device=DEV)
        got2, ref2 = _both(b)
        assert_bf16(got2, ref2, "no-alloc call 2")
        assert errors(got2, ref2)[1] <= 1e-6
        assert (got2[1] == 0).all()
        got3, ref3 = _both(b, rho=False)
        assert errors(got3, ref3)[1] <= 1e-6
    finally:
        px.parallax_attn_set_decode_chunk_keys(0)


def test_oversized_split_is_refused():
    # 1024 heads x 8 chunks of 256 keys needs about 8.5 MB of scratch: more than the
    # fixed array holds, so the call must fail before launching anything
    px.parallax_attn_set_decode_chunk_keys(256)
    try:
        inp = configs.decode_inputs(64, 16, 128, 2048, 2048, seed=43, device=DEV)
        o = torch.zeros((64, 16, 128), dtype=torch.float32, device=DEV)
        with pytest.raises(px.ParallaxError) as err:
            px.parallax_attn_decode_noalloc(inp.q, inp.rho, inp.k_cache, inp.v_cache,
                                            inp.seqlens, o)
        assert err.value.code == px.PARALLAX_ERR_UNSUPPORTED
        assert "scratch" in str(err.value)
        torch.cuda.synchronize()
        assert (o == 0).all()
        assert px.parallax_check_device_error() == 0
    finally:
        px.parallax_attn_set_decode_chunk_keys(0)


def test_allocates_nothing():
    """The defining property: with the regular workspace released, a no-allocation call
    that splits its heads leaves the device's free memory and the regular workspace as they
    were.  A first call of the same shape comes before the measurement: it looks up the
    array's address and lets CUDA load the decode kernels, which may take device memory
    for their code under lazy module loading."""
    px.parallax_attn_set_decode_chunk_keys(0)
    torch.cuda.synchronize()
    px.parallax_attn_release_workspace()
    assert px.parallax_attn_workspace_bytes() == 0
    a = configs.decode_inputs(4, 16, 128, 8192, 8192, seed=44, device=DEV)
    b = configs.decode_inputs(4, 16, 128, 8192, 8192, seed=45, device=DEV)
    assert px.parallax_attn_decode_chunk_keys(4, 16, 8192, 128, 2) < 8192  # a split plan
    o1 = torch.empty((4, 16, 128), dtype=torch.float32, device=DEV)
    o2 = torch.empty_like(o1)
    px.parallax_attn_decode_noalloc(a.q, a.rho, a.k_cache, a.v_cache, a.seqlens, o1)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    px.parallax_attn_decode_noalloc(b.q, b.rho, b.k_cache, b.v_cache, b.seqlens, o2)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert px.parallax_check_device_error() == 0
    assert free1 == free0
    assert px.parallax_attn_workspace_bytes() == 0
    # the regular entry point (which grows its own workspace) agrees
    ref = torch.empty_like(o2)
    px.parallax_attn_decode(b.q, b.rho, b.k_cache, b.v_cache, b.seqlens, ref)
    assert px.parallax_check_device_error() == 0
    assert errors(o2, ref)[1] <= 1e-6

