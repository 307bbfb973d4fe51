"""The no-allocation decode entry point against the regular one.

parallax_attn_decode_noalloc serves callers that cannot let the library call
cudaMalloc (engines that pre-reserve device memory for their own KV-cache pool,
and decode loops that cannot afford an allocation's device synchronisation).
It keeps the split-KV partial states in a fixed array inside the library, so
these tests check, through the C ABI, that two calls in a row give the same
output as parallax_attn_decode, and that a shape needing more scratch than the
array holds is refused before anything is launched.  This file is collected
last on purpose.
"""
import pytest
import torch

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
