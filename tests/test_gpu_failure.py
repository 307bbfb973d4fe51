"""Failure path of the bounded pipeline waits, on the GPU, without a fault or a hang.

Every wait in the library's kernels gives up after a time limit.  The self-test hook
launches one thread that waits, with a 2 ms limit, on an mbarrier that nothing ever
arrives on; the wait must give up, raise DEVERR_WAIT_TIMEOUT in its kernel family's
error word, and later launches of that family must see the bit and return without
work (their outputs stay untouched) until parallax_check_device_error() reads and
clears it.  After that the same call works again.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import softmax_covariance_correction_pass_b300 as px
from softmax_covariance_correction_pass_b300 import configs
from parity_util import assert_bf16

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_decode_wait_gives_up_and_later_launches_stand_down():
    assert px.parallax_check_device_error() == 0
    # 200 keys: one chunk per head, so the decode kernel alone writes o (no combine)
    inp = configs.decode_inputs(2, 4, 128, [200, 77], 200, seed=71, device=DEV)
    assert px.parallax_attn_decode_chunk_keys(2, 4, 200, 128, 2) >= 200
    o = torch.full((2, 4, 128), float("nan"), dtype=torch.float32, device=DEV)
    t0 = time.perf_counter()
    px.parallax_selftest_wait_timeout(px.SELFTEST_DECODE, 2000)
    px.parallax_attn_decode(inp.q, inp.rho, inp.k_cache, inp.v_cache, inp.seqlens, o)
    bits = px.parallax_check_device_error()
    elapsed = time.perf_counter() - t0
    assert bits == px.DEVERR_WAIT_TIMEOUT
    assert elapsed < 0.5, elapsed          # the wait ended near its 2 ms limit
    assert torch.isnan(o).all()            # the decode launch saw the bit and did nothing
    # the word is clear again: the same call now computes the result
    px.parallax_attn_decode(inp.q, inp.rho, inp.k_cache, inp.v_cache, inp.seqlens, o)
    assert px.parallax_check_device_error() == 0
    ref = oracle.decode(inp.q, inp.rho, inp.k_cache, inp.v_cache, inp.seqlens)
    assert_bf16(o, ref, "decode after the timeout was cleared")


def test_prefill_wait_gives_up_and_later_launches_stand_down():
    assert px.parallax_check_device_error() == 0
    inp = configs.prefill_inputs(1, 2, 300, 128, seed=72, device=DEV, dtype=torch.bfloat16)
    o = torch.full((1, 2, 300, 128), float("nan"), dtype=torch.float32, device=DEV)
    px.parallax_selftest_wait_timeout(px.SELFTEST_PREFILL, 2000)
    px.parallax_attn_prefill(inp.q, inp.rho, inp.k, inp.v, o, causal=True, scale=inp.scale)
    assert px.parallax_check_device_error() == px.DEVERR_WAIT_TIMEOUT
    assert torch.isnan(o).all()  # every CTA skipped its work (and freed its TMEM)
    px.parallax_attn_prefill(inp.q, inp.rho, inp.k, inp.v, o, causal=True, scale=inp.scale)
    assert px.parallax_check_device_error() == 0
    ref = oracle.prefill(inp.q, inp.rho, inp.k, inp.v, causal=True, scale=inp.scale)
    assert_bf16(o, ref, "prefill after the timeout was cleared")


def test_selftest_argument_errors():
    with pytest.raises(px.ParallaxError):
        px.parallax_selftest_wait_timeout(7, 100)
    with pytest.raises(px.ParallaxError):
        px.parallax_selftest_wait_timeout(px.SELFTEST_DECODE, 0)
    with pytest.raises(px.ParallaxError):
        px.parallax_selftest_wait_timeout(px.SELFTEST_DECODE, 2_000_000)
    assert px.parallax_check_device_error() == 0


def test_other_families_unaffected_by_a_decode_timeout():
    """A timeout in the decode family leaves the prefill family's word alone."""
    inp = configs.prefill_inputs(1, 1, 64, 64, seed=73, device=DEV, dtype=torch.bfloat16)
    px.parallax_selftest_wait_timeout(px.SELFTEST_DECODE, 1000)
    o = px.parallax_attn_prefill(inp.q, inp.rho, inp.k, inp.v, causal=True, scale=inp.scale)
    assert px.parallax_check_device_error() == px.DEVERR_WAIT_TIMEOUT
    ref = oracle.prefill(inp.q, inp.rho, inp.k, inp.v, causal=True, scale=inp.scale)
    assert np.isfinite(o.cpu().numpy()).all()
    assert_bf16(o, ref, "prefill beside a decode timeout")
