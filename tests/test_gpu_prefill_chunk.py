"""GPU parity of the chunked causal prefill (a chunk of new tokens continuing
cached sequences) against the fp64 oracle, plus the structural facts the
call promises: the chunk's keys and values land in the cache rows after the
cached prefix, and prefilling a sequence chunk by chunk gives the rows of one
whole-sequence prefill.

Tolerance: bf16 inputs with fp32 accumulation, rel-L2 <= 1e-2 and max-abs <=
2e-2 over the whole output.  The cache rows past the prefix are filled with
NaN before the call: the kernels must neither read them into a result nor
fail because of them.
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


def _case(B, H, Lq, Lmax, d, cache_lens, seed):
    g = configs.prefill_inputs(B, H, Lq, d, seed=seed, device=DEV, dtype=torch.bfloat16)
    cache = configs.prefill_inputs(B, H, Lmax, d, seed=seed + 1, device=DEV, dtype=torch.bfloat16)
    kc, vc = cache.k.clone(), cache.v.clone()
    for b, n in enumerate(cache_lens):
        kc[b, :, n:] = float("nan")
        vc[b, :, n:] = float("nan")
    cl = torch.tensor(cache_lens, dtype=torch.int32, device=DEV)
    return g, kc, vc, cl


@pytest.mark.parametrize("B,H,Lq,Lmax,d,cache_lens", [
    (2, 2, 128, 512, 128, [0, 384]),      # empty prefix; prefix of whole tiles
    (2, 2, 200, 700, 128, [37, 500]),     # ragged prefix and chunk, two query blocks
    (1, 3, 1, 300, 64, [299]),            # a single new token (decode as a chunk)
    (3, 1, 300, 1000, 64, [1, 129, 700]),
])
@pytest.mark.parametrize("with_rho", [True, False])
def test_chunk_matches_oracle(B, H, Lq, Lmax, d, cache_lens, with_rho):
    g, kc, vc, cl = _case(B, H, Lq, Lmax, d, cache_lens, seed=Lq + d)
    rho = g.rho if with_rho else None
    kc0, vc0 = kc.clone(), vc.clone()
    o = px.parallax_attn_prefill_chunk(g.q, rho, g.k, g.v, kc, vc, cl)
    torch.cuda.synchronize()
    assert px.parallax_check_device_error() == 0
    assert torch.isfinite(o).all()
    ref = oracle.prefill_chunk(g.q, rho, g.k, g.v, kc0, vc0, cache_lens)
    assert_bf16(o, ref, f"chunk B={B} H={H} Lq={Lq} prefix={cache_lens} rho={with_rho}")
    # the chunk's rows were appended after each prefix; the prefix is untouched
    for b, n in enumerate(cache_lens):
        assert torch.equal(kc[b, :, n:n + Lq], g.k[b])
        assert torch.equal(vc[b, :, n:n + Lq], g.v[b])
        assert torch.equal(kc[b, :, :n], kc0[b, :, :n])


def test_chunks_compose_to_one_prefill():
    """A 1000-token sequence prefilled in chunks of 300, 300, 256 and 144 tokens
    matches one causal parallax_attn_prefill over all 1000 (same kernel
    arithmetic per key tile; bf16 tolerance)."""
    B, H, L, d = 2, 2, 1000, 128
    full = configs.prefill_inputs(B, H, L, d, seed=3, device=DEV, dtype=torch.bfloat16)
    ref = px.parallax_attn_prefill(full.q, full.rho, full.k, full.v, causal=True)
    kc = torch.full((B, H, L, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    vc = torch.full_like(kc, float("nan"))
    cl = torch.zeros(B, dtype=torch.int32, device=DEV)
    outs, pos = [], 0
    for n in (300, 300, 256, 144):
        sl = slice(pos, pos + n)
        outs.append(px.parallax_attn_prefill_chunk(
            full.q[:, :, sl].contiguous(), full.rho[:, :, sl].contiguous(),
            full.k[:, :, sl].contiguous(), full.v[:, :, sl].contiguous(), kc, vc, cl))
        cl += n
        pos += n
    torch.cuda.synchronize()
    assert px.parallax_check_device_error() == 0
    got = torch.cat(outs, dim=2)
    assert torch.equal(kc, full.k) and torch.equal(vc, full.v)
    assert_bf16(got, ref.double().cpu().numpy(), "chunked vs whole prefill")
    oref = oracle.prefill(full.q, full.rho, full.k, full.v, causal=True)
    assert_bf16(got, oref, "chunked prefill vs oracle")


def test_chunk_prefix_clamped_and_flagged():
    g, kc, vc, _ = _case(1, 1, 64, 128, 64, [0], seed=1)
    cl = torch.tensor([100], dtype=torch.int32, device=DEV)  # 100 + 64 > 128
    px.parallax_attn_prefill_chunk(g.q, g.rho, g.k, g.v, kc, vc, cl)
    assert px.parallax_check_device_error() == px.DEVERR_SEQLEN_CLAMPED


def test_chunk_layer_size_sampled():
    """The layer-shaped prefill split in two: the first 3072 tokens as the cache,
    the last 1024 as a chunk (B=8, H=16, d=128); 4 heads checked against the
    oracle on sampled rows, every row against the whole-sequence prefill."""
    full = configs.layer_prefill_inputs(DEV)
    B, H, L, d = full.q.shape
    off, Lq = 3072, 1024
    kc, vc = full.k.clone(), full.v.clone()
    kc[:, :, off:] = float("nan")
    vc[:, :, off:] = float("nan")
    cl = torch.full((B,), off, dtype=torch.int32, device=DEV)
    sl = slice(off, L)
    o = px.parallax_attn_prefill_chunk(full.q[:, :, sl].contiguous(),
                                       full.rho[:, :, sl].contiguous(),
                                       full.k[:, :, sl].contiguous(),
                                       full.v[:, :, sl].contiguous(), kc, vc, cl)
    whole = px.parallax_attn_prefill(full.q, full.rho, full.k, full.v, causal=True)
    torch.cuda.synchronize()
    assert px.parallax_check_device_error() == 0
    assert_bf16(o, whole[:, :, sl].double().cpu().numpy(), "layer chunk vs whole")
    rng = np.random.default_rng(2)
    rows = np.sort(rng.choice(Lq, 16, replace=False))
    for b, h in ((0, 0), (3, 7), (5, 11), (7, 15)):
        q = full.q[b, h, off + rows]
        rho = full.rho[b, h, off + rows]
        ref = oracle.rows(q, rho, full.k[b, h], full.v[b, h], off + rows + 1, 1.0 / np.sqrt(d),
                          form="contracted")
        assert_bf16(o[b, h, rows], ref, f"layer chunk sample b={b} h={h}")
