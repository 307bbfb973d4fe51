"""GPU parity of the q/k/v/probe projection (tcgen05 GEMM) against the fp64 oracle.

The kernel multiplies bf16 inputs with fp32 accumulation and rounds the result
to bf16, so each output element obeys
    |got - y| <= 2^-8 |y| + 2 * width * 2^-24 * sum_a |x_a| |w_a|
(y the exact product: bf16 round-to-nearest loses at most half an ulp, 2^-8
relative; the fp32 sum of `width` products at most width * 2^-24 times the sum
of their magnitudes, doubled for slack).  The tests check that bound element
by element and the bf16 criterion (rel-L2 <= 1e-2, max-abs <= 2e-2) over the
whole output.
"""
import numpy as np
import pytest
import torch

import oracle
import softmax_covariance_correction_pass_b300 as px
from softmax_covariance_correction_pass_b300 import configs
from parity_util import assert_bf16, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _check(outs, x, w, H, d, what):
    ref = oracle.qkvr_projection(x, w, H, d)
    mag = oracle.qkvr_projection(to_np(x).__abs__(), to_np(w).__abs__(), H, d)
    width = x.shape[-1]
    assert len([o for o in outs if o is not None]) == len(ref)
    for t, (got, r, m) in enumerate(zip(outs, ref, mag)):
        g = to_np(got)
        bound = 2.0 ** -8 * np.abs(r) + 2 * width * 2.0 ** -24 * m + 1e-30
        bad = np.abs(g - r) > bound
        assert not bad.any(), (f"{what} output {t}: {bad.sum()} elements beyond the rounding "
                               f"bound, worst {np.max(np.abs(g - r) - bound):.3e}")
        assert_bf16(g, r, f"{what} output {t}")


@pytest.mark.parametrize("B,L,width,H,d", [
    (1, 128, 64, 2, 64),      # one tile, 128-wide feature tiles
    (2, 300, 200, 2, 128),    # ragged L and ragged width (zero-filled K tail)
    (1, 1, 8, 1, 128),        # a single token, the smallest width
    (3, 77, 512, 4, 64),      # 256-wide feature tiles, L shorter than a tile
    (2, 257, 2048, 16, 128),  # full layer width and heads, ragged tail
])
@pytest.mark.parametrize("with_rho", [True, False])
def test_projection_matches_oracle(B, L, width, H, d, with_rho):
    n_out = 4 if with_rho else 3
    x, w = configs.projection_inputs(B, L, width, H, d, n_out, seed=B * 1000 + L, device=DEV)
    outs = px.parallax_attn_qkvr_projection(x, w, H, d, with_rho=with_rho)
    torch.cuda.synchronize()
    assert px.parallax_check_device_error() == 0
    if not with_rho:
        assert outs[3] is None
    _check(outs, x, w, H, d, f"B={B} L={L} width={width} H={H} d={d} rho={with_rho}")


def test_layer_size_sampled_rows():
    """The layer-shaped workload at full size (B=8, L=4096, width 2048, H=16,
    d=128): 64 sampled tokens checked against the oracle, and every output
    against torch's own bf16 projection of the same draws (same inputs,
    different summation order: equal up to a few bf16 ulps)."""
    x, w = configs.layer_projection_inputs(DEV)
    c = configs.LAYER_PREFILL
    H, d = c["H"], c["d"]
    outs = px.parallax_attn_qkvr_projection(x, w, H, d)
    torch.cuda.synchronize()
    assert px.parallax_check_device_error() == 0
    B, L, width = x.shape
    rng = np.random.default_rng(5)
    ls = np.sort(rng.choice(L, 64, replace=False))
    ls[0], ls[-1] = 0, L - 1
    idx = torch.as_tensor(ls, device=DEV)
    sub = [o.index_select(2, idx) for o in outs]
    _check(sub, x.index_select(1, idx), w, H, d, "layer-size sample")
    ref = configs.layer_prefill_inputs(DEV)
    for got, r in zip(outs, (ref.q, ref.k, ref.v, ref.rho)):
        diff = (got.float() - r.float()).abs()
        assert float(diff.max()) <= 2.0 ** -6 * float(r.float().abs().max())
        assert float(diff.norm() / r.float().norm()) <= 4e-3


def test_projection_feeds_prefill():
    """The projection's outputs go straight into the prefill: the whole layer
    (projection then attention) against the oracle on a small case."""
    B, L, width, H, d = 1, 200, 256, 2, 128
    x, w = configs.projection_inputs(B, L, width, H, d, 4, seed=21, device=DEV)
    w[3 * H * d:] *= 0.1  # a small probe, as a learned W_R would be near its init
    q, k, v, rho = px.parallax_attn_qkvr_projection(x, w, H, d)
    o = px.parallax_attn_prefill(q, rho, k, v, causal=True)
    torch.cuda.synchronize()
    assert px.parallax_check_device_error() == 0
    # the oracle attends over the bf16 values the kernel produced
    ref = oracle.prefill(q, rho, k, v, causal=True, scale=1.0 / np.sqrt(d))
    assert_bf16(o, ref, "projection + prefill")


def test_projection_rejects_bad_arguments():
    x = torch.zeros((1, 8, 64), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(px.ParallaxError) as e:  # H*d not a multiple of 128
        px.parallax_attn_qkvr_projection(x, torch.zeros((4 * 1 * 64, 64), dtype=torch.bfloat16,
                                                        device=DEV), 1, 64)
    assert e.value.code == px.PARALLAX_ERR_UNSUPPORTED
    x = torch.zeros((1, 8, 60), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(px.ParallaxError) as e:  # width not a multiple of 8
        px.parallax_attn_qkvr_projection(x, torch.zeros((4 * 128, 60), dtype=torch.bfloat16,
                                                        device=DEV), 1, 128)
    assert e.value.code == px.PARALLAX_ERR_UNSUPPORTED
