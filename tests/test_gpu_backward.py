"""GPU parity of the training forward's row statistics and of the prefill
backward pass (dq, drho, dk, dv) against the fp64 oracle.

Tolerance for each gradient tensor: rel-L2 <= 1e-2 (the bf16 criterion of the
forward) and max-abs <= 2e-2 * max|ref| -- the forward's 2e-2 absolute bar
taken relative to the tensor's own scale, since gradients are not O(1) values:
the kernels round the p-weighted terms (W, dS, dR) to bf16 before the fp32
tensor-core accumulation, an error of at most 2^-8 relative per term.  The
oracle gets the exact bf16 values of q, rho, k, v and dout.
"""
import numpy as np
import pytest
import torch

import oracle
import softmax_covariance_correction_pass_b300 as px
from softmax_covariance_correction_pass_b300 import configs
from parity_util import assert_bf16, errors, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def assert_grad(got, ref, what):
    rel, mx = errors(got, ref)
    scale = float(np.abs(ref).max())
    if scale == 0.0:
        # an exactly-zero gradient (one key per row: dq = drho = 0): only rounding, of
        # a p (abar - D) difference of O(1) terms times O(1) keys
        assert mx <= 1e-4, f"{what}: zero gradient expected, max-abs {mx:.3e}"
        return rel, mx
    print(f"PARITY {what}: rel-L2 {rel:.3e} max-abs {mx:.3e} max|ref| {scale:.3g}")
    assert rel <= 1e-2 and mx <= 2e-2 * scale, \
        f"{what}: rel-L2 {rel:.3e} (<= 1e-2), max-abs {mx:.3e} (<= {2e-2 * scale:.3e})"
    return rel, mx


def _inputs(B, H, L, d, seed, with_rho=True):
    inp = configs.prefill_inputs(B, H, L, d, seed=seed, device=DEV, dtype=torch.bfloat16)
    g = torch.Generator(device=DEV).manual_seed(seed + 100)
    dout = torch.randn((B, H, L, d), generator=g, device=DEV).to(torch.bfloat16)
    return inp.q, (inp.rho if with_rho else None), inp.k, inp.v, dout, inp.scale


@pytest.mark.parametrize("B,H,L,d", [(1, 2, 128, 64), (2, 2, 300, 128), (1, 1, 77, 128)])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("with_rho", [True, False])
def test_train_forward_stats(B, H, L, d, causal, with_rho):
    q, rho, k, v, _, scale = _inputs(B, H, L, d, seed=L + d, with_rho=with_rho)
    o, lse, rbar, mu = px.parallax_attn_prefill_train(q, rho, k, v, causal=causal, scale=scale)
    o_plain = px.parallax_attn_prefill(q, rho, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert px.parallax_check_device_error() == 0
    assert torch.equal(o, o_plain)  # the statistics do not change the output
    rl, rr, rm = oracle.prefill_stats(q, rho, k, v, causal=causal, scale=scale)
    np.testing.assert_allclose(to_np(lse), rl, rtol=0, atol=1e-4)
    np.testing.assert_allclose(to_np(rbar), rr, rtol=0, atol=2e-3)
    assert_bf16(mu, rm, "mu_v")


# (1, 20, 200, 64): 20 heads = one full CTA-scheduling group of 16 heads plus a partial one
@pytest.mark.parametrize("B,H,L,d", [(1, 2, 128, 64), (2, 2, 300, 128), (1, 3, 200, 64),
                                     (1, 1, 1, 128), (1, 20, 200, 64)])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("with_rho", [True, False])
def test_backward_matches_oracle(B, H, L, d, causal, with_rho):
    q, rho, k, v, dout, scale = _inputs(B, H, L, d, seed=7 * L + d, with_rho=with_rho)
    o, lse, rbar, mu = px.parallax_attn_prefill_train(q, rho, k, v, causal=causal, scale=scale)
    dq, drho, dk, dv = px.parallax_attn_prefill_backward(q, rho, k, v, o, mu, lse, rbar, dout,
                                                         causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert px.parallax_check_device_error() == 0
    ref = oracle.prefill_backward(q, rho, k, v, dout, causal=causal, scale=scale)
    names = ("dq", "drho", "dk", "dv")
    for name, g, r in zip(names, (dq, drho, dk, dv), ref):
        if name == "drho" and not with_rho:
            assert g is None
            continue
        assert_grad(g, r, f"{name} B={B} H={H} L={L} d={d} causal={causal} rho={with_rho}")


def test_backward_layer_size_sampled_heads():
    """The layer-shaped workload at full size (B=8, H=16, L=4096, d=128): every
    gradient of eight whole heads -- (0, 0) and one random head of every other sequence --
    against the oracle."""
    inp = configs.layer_prefill_inputs(DEV)
    g = torch.Generator(device=DEV).manual_seed(44)
    dout = torch.randn(inp.q.shape, generator=g, device=DEV).to(torch.bfloat16)
    o, lse, rbar, mu = px.parallax_attn_prefill_train(inp.q, inp.rho, inp.k, inp.v, causal=True,
                                                      scale=inp.scale)
    grads = px.parallax_attn_prefill_backward(inp.q, inp.rho, inp.k, inp.v, o, mu, lse, rbar,
                                              dout, causal=True, scale=inp.scale)
    torch.cuda.synchronize()
    assert px.parallax_check_device_error() == 0
    rng = np.random.default_rng(66)
    for b, h in [(0, 0)] + [(b, int(rng.integers(16))) for b in range(1, 8)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = oracle.prefill_backward(inp.q[sl], inp.rho[sl], inp.k[sl], inp.v[sl], dout[sl],
                                      causal=True, scale=inp.scale)
        for name, gg, r in zip(("dq", "drho", "dk", "dv"), grads, ref):
            assert_grad(gg[sl], r, f"layer {name} b={b} h={h}")
