"""Pins for the oracle's backward pass (gradients of the Parallax prefill) and
for the per-row quantities a training forward keeps.

The gradient formulas in oracle.prefill_backward are derived by hand; they are
pinned to things that do not share that derivation:
  * central finite differences of the forward oracle (itself pinned by the
    base pins);
  * torch.autograd through an fp64 torch restatement of the forward written
    with the explicit d x d covariance (o = mu_v - C^T rho), a different
    algebra from the weighted-sum form the gradients use;
  * W_R = 0: the q, k, v gradients equal those of torch's fp64
    scaled_dot_product_attention (Parallax keeps softmax attention exactly,
    "Parallax mantem softmax ...", paragraph 2).
Planted mistakes in the gradient formulas fail at least one of them.
"""
import inspect
import textwrap

import numpy as np
import pytest
import torch

import oracle


def _torch_forward(q, rho, k, v, causal, scale):
    """fp64 torch restatement with the explicit covariance (autograd-able)."""
    L = q.shape[-2]
    s = scale * q @ k.transpose(-1, -2)
    if causal:
        s = s.masked_fill(~torch.ones(L, L, dtype=torch.bool).tril(), float("-inf"))
    p = torch.softmax(s, dim=-1)
    mu_v = p @ v
    mu_k = p @ k
    kc = k.unsqueeze(-3) - mu_k.unsqueeze(-2)          # [.., L_q, L_k, d]
    vc = v.unsqueeze(-3) - mu_v.unsqueeze(-2)
    C = torch.einsum("...ij,...ija,...ijc->...iac", p, kc, vc)  # [.., L_q, d, d]
    return mu_v - torch.einsum("...ia,...iac->...ic", rho, C)


def _draw(seed, B, H, L, d, rho_scale=0.5):
    rng = np.random.default_rng(seed)
    q, k, v, do = (rng.standard_normal((B, H, L, d)) for _ in range(4))
    rho = rho_scale * rng.standard_normal((B, H, L, d))
    return q, rho, 1.3 * k, v, do


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("seed,L,d", [(0, 4, 3), (1, 6, 2), (2, 1, 4)])
def test_finite_differences(causal, seed, L, d):
    q, rho, k, v, do = _draw(seed, 1, 2, L, d)
    scale = 1.0 / np.sqrt(d)
    grads = oracle.prefill_backward(q, rho, k, v, do, causal=causal, scale=scale)
    eps = 1e-6
    args = dict(q=q, rho=rho, k=k, v=v)
    for name, g in zip(("q", "rho", "k", "v"), grads):
        x = args[name]
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            fp = (oracle.prefill(**{**args, name: xp}, causal=causal, scale=scale) * do).sum()
            fm = (oracle.prefill(**{**args, name: xm}, causal=causal, scale=scale) * do).sum()
            num[idx] = (fp - fm) / (2 * eps)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-7, err_msg=f"d{name}")


@pytest.mark.parametrize("causal", [True, False])
def test_autograd_explicit_covariance(causal):
    q, rho, k, v, do = _draw(7, 2, 2, 7, 5)
    scale = 0.4
    grads = oracle.prefill_backward(q, rho, k, v, do, causal=causal, scale=scale)
    t = [torch.tensor(a, requires_grad=True) for a in (q, rho, k, v)]
    o = _torch_forward(*t, causal, scale)
    (o * torch.tensor(do)).sum().backward()
    for name, g, ti in zip(("q", "rho", "k", "v"), grads, t):
        np.testing.assert_allclose(g, ti.grad.numpy(), rtol=1e-11, atol=1e-12,
                                   err_msg=f"d{name}")


@pytest.mark.parametrize("causal", [True, False])
def test_zero_probe_is_softmax_attention(causal):
    q, _, k, v, do = _draw(3, 1, 3, 6, 4)
    dq, drho, dk, dv = oracle.prefill_backward(q, None, k, v, do, causal=causal)
    t = [torch.tensor(a, requires_grad=True) for a in (q, k, v)]
    o = torch.nn.functional.scaled_dot_product_attention(*t, is_causal=causal)
    (o * torch.tensor(do)).sum().backward()
    for g, ti in zip((dq, dk, dv), t):
        np.testing.assert_allclose(g, ti.grad.numpy(), rtol=1e-11, atol=1e-12)
    # the probe still gets a gradient at rho = 0 (W_R is trained from there)
    assert np.abs(drho).max() > 1e-3


def test_stats_against_library():
    q, rho, k, v, _ = _draw(4, 1, 2, 5, 3)
    scale = 1.0 / np.sqrt(3)
    lse, rbar, mu = oracle.prefill_stats(q, rho, k, v, causal=True, scale=scale)
    s = scale * torch.tensor(q) @ torch.tensor(k).transpose(-1, -2)
    s = s.masked_fill(~torch.ones(5, 5, dtype=torch.bool).tril(), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), rtol=1e-13, atol=1e-13)
    sdpa = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q), torch.tensor(k), torch.tensor(v), is_causal=True, scale=scale)
    np.testing.assert_allclose(mu, sdpa.numpy(), rtol=1e-12, atol=1e-12)
    p = torch.softmax(s, -1).numpy()
    r = np.einsum("bhid,bhjd->bhij", rho, k)
    np.testing.assert_allclose(rbar, (p * r).sum(-1), rtol=1e-12, atol=1e-12)


MUTANTS = {
    "dr sign": ("dR = P * (abar[:, None] - Dm)", "dR = P * (Dm - abar[:, None])"),
    "ds drops D": ("+ Dm - delta[:, None])", "- delta[:, None])"),
    "dk misses probe term": ("dk[b, h] = scale * (dS.T @ qh) + dR.T @ rh",
                             "dk[b, h] = scale * (dS.T @ qh)"),
    "dv with softmax weights": ("dv[b, h] = Wt.T @ doh", "dv[b, h] = P.T @ doh"),
    "rbar shift sign": ("(rbar[:, None] - R) + Dm", "(R - rbar[:, None]) + Dm"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_planted_mistake(name):
    old, new = MUTANTS[name]
    src = textwrap.dedent(inspect.getsource(oracle.prefill_backward))
    assert old in src, old
    ns = dict(vars(oracle))
    exec(src.replace(old, new), ns)
    q, rho, k, v, do = _draw(9, 1, 2, 6, 3)
    got = ns["prefill_backward"](q, rho, k, v, do, causal=True, scale=0.5)
    t = [torch.tensor(a, requires_grad=True) for a in (q, rho, k, v)]
    (_torch_forward(*t, True, 0.5) * torch.tensor(do)).sum().backward()
    assert not all(np.allclose(g, ti.grad.numpy(), rtol=1e-9, atol=1e-9)
                   for g, ti in zip(got, t)), f"mutant survived: {name}"
