"""Pins for the oracle's exact local linear attention (LLA) decode, the method
the Parallax probe replaces.

  * the conjugate-gradient step: with d iterations it solves a symmetric
    positive definite system exactly up to rounding (numpy.linalg.solve);
  * the LLA output is the intercept of the softmax-weighted least-squares fit
    of v on [1, k - q] (numpy.linalg.lstsq): local linear regression around
    the query, whose intercept is mu_v - C^T Sigma_kk^-1 (mu_k - q);
  * the returned probe satisfies Sigma_kk rho = mu_k - q.
Planted mistakes (sign of the right-hand side, an uncentered key covariance,
the value covariance in place of the key covariance) fail the fit pin.
"""
import inspect
import textwrap

import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("n,seed", [(3, 0), (8, 1), (16, 2)])
def test_cg_solves_spd_systems(n, seed):
    rng = np.random.default_rng(seed)
    M = rng.standard_normal((n, n))
    A = M @ M.T / n + 0.5 * np.eye(n)  # well conditioned: CG is exact to rounding in n steps
    b = rng.standard_normal(n)
    x = oracle.conjugate_gradient(A, b, n)
    np.testing.assert_allclose(x, np.linalg.solve(A, b), rtol=1e-9, atol=1e-10)


def _fit_intercept(q, K, V, scale):
    s = scale * (K @ q)
    p = np.exp(s - s.max())
    p /= p.sum()
    X = np.hstack([np.ones((len(K), 1)), K - q])
    sw = np.sqrt(p)[:, None]
    coef, *_ = np.linalg.lstsq(X * sw, V * sw, rcond=None)
    return coef[0]


def _draw(seed, B=2, H=2, L=24, d=4):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, d))
    k = rng.standard_normal((B, H, L, d))
    v = rng.standard_normal((B, H, L, d))
    return q, k, v


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_lla_is_local_linear_fit_intercept(seed):
    q, k, v = _draw(seed)
    sl = np.array([24, 13])
    o, rho = oracle.lla_decode(q, k, v, sl)
    d = q.shape[-1]
    for b in range(2):
        for h in range(2):
            n = sl[b]
            ref = _fit_intercept(q[b, h], k[b, h, :n], v[b, h, :n], 1.0 / np.sqrt(d))
            np.testing.assert_allclose(o[b, h], ref, rtol=1e-9, atol=1e-10)


def test_probe_solves_the_normal_equations():
    q, k, v = _draw(5)
    sl = np.array([24, 24])
    _, rho = oracle.lla_decode(q, k, v, sl)
    d = q.shape[-1]
    for b in range(2):
        for h in range(2):
            K = k[b, h]
            s = (K @ q[b, h]) / np.sqrt(d)
            p = np.exp(s - s.max())
            p /= p.sum()
            mu = p @ K
            sigma = ((K - mu) * p[:, None]).T @ (K - mu)
            np.testing.assert_allclose(sigma @ rho[b, h], mu - q[b, h], rtol=1e-9, atol=1e-10)


def test_empty_sequence():
    q, k, v = _draw(6)
    o, rho = oracle.lla_decode(q, k, v, np.array([0, 5]))
    assert np.all(o[0] == 0) and np.all(rho[0] == 0)


MUTANTS = {
    "rhs sign": ("mu_k - q[b, h], iters", "q[b, h] - mu_k, iters"),
    "uncentered key covariance": ("Kc = K - mu_k", "Kc = K"),
    "value covariance": ("sigma = (Kc * p[:, None]).T @ Kc",
                         "sigma = (Kc * p[:, None]).T @ (vc[b, h, :n] - p @ vc[b, h, :n])"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_planted_mistake(name):
    old, new = MUTANTS[name]
    src = textwrap.dedent(inspect.getsource(oracle.lla_decode))
    assert old in src, old
    ns = dict(vars(oracle))
    exec(src.replace(old, new), ns)
    q, k, v = _draw(7)
    sl = np.array([24, 20])
    o, _ = ns["lla_decode"](q, k, v, sl)
    ref = _fit_intercept(q[0, 0], k[0, 0], v[0, 0], 0.5)
    assert not np.allclose(o[0, 0], ref, rtol=1e-6, atol=1e-6), f"mutant survived: {name}"
