"""The CUDA kernels evaluate the method through rearranged formulas; this file restates
each rearrangement in numpy (fp64, on the CPU) and checks it against the oracle's direct
form on random values, so that a sign or term slip in the restatement is caught without a
GPU.  (The GPU tests compare the kernels themselves with the oracle.)

  * backward, per (query, key): the row statistics are stored as nl = -lse log2(e),
    rb1 = 1 + rbar, ab = abar, ne = delta - abar; with g = rb1 - r and u = ab - D,
      w = p g,   dr = p u,   ds * scale = -scale * p * (u g + ne),   p = 2^(s * scale * log2(e) + nl);
  * forward: o = U/l - (W/l - (A/l)(U/l)) with W and A taken over r - c for a per-row shift c
    (any c gives the same o) and with the exponentials taken against a stale running max;
  * exact LLA: Sigma_kk = G_kk / l - mu_k mu_k^T and C = G_kv / l - mu_k mu_v^T from the
    unnormalised weights, accumulated in two interleaved partial sums.
"""
import numpy as np

import oracle

LOG2E = 1.4426950408889634


def test_backward_pair_terms_match_the_direct_form():
    rng = np.random.default_rng(3)
    n = 4000
    s, r, D = rng.normal(size=n), rng.normal(size=n), rng.normal(size=n)
    lse, rbar = rng.normal(size=n) + 2.0, 0.3 * rng.normal(size=n)
    abar, delta = rng.normal(size=n), rng.normal(size=n)
    scale = 1.0 / np.sqrt(128.0)
    # direct form (the oracle's backward, per pair)
    p = np.exp(scale * s - lse)
    w_ref = p * (1.0 + rbar - r)
    dr_ref = p * (abar - D)
    ds_ref = p * ((D - abar) * (rbar - r) + D - delta) * scale
    # the kernels' form
    nl, rb1, ab, ne = -lse * LOG2E, 1.0 + rbar, abar, delta - abar
    p2 = np.exp2(s * scale * LOG2E + nl)
    g = rb1 - r
    u = ab - D
    np.testing.assert_allclose(p2, p, rtol=1e-13)
    np.testing.assert_allclose(p2 * g, w_ref, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(p2 * u, dr_ref, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(-scale * p2 * (u * g + ne), ds_ref, rtol=1e-10, atol=1e-14)


def test_forward_shift_and_stale_max_do_not_change_the_output():
    rng = np.random.default_rng(4)
    L, d = 37, 16
    q, k, v = (rng.normal(size=(L, d)) for _ in range(3))
    rho = 0.1 * rng.normal(size=(L, d))
    scale = 1.0 / np.sqrt(d)
    ref = oracle.prefill(q[None, None], rho[None, None], k[None, None], v[None, None],
                         causal=False, scale=scale)[0, 0]
    s = scale * (q @ k.T)
    r = rho @ k.T
    for c_shift, m_lag in ((0.0, 0.0), (0.7, 3.0), (-2.5, 7.9)):
        m = s.max(axis=1, keepdims=True) - m_lag  # a running max that lags the true one
        p = np.exp(s - m)
        c = c_shift + (p * r).sum(axis=1, keepdims=True) / p.sum(axis=1, keepdims=True)
        l = p.sum(axis=1, keepdims=True)
        U = p @ v
        W = (p * (r - c)) @ v
        A = (p * (r - c)).sum(axis=1, keepdims=True)
        o = U / l - (W / l - (A / l) * (U / l))
        np.testing.assert_allclose(o, ref, rtol=1e-11, atol=1e-12)


def test_lla_moments_from_unnormalised_interleaved_sums():
    rng = np.random.default_rng(5)
    n, d = 300, 8
    K, V = rng.normal(size=(n, d)) + 0.5, rng.normal(size=(n, d))
    q = rng.normal(size=d)
    s = (K @ q) / np.sqrt(d)
    pt = np.exp(s - s.max() + 3.0)  # weights against a lagging max, not normalised
    # two partial sums over interleaved 64-key tiles, added at the end
    tiles = [slice(j, min(j + 64, n)) for j in range(0, n, 64)]
    Gkk = sum((K[t] * pt[t, None]).T @ K[t] for t in tiles[0::2]) + \
        sum((K[t] * pt[t, None]).T @ K[t] for t in tiles[1::2])
    Gkv = sum((K[t] * pt[t, None]).T @ V[t] for t in tiles[0::2]) + \
        sum((K[t] * pt[t, None]).T @ V[t] for t in tiles[1::2])
    l = pt.sum()
    mk, mv = pt @ K / l, pt @ V / l
    sigma = Gkk / l - np.outer(mk, mk)
    C = Gkv / l - np.outer(mk, mv)
    p = pt / l
    sigma_ref = ((K - mk) * p[:, None]).T @ (K - mk)
    C_ref = ((K - mk) * p[:, None]).T @ (V - mv)
    np.testing.assert_allclose(sigma, sigma_ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(C, C_ref, rtol=1e-10, atol=1e-12)
    # and the output o = mu_v - C^T rho with rho = Sigma^-1 (mu_k - q) is the oracle's
    rho = np.linalg.solve(sigma, mk - q)
    o = mv - C.T @ rho
    ro, rr = oracle.lla_decode(q[None, None], K[None, None], V[None, None], np.array([n]))
    np.testing.assert_allclose(rho, rr[0, 0], rtol=1e-7, atol=1e-9)
    np.testing.assert_allclose(o, ro[0, 0], rtol=1e-7, atol=1e-9)
