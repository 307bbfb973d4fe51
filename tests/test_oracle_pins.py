"""Pins for the fp64 oracle against facts that do not come from the oracle itself.

Each test names what fixes the expected value:
  * brute force in 50-digit decimal arithmetic with a different algebra
    (raw second moments, C = E[k v^T] - E[k] E[v]^T);
  * closed forms derived by hand from the definition;
  * library routines: torch's fp64 scaled_dot_product_attention (W_R = 0 gives
    plain softmax attention: "Parallax mantem softmax", paragraph 2) and numpy's
    weighted least squares (the probe that makes the output the intercept of a
    local linear fit, the "local linear attention" reading of the same pages);
  * invariances that hold for the exact function.
A plausible mistake in the oracle (a dropped term, a flipped sign, a
transposed covariance, a wrong mask index, a wrong scale) fails at least one.
"""
import decimal
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FORMS = ["explicit", "contracted", "uncentered"]


# ----------------------------------------------------------------------------
# brute force: 50-digit decimal, uncentered second moments
# ----------------------------------------------------------------------------
def _brute_row(q, rho, K, V, scale):
    """o = mu_v - C^T rho with C = E_p[k v^T] - E_p[k] E_p[v]^T, all in Decimal."""
    D = decimal.Decimal
    with decimal.localcontext() as ctx:
        ctx.prec = 50
        n, d = len(K), len(q)
        if n == 0:
            return [0.0] * d
        s = [D(scale) * sum(D(q[a]) * D(K[j][a]) for a in range(d)) for j in range(n)]
        mx = max(s)
        w = [(sj - mx).exp() for sj in s]
        z = sum(w)
        p = [wj / z for wj in w]
        Ek = [sum(p[j] * D(K[j][a]) for j in range(n)) for a in range(d)]
        Ev = [sum(p[j] * D(V[j][c]) for j in range(n)) for c in range(d)]
        Ekv = [[sum(p[j] * D(K[j][a]) * D(V[j][c]) for j in range(n)) for c in range(d)]
               for a in range(d)]
        out = []
        for c in range(d):
            corr = D(0)
            if rho is not None:
                corr = sum(D(rho[a]) * (Ekv[a][c] - Ek[a] * Ev[c]) for a in range(d))
            out.append(float(Ev[c] - corr))
        return out


def _brute_prefill(q, rho, k, v, causal, scale):
    B, H, L, d = q.shape
    o = np.zeros_like(q)
    for b in range(B):
        for h in range(H):
            for i in range(L):
                n = i + 1 if causal else L
                o[b, h, i] = _brute_row(q[b, h, i], None if rho is None else rho[b, h, i],
                                        k[b, h, :n], v[b, h, :n], scale)
    return o


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("seed,L,d", [(0, 1, 1), (1, 3, 2), (2, 5, 3), (3, 6, 4), (4, 4, 4)])
def test_brute_force_decimal(form, causal, seed, L, d):
    rng = np.random.default_rng(seed)
    q, rho, k, v = (rng.standard_normal((1, 2, L, d)) for _ in range(4))
    k *= 1.5
    scale = 1.0 / np.sqrt(d)
    ref = _brute_prefill(q, rho, k, v, causal, scale)
    got = oracle.prefill(q, rho, k, v, causal=causal, scale=scale, form=form)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13 * max(1.0, np.abs(ref).max()))


def test_brute_force_hand_chosen():
    # large logits (softmax nearly one-hot), a tied pair, negative values
    q = np.array([[[[4.0, -2.0, 0.5], [0.0, 0.0, 0.0], [3.0, 3.0, -1.0], [1.0, -1.0, 2.0]]]])
    k = np.array([[[[2.0, 1.0, 0.0], [2.0, 1.0, 0.0], [-1.0, 3.0, 0.25], [0.5, 0.5, 0.5]]]])
    v = np.array([[[[1.0, -2.0, 3.0], [0.0, 4.0, -1.0], [2.5, 0.0, 1.0], [-3.0, 1.0, 1.0]]]])
    rho = np.array([[[[0.3, -0.7, 1.1], [2.0, 0.0, -1.0], [-0.5, 0.25, 0.0], [1.0, 1.0, 1.0]]]])
    for causal in (True, False):
        ref = _brute_prefill(q, rho, k, v, causal, 0.9)
        for form in FORMS:
            got = oracle.prefill(q, rho, k, v, causal=causal, scale=0.9, form=form)
            np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13)


def test_brute_force_decode_ragged():
    rng = np.random.default_rng(7)
    B, H, Lmax, d = 3, 2, 5, 3
    q, rho = rng.standard_normal((B, H, d)), rng.standard_normal((B, H, d))
    kc, vc = rng.standard_normal((B, H, Lmax, d)), rng.standard_normal((B, H, Lmax, d))
    seqlens = np.array([5, 1, 3], dtype=np.int32)
    for form in FORMS:
        got = oracle.decode(q, rho, kc, vc, seqlens, scale=0.6, form=form)
        for b in range(B):
            for h in range(H):
                n = seqlens[b]
                ref = _brute_row(q[b, h], rho[b, h], kc[b, h, :n], vc[b, h, :n], 0.6)
                np.testing.assert_allclose(got[b, h], ref, rtol=0, atol=1e-13)


# ----------------------------------------------------------------------------
# closed forms
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("form", FORMS)
def test_causal_row0_is_v0(form):
    # one key: p = 1, C = 0, so o_0 = v_0 whatever q, rho
    rng = np.random.default_rng(11)
    q, rho, k, v = (rng.standard_normal((2, 3, 7, 8)) for _ in range(4))
    rho *= 5.0
    o = oracle.prefill(q, rho, k, v, causal=True, form=form)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], rtol=0, atol=1e-14)


@pytest.mark.parametrize("form", FORMS)
def test_two_keys_closed_form(form):
    # keys k0, k1 with weights p, 1-p:
    #   mu_v = p v0 + (1-p) v1 ;  C = p (1-p) (k0 - k1)(v0 - v1)^T
    #   o = mu_v - p (1-p) (rho . (k0 - k1)) (v0 - v1)
    rng = np.random.default_rng(12)
    d, scale = 6, 0.37
    for _ in range(20):
        q, rho, k0, k1, v0, v1 = (rng.standard_normal(d) for _ in range(6))
        s0, s1 = scale * q @ k0, scale * q @ k1
        p = 1.0 / (1.0 + np.exp(s1 - s0))
        want = p * v0 + (1 - p) * v1 - p * (1 - p) * (rho @ (k0 - k1)) * (v0 - v1)
        got = oracle.rows(q[None], rho[None], np.stack([k0, k1]), np.stack([v0, v1]),
                          [2], scale, form=form)[0]
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-14)


@pytest.mark.parametrize("form", FORMS)
def test_identical_keys_zero_correction(form):
    # all k_j equal: p uniform over the visible keys and C = 0, so o_i = mean_{j<=i} v_j
    rng = np.random.default_rng(13)
    B, H, L, d = 1, 2, 9, 5
    q, rho, v = (rng.standard_normal((B, H, L, d)) for _ in range(3))
    k = np.broadcast_to(rng.standard_normal((B, H, 1, d)), (B, H, L, d)).copy()
    o = oracle.prefill(q, 10.0 * rho, k, v, causal=True, form=form)
    want = np.cumsum(v, axis=2) / np.arange(1, L + 1)[None, None, :, None]
    np.testing.assert_allclose(o, want, rtol=0, atol=1e-13)


def _golden_cases():
    path = os.path.join(GOLDEN, "closed_form_cases.txt")
    cases, cur = [], {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split("=", 1)
            key = key.strip()
            if key == "case":
                if cur:
                    cases.append(cur)
                cur = {"name": val.strip()}
            else:
                cur[key] = np.array(eval(val, {"__builtins__": {}}), dtype=np.float64)
    if cur:
        cases.append(cur)
    return cases


@pytest.mark.parametrize("form", FORMS)
def test_golden_closed_form_cases(form):
    cases = _golden_cases()
    assert len(cases) >= 3
    for c in cases:
        got = oracle.rows(c["q"][None], c["rho"][None], c["k"], c["v"], [len(c["k"])],
                          float(c["scale"]), form=form)[0]
        np.testing.assert_allclose(got, c["o"], rtol=0, atol=1e-14, err_msg=c["name"])


# ----------------------------------------------------------------------------
# library special cases
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("form", FORMS)
def test_rho_zero_is_sdpa(causal, form):
    # W_R = 0 recovers standard softmax attention exactly
    g = torch.Generator().manual_seed(21)
    B, H, L, d = 2, 3, 33, 16
    q, k, v = (torch.randn(B, H, L, d, generator=g, dtype=torch.float64) for _ in range(3))
    scale = 0.3
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale)
    for rho in (None, torch.zeros_like(q)):
        got = oracle.prefill(q, rho, k, v, causal=causal, scale=scale, form=form)
        np.testing.assert_allclose(got, ref.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("form", FORMS)
def test_local_linear_intercept(form):
    # With rho = Sigma_kk^{-1} (mu_k - q) the output equals the intercept of the
    # softmax-weighted least-squares fit v ~ b0 + B (k - q): exact local linear
    # attention is the probe choice that reproduces the local linear estimate.
    rng = np.random.default_rng(31)
    for d, n in [(2, 7), (3, 9), (4, 12)]:
        for _ in range(5):
            q = rng.standard_normal(d)
            K = rng.standard_normal((n, d))
            V = rng.standard_normal((n, d))
            scale = 0.8
            s = scale * K @ q
            p = np.exp(s - s.max())
            p /= p.sum()
            mu_k = p @ K
            Skk = (K - mu_k).T @ ((K - mu_k) * p[:, None])
            rho = np.linalg.solve(Skk, mu_k - q)
            X = np.hstack([np.ones((n, 1)), K - q])
            sw = np.sqrt(p)[:, None]
            coef, *_ = np.linalg.lstsq(X * sw, V * sw, rcond=None)
            want = coef[0]
            got = oracle.rows(q[None], rho[None], K, V, [n], scale, form=form)[0]
            np.testing.assert_allclose(got, want, rtol=0, atol=1e-10)


# ----------------------------------------------------------------------------
# invariances of the exact function
# ----------------------------------------------------------------------------
def _rand(seed, shape=(2, 2, 17, 8)):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal(shape) for _ in range(4)]


@pytest.mark.parametrize("form", FORMS)
def test_value_shift_shifts_output(form):
    q, rho, k, v = _rand(41)
    b = np.random.default_rng(42).standard_normal(8)
    o1 = oracle.prefill(q, rho, k, v, form=form)
    o2 = oracle.prefill(q, rho, k, v + b, form=form)
    np.testing.assert_allclose(o2, o1 + b, rtol=0, atol=1e-12)


@pytest.mark.parametrize("form", FORMS)
def test_key_shift_leaves_output(form):
    q, rho, k, v = _rand(43)
    a = np.random.default_rng(44).standard_normal(8)
    o1 = oracle.prefill(q, rho, k, v, form=form)
    o2 = oracle.prefill(q, rho, k + a, v, form=form)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)


@pytest.mark.parametrize("form", FORMS)
def test_affine_in_rho(form):
    q, rho1, k, v = _rand(45)
    rho2 = np.random.default_rng(46).standard_normal(rho1.shape)
    al = 0.3
    o = oracle.prefill(q, al * rho1 + (1 - al) * rho2, k, v, form=form)
    o1 = oracle.prefill(q, rho1, k, v, form=form)
    o2 = oracle.prefill(q, rho2, k, v, form=form)
    np.testing.assert_allclose(o, al * o1 + (1 - al) * o2, rtol=0, atol=1e-12)


@pytest.mark.parametrize("form", FORMS)
def test_noncausal_key_permutation(form):
    q, rho, k, v = _rand(47)
    perm = np.random.default_rng(48).permutation(k.shape[2])
    o1 = oracle.prefill(q, rho, k, v, causal=False, form=form)
    o2 = oracle.prefill(q, rho, k[:, :, perm], v[:, :, perm], causal=False, form=form)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)


def test_causal_mask_uses_prefix_only():
    # changing keys/values after position i must not change row i
    q, rho, k, v = _rand(49)
    o1 = oracle.prefill(q, rho, k, v, causal=True)
    k2, v2 = k.copy(), v.copy()
    k2[:, :, 9:] += 3.0
    v2[:, :, 9:] -= 2.0
    o2 = oracle.prefill(q, rho, k2, v2, causal=True)
    np.testing.assert_allclose(o2[:, :, :9], o1[:, :, :9], rtol=0, atol=0)
    assert np.abs(o2[:, :, 9:] - o1[:, :, 9:]).max() > 1e-3


# ----------------------------------------------------------------------------
# cross-form and cross-entry agreement
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [True, False])
def test_forms_agree(causal):
    q, rho, k, v = _rand(51, (1, 2, 64, 32))
    rho *= 3.0
    oe = oracle.prefill(q, rho, k, v, causal=causal, form="explicit")
    for form in ("contracted", "uncentered"):
        o = oracle.prefill(q, rho, k, v, causal=causal, form=form)
        np.testing.assert_allclose(o, oe, rtol=0, atol=1e-12 * np.abs(oe).max())


def test_decode_matches_prefill_last_row():
    # a decode step over n cached keys is the causal prefill row i = n-1
    q, rho, k, v = _rand(53, (2, 3, 12, 8))
    o = oracle.prefill(q, rho, k, v, causal=True)
    for n in (1, 5, 12):
        od = oracle.decode(q[:, :, n - 1], rho[:, :, n - 1], k, v,
                           np.full(2, n, dtype=np.int32))
        np.testing.assert_allclose(od, o[:, :, n - 1], rtol=0, atol=1e-14)


def test_empty_key_set_gives_zero():
    q, rho, k, v = _rand(55, (2, 1, 4, 8))
    od = oracle.decode(q[:, :, 0], rho[:, :, 0], k, v, np.array([0, 4], dtype=np.int32))
    assert np.all(od[0] == 0.0)
    assert np.abs(od[1]).max() > 0


def test_rejects_bad_seqlens():
    q, rho, k, v = _rand(57, (1, 1, 4, 8))
    with pytest.raises(RuntimeError):
        oracle.decode(q[:, :, 0], rho[:, :, 0], k, v, np.array([5], dtype=np.int32))
