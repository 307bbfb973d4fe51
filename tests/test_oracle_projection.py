"""Pins for the oracle's q/k/v/probe projection (rho = W_R x, "Parallax mantem
softmax ...", paragraph 2), against facts that do not come from the oracle:

  * brute force: exact integer arithmetic in pure Python, indexing the output
    [B, H, L, d] and the stacked weight rows by hand;
  * closed form: a one-hot token x_l = e_a yields column a of the weight,
    scattered to the head-major layout;
  * linearity in x and in w.
A transposed layout (L and H swapped), a wrong block order (q/k/v/rho) or a
transposed weight fails at least one of them.
"""
import numpy as np
import pytest

import oracle


def _brute(x, w, H, d):
    B, L, width = len(x), len(x[0]), len(x[0][0])
    n_out = len(w) // (H * d)
    out = [[[[[0] * d for _ in range(L)] for _ in range(H)] for _ in range(B)]
           for _ in range(n_out)]
    for t in range(n_out):
        for b in range(B):
            for h in range(H):
                for l in range(L):
                    for c in range(d):
                        row = t * H * d + h * d + c
                        out[t][b][h][l][c] = sum(x[b][l][a] * w[row][a] for a in range(width))
    return out


@pytest.mark.parametrize("B,L,width,H,d,n_out", [(1, 1, 1, 1, 1, 1), (2, 3, 5, 2, 3, 4),
                                                 (1, 4, 7, 3, 2, 3), (3, 2, 4, 1, 4, 4)])
def test_brute_force_integers(B, L, width, H, d, n_out):
    rng = np.random.default_rng(B * 100 + L * 10 + width)
    x = rng.integers(-9, 10, (B, L, width))
    w = rng.integers(-9, 10, (n_out * H * d, width))
    ref = _brute(x.tolist(), w.tolist(), H, d)
    got = oracle.qkvr_projection(x, w, H, d)
    assert len(got) == n_out
    for t in range(n_out):
        assert got[t].shape == (B, H, L, d)
        np.testing.assert_array_equal(got[t], np.array(ref[t], dtype=np.float64))


def test_one_hot_token_selects_weight_columns():
    B, L, width, H, d = 2, 5, 6, 3, 4
    rng = np.random.default_rng(7)
    w = rng.standard_normal((4 * H * d, width))
    x = np.zeros((B, L, width))
    picks = {(0, 0): 2, (0, 3): 5, (1, 1): 0, (1, 4): 3}
    for (b, l), a in picks.items():
        x[b, l, a] = 1.0
    q, k, v, rho = oracle.qkvr_projection(x, w, H, d)
    for (b, l), a in picks.items():
        for t, out in enumerate((q, k, v, rho)):
            for h in range(H):
                np.testing.assert_array_equal(out[b, h, l], w[t * H * d + h * d:
                                                              t * H * d + (h + 1) * d, a])
    # tokens with x = 0 project to 0
    assert np.all(q[0, :, 1] == 0) and np.all(rho[1, :, 2] == 0)


def test_linear_in_x_and_w():
    B, L, width, H, d = 2, 3, 8, 2, 4
    rng = np.random.default_rng(3)
    x1, x2 = rng.standard_normal((2, B, L, width))
    w1, w2 = rng.standard_normal((2, 4 * H * d, width))
    a = 0.37
    lhs = oracle.qkvr_projection(a * x1 + x2, w1, H, d)
    rhs = [a * p + r for p, r in zip(oracle.qkvr_projection(x1, w1, H, d),
                                     oracle.qkvr_projection(x2, w1, H, d))]
    for u, v in zip(lhs, rhs):
        np.testing.assert_allclose(u, v, rtol=1e-12, atol=1e-12)
    lhs = oracle.qkvr_projection(x1, a * w1 + w2, H, d)
    rhs = [a * p + r for p, r in zip(oracle.qkvr_projection(x1, w1, H, d),
                                     oracle.qkvr_projection(x1, w2, H, d))]
    for u, v in zip(lhs, rhs):
        np.testing.assert_allclose(u, v, rtol=1e-12, atol=1e-12)


def test_three_blocks_without_probe():
    """A weight with three blocks (W_R = 0 dropped) gives q, k, v only, equal to
    the first three outputs of the four-block weight."""
    rng = np.random.default_rng(11)
    x = rng.standard_normal((1, 4, 8))
    w = rng.standard_normal((4 * 2 * 4, 8))
    four = oracle.qkvr_projection(x, w, 2, 4)
    three = oracle.qkvr_projection(x, w[:3 * 2 * 4], 2, 4)
    assert len(three) == 3
    for u, v in zip(three, four[:3]):
        np.testing.assert_array_equal(u, v)


# ----------------------------------------------------------------------------
# planted mistakes: each textual mutation of the oracle's projection must fail
# one of the pins above
# ----------------------------------------------------------------------------
import inspect  # noqa: E402
import textwrap  # noqa: E402

MUTANTS = {
    "L and H swapped in the output layout": (".transpose(0, 2, 1, 3)", ""),
    "weight not transposed": ("@ w.T", "@ w.reshape(w.shape[1], w.shape[0])"),
    "blocks read head-major": ("y.reshape(B, L, n_out, H, d)",
                               "y.reshape(B, L, H, n_out, d).transpose(0, 1, 3, 2, 4)"),
    "columns within a head reversed": ("y[:, :, t]", "y[:, :, t, :, ::-1]"),
}


def _mutant(old, new):
    src = textwrap.dedent(inspect.getsource(oracle.qkvr_projection))
    assert old in src, old
    ns = {"np": np, "_f64": oracle._f64}
    exec(src.replace(old, new), ns)
    return ns["qkvr_projection"]


def _pins_pass(fn) -> bool:
    try:
        rng = np.random.default_rng(0)
        for B, L, width, H, d, n_out in [(2, 3, 5, 2, 3, 4), (1, 4, 7, 3, 2, 3)]:
            x = rng.integers(-9, 10, (B, L, width))
            w = rng.integers(-9, 10, (n_out * H * d, width))
            ref = _brute(x.tolist(), w.tolist(), H, d)
            got = fn(x, w, H, d)
            for t in range(n_out):
                if got[t].shape != (B, H, L, d) or not np.array_equal(got[t], np.array(ref[t])):
                    return False
        return True
    except Exception:
        return False


def test_pins_accept_the_oracle():
    assert _pins_pass(oracle.qkvr_projection)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_planted_mistake(name):
    old, new = MUTANTS[name]
    assert not _pins_pass(_mutant(old, new)), f"mutant survived: {name}"
