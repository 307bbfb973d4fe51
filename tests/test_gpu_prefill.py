"""Prefill parity: the CUDA path (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import softmax_covariance_correction_pass_b300 as px
from softmax_covariance_correction_pass_b300 import configs
from parity_util import assert_bf16, assert_f32, errors

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(inp, causal=True, rho=True):
    o = torch.full(inp.q.shape, float("nan"), dtype=torch.float32, device=DEV)
    px.parallax_attn_prefill(inp.q, inp.rho if rho else None, inp.k, inp.v, o, causal=causal,
                             scale=inp.scale)
    assert px.parallax_check_device_error() == 0
    return o


def _ref(inp, causal=True, rho=True, form="explicit"):
    return oracle.prefill(inp.q, inp.rho if rho else None, inp.k, inp.v, causal=causal,
                          scale=inp.scale, form=form)


# ---------------------------------------------------------------- fp32 (CUDA cores)
@pytest.mark.parametrize("variant", ["base", "rho0", "same_k"])
def test_causal_f32_workload(variant):
    inp = configs.causal_f32_inputs(DEV, variant)
    o = _run(inp)
    assert_f32(o, _ref(inp), variant)
    if variant == "same_k":  # zero correction: o_i = mean_{j<=i} v_j
        v = inp.v.double()
        mean = torch.cumsum(v, 2) / torch.arange(1, v.shape[2] + 1, device=DEV).view(1, 1, -1, 1)
        assert_f32(o, mean, "identical keys")
    if variant == "rho0":  # W_R = 0: plain softmax attention, and the rho = NULL path agrees
        o0 = _run(inp, rho=False)
        assert torch.equal(o0, o) or errors(o0, o)[0] < 1e-7
        sdpa = torch.nn.functional.scaled_dot_product_attention(
            inp.q.double(), inp.k.double(), inp.v.double(), is_causal=True, scale=inp.scale)
        assert_f32(o, sdpa, "sdpa")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("L", [1, 3, 37, 129, 300])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("rho", [True, False])
def test_f32_shapes(d, L, causal, rho):
    inp = configs.prefill_inputs(2, 2, L, d, seed=100 + L, device=DEV)
    assert_f32(_run(inp, causal, rho), _ref(inp, causal, rho), f"L={L} d={d}")


# ---------------------------------------------------------------- bf16 (tcgen05)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("L", [1, 2, 100, 128, 129, 256, 383, 640])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("rho", [True, False])
def test_bf16_shapes(d, L, causal, rho):
    inp = configs.prefill_inputs(1, 3, L, d, seed=200 + L, device=DEV, dtype=torch.bfloat16)
    assert_bf16(_run(inp, causal, rho), _ref(inp, causal, rho), f"L={L} d={d}")


@pytest.mark.parametrize("d", [64, 128])
def test_bf16_large_probe(d):
    # probe of layer-like size (rho entries ~ 0.9, so r = rho.k ~ 10): the
    # correction term is comparable to the output itself
    inp = configs.prefill_inputs(2, 2, 1024, d, seed=300, rho_scale=0.9, device=DEV,
                                 dtype=torch.bfloat16)
    rel, mx = assert_bf16(_run(inp), _ref(inp, form="contracted"), "large probe")


@pytest.mark.parametrize("kind", ["ramp", "tile_steps", "small_steps"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("rho", [True, False])
def test_bf16_growing_scores(kind, causal, rho):
    # Scores that grow along the keys, so that the running row maximum moves by more
    # than the lazy-rescale threshold after the first key tile: "ramp" raises it inside
    # every tile (both halves of a tile exceed the maximum so far), "tile_steps" raises
    # it once at the start of every 128-key tile; "small_steps" raises it by ~3 (log2
    # units) per tile, so that a tile's weights sum to more than 2^8 while its maximum is
    # still within the threshold of the running one (until the steps add up).
    inp = configs.prefill_inputs(1, 2, 640, 128, seed=303, device=DEV, dtype=torch.bfloat16)
    q, k = inp.q.float().clone(), inp.k.float().clone() * 0.5
    q[..., 0] = 8.0
    j = torch.arange(640, device=DEV, dtype=torch.float32)
    # per key, in log2 units of the softmax: 8 * k0 * scale * log2(e)
    step = {"tile_steps": 12.0, "small_steps": 3.0}.get(kind, 0.0)
    k[..., 0] = 0.245 * j if kind == "ramp" else step * torch.div(j, 128, rounding_mode="floor")
    rh = inp.rho.clone()
    rh[..., 0] = 0  # keeps r = rho.k of ordinary size
    inp = configs.PrefillInputs(q.bfloat16(), k.bfloat16(), inp.v, rh, inp.scale)
    assert_bf16(_run(inp, causal, rho), _ref(inp, causal, rho, form="contracted"),
                f"{kind} causal={causal} rho={rho}")


def test_bf16_rho_zero_is_softmax():
    inp = configs.prefill_inputs(2, 4, 700, 128, seed=301, device=DEV, dtype=torch.bfloat16)
    inp.rho = torch.zeros_like(inp.rho)
    o = _run(inp)
    o_none = _run(inp, rho=False)
    # rho = 0 runs the correction kernel, rho = NULL the softmax-only one: both must
    # be softmax attention (they may differ by bf16 rounding of P)
    sdpa = torch.nn.functional.scaled_dot_product_attention(
        inp.q.double(), inp.k.double(), inp.v.double(), is_causal=True, scale=inp.scale)
    assert_bf16(o_none, sdpa, "rho=NULL vs sdpa")
    assert_bf16(o, sdpa, "rho=0 vs sdpa")
    assert_bf16(o, o_none, "rho=0 vs rho=NULL")


def test_bf16_invariants():
    inp = configs.prefill_inputs(1, 2, 513, 128, seed=302, device=DEV, dtype=torch.bfloat16)
    # value shift: v on a 1/8 grid so that v + b is exact in bf16
    vq = ((inp.v.float() * 8).round() / 8).bfloat16()
    inp = configs.PrefillInputs(inp.q, inp.k, vq, inp.rho, inp.scale)
    o = _run(inp).double()
    b = torch.tensor([0.5, -1.0, 2.0, 0.25] * 32, device=DEV)
    shifted = configs.PrefillInputs(inp.q, inp.k, (vq.float() + b).bfloat16(), inp.rho, inp.scale)
    assert torch.equal(shifted.v.float(), vq.float() + b)
    o2 = _run(shifted).double()
    assert (o2 - o - b).abs().max().item() < 2e-2
    # affine in rho: o(a r1 + (1-a) r2) = a o(r1) + (1-a) o(r2), with exact bf16 combinations
    r2 = torch.zeros_like(inp.rho)
    mid = configs.PrefillInputs(inp.q, inp.k, inp.v, (inp.rho.float() * 0.5).bfloat16(), inp.scale)
    o_mid = _run(mid).double()
    o_zero = _run(configs.PrefillInputs(inp.q, inp.k, inp.v, r2, inp.scale)).double()
    assert (o_mid - 0.5 * (o + o_zero)).abs().max().item() < 2e-2


def test_layer_prefill_full_size_sampled():
    """Full layer shape (B=8, H=16, L=4096, d=128, projections of x): sampled rows (rows 0-3
    and L-1 of every head plus 2048 random rows), each against the explicit d x d covariance
    form of the oracle."""
    inp = configs.layer_prefill_inputs(DEV)
    o = _run(inp)
    B, H, L, d = inp.q.shape
    rng = np.random.default_rng(5)
    rows = {}
    for b in range(B):
        for h in range(H):
            rows.setdefault((b, h), set()).update({0, 1, 2, 3, L - 1})
    for _ in range(2048):
        rows.setdefault((int(rng.integers(B)), int(rng.integers(H))), set()).add(
            int(rng.integers(L)))
    got, want = [], []
    for (b, h), idx in sorted(rows.items()):
        idx = np.array(sorted(idx))
        K, V = inp.k[b, h], inp.v[b, h]
        ref = oracle.rows(inp.q[b, h, idx], inp.rho[b, h, idx], K, V, idx + 1, inp.scale,
                          "explicit")
        got.append(o[b, h, idx].double().cpu().numpy())
        want.append(ref)
    got, want = np.concatenate(got), np.concatenate(want)
    rel, mx = assert_bf16(got, want, "layer prefill sampled rows")
    print(f"layer prefill sampled rows: rel-L2 {rel:.3e} max-abs {mx:.3e} over {len(got)} rows")


def test_layer_prefill_full_size_whole_heads():
    """Full layer shape: eight whole heads -- (0, 0) and one random head of every other
    sequence, all 4096 rows of each -- against the oracle's contracted form (the same
    function as the explicit covariance form, pinned to it on the CPU), so the max-abs
    bound is checked on every row of those heads, not on a sample."""
    inp = configs.layer_prefill_inputs(DEV)
    o = _run(inp)
    B, H, L, d = inp.q.shape
    rng = np.random.default_rng(55)
    heads = [(0, 0)] + [(b, int(rng.integers(H))) for b in range(1, B)]
    got, want = [], []
    for b, h in heads:
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = oracle.prefill(inp.q[sl], inp.rho[sl], inp.k[sl], inp.v[sl], causal=True,
                             scale=inp.scale, form="contracted")
        got.append(o[sl].double().cpu().numpy())
        want.append(ref)
        rel_h, mx_h = errors(got[-1], ref)
        print(f"layer prefill head ({b},{h}): rel-L2 {rel_h:.3e} max-abs {mx_h:.3e}")
    rel, mx = assert_bf16(np.concatenate(got), np.concatenate(want), "layer prefill whole heads")
    print(f"layer prefill whole heads: rel-L2 {rel:.3e} max-abs {mx:.3e} over {len(heads) * L} rows")


def test_layer_prefill_full_size_properties():
    """Whole-tensor checks at full size: every element written and finite, and the
    rho = NULL path equals torch's SDPA on the same bf16 tensors."""
    inp = configs.layer_prefill_inputs(DEV)
    o = _run(inp, rho=False)
    assert torch.isfinite(o).all()
    sdpa = torch.nn.functional.scaled_dot_product_attention(
        inp.q.float(), inp.k.float(), inp.v.float(), is_causal=True, scale=inp.scale)
    rel, mx = errors(o, sdpa)
    assert rel < 1e-2 and mx < 2e-2, (rel, mx)
