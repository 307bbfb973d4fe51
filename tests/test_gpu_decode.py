"""Decode parity: split-KV decode + combine (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import softmax_covariance_correction_pass_b300 as px
from softmax_covariance_correction_pass_b300 import configs
from parity_util import assert_bf16, assert_f32, errors

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _reset_chunk():
    px.parallax_attn_set_decode_chunk_keys(0)
    yield
    px.parallax_attn_set_decode_chunk_keys(0)


def _run(inp, rho=True):
    B, H, d = inp.q.shape
    o = torch.full((B, H, d), float("nan"), dtype=torch.float32, device=DEV)
    px.parallax_attn_decode(inp.q, inp.rho if rho else None, inp.k_cache, inp.v_cache,
                            inp.seqlens, o)
    assert px.parallax_check_device_error() == 0
    return o


def _ref_heads(inp, heads, rho=True, form="contracted"):
    """Oracle rows for a list of (b, h), copying only those heads to the host."""
    d = inp.q.shape[-1]
    out = []
    for b, h in heads:
        n = int(inp.seqlens[b])
        K = inp.k_cache[b, h, :max(n, 1)]
        V = inp.v_cache[b, h, :max(n, 1)]
        out.append(oracle.rows(inp.q[b, h][None], inp.rho[b, h][None] if rho else None, K, V,
                               [n], 1.0 / np.sqrt(d), form)[0])
    return np.stack(out)


def _small(B, H, Lmax, d, seqlens, dtype, seed):
    return configs.decode_inputs(B, H, d, seqlens, Lmax, seed, device=DEV, dtype=dtype)


SEQ_CASES = [
    (1, [1]), (255, [255, 1, 100]), (256, [256, 0, 17]), (257, [257, 256, 1]),
    (1000, [1000, 999, 513]), (2049, [2049, 1, 1024]),
]


@pytest.mark.parametrize("chunk", [0, 256])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Lmax,seqlens", SEQ_CASES)
@pytest.mark.parametrize("rho", [True, False])
def test_bf16_small(chunk, d, Lmax, seqlens, rho):
    px.parallax_attn_set_decode_chunk_keys(chunk)
    inp = _small(len(seqlens), 3, Lmax, d, seqlens, torch.bfloat16, seed=Lmax + d)
    o = _run(inp, rho)
    ref = oracle.decode(inp.q, inp.rho if rho else None, inp.k_cache, inp.v_cache, inp.seqlens)
    assert_bf16(o, ref, f"Lmax={Lmax} d={d} chunk={chunk}")
    for b, n in enumerate(seqlens):
        if n == 0:
            assert (o[b] == 0).all()


@pytest.mark.parametrize("chunk", [0, 256])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Lmax,seqlens", SEQ_CASES)
def test_f32_small(chunk, d, Lmax, seqlens):
    px.parallax_attn_set_decode_chunk_keys(chunk)
    inp = _small(len(seqlens), 2, Lmax, d, seqlens, torch.float32, seed=7 * Lmax + d)
    o = _run(inp)
    ref = oracle.decode(inp.q, inp.rho, inp.k_cache, inp.v_cache, inp.seqlens)
    assert_f32(o, ref, f"Lmax={Lmax} d={d} chunk={chunk}")


def test_split_matches_unsplit():
    inp = _small(4, 4, 5000, 128, [5000, 4097, 3, 2500], torch.bfloat16, seed=11)
    o1 = _run(inp)
    px.parallax_attn_set_decode_chunk_keys(512)
    o2 = _run(inp)
    assert errors(o1, o2)[1] < 1e-5


def test_seqlen_out_of_range_is_clamped_and_flagged():
    inp = _small(3, 2, 300, 128, [300, 300, 5], torch.bfloat16, seed=12)
    ref = _run(inp)
    bad = configs.DecodeInputs(inp.q, inp.k_cache, inp.v_cache, inp.rho,
                               torch.tensor([301, -7, 5], dtype=torch.int32, device=DEV))
    o = torch.empty_like(ref)
    px.parallax_attn_decode(bad.q, bad.rho, bad.k_cache, bad.v_cache, bad.seqlens, o)
    bits = px.parallax_check_device_error()
    assert bits & px.DEVERR_SEQLEN_CLAMPED
    assert torch.equal(o[0], ref[0])      # 301 -> 300
    assert (o[1] == 0).all()              # -7 -> 0
    assert torch.equal(o[2], ref[2])


def test_invariants_bf16():
    inp = _small(2, 4, 3000, 128, [3000, 1234], torch.bfloat16, seed=13)
    # v on a 1/8 grid so that v + b is exact in bf16
    vq = ((inp.v_cache.float() * 8).round() / 8).bfloat16()
    inp = configs.DecodeInputs(inp.q, inp.k_cache, vq, inp.rho, inp.seqlens)
    o = _run(inp).double()
    b = torch.tensor([1.0, -0.5, 0.25, 2.0] * 32, device=DEV)
    sh = configs.DecodeInputs(inp.q, inp.k_cache, (vq.float() + b).bfloat16(), inp.rho,
                              inp.seqlens)
    assert torch.equal(sh.v_cache.float(), vq.float() + b)
    assert ((_run(sh).double() - o) - b).abs().max().item() < 2e-2
    z = configs.DecodeInputs(inp.q, inp.k_cache, inp.v_cache, torch.zeros_like(inp.rho),
                             inp.seqlens)
    assert errors(_run(z), _run(inp, rho=False))[1] < 1e-6


def test_uniform_workload_full_size():
    """B=64, H=16, d=128, 8192 keys each: 128 sampled heads against the oracle
    (explicit covariance on every 8th), and rho = NULL against torch SDPA on all heads."""
    inp = configs.decode_uniform_inputs(DEV)
    o = _run(inp)
    rng = np.random.default_rng(1)
    heads = [(int(b), int(h)) for b, h in zip(rng.integers(0, 64, 128), rng.integers(0, 16, 128))]
    got = np.stack([o[b, h].double().cpu().numpy() for b, h in heads])
    ref = np.concatenate([_ref_heads(inp, heads[i:i + 1], form="explicit" if i % 8 == 0 else
                                     "contracted") for i in range(len(heads))])
    rel, mx = assert_bf16(got, ref, "uniform decode sampled heads")
    print(f"uniform decode: rel-L2 {rel:.3e} max-abs {mx:.3e}")
    o0 = _run(inp, rho=False)
    sdpa = torch.nn.functional.scaled_dot_product_attention(
        inp.q.float().unsqueeze(2), inp.k_cache.float(), inp.v_cache.float()).squeeze(2)
    assert_bf16(o0, sdpa, "rho=NULL vs sdpa")


def _sweep_params():
    """Every cell of the decode sweep (batch x context, caches up to 64e9 bytes), plus the
    (256, 32768) cell whose cache is exactly 64 GiB, flagged by its id."""
    cells = configs.decode_sweep_cells()
    out = [pytest.param(B, L, id=f"B{B}-L{L}") for B, L in cells]
    out += [pytest.param(B, L, id=f"B{B}-L{L}-64GiB-boundary")
            for B, L in configs.decode_sweep_cells(include_boundary=True) if (B, L) not in cells]
    return out


@pytest.mark.parametrize("B,L", _sweep_params())
def test_sweep_cells_full_size(B, L):
    """One sweep cell at full size through the launch configuration the plan picks for it:
    the first and last head of the first and last sequence plus random heads (32 in all,
    fewer when the cell has fewer) against the oracle."""
    inp = configs.decode_sweep_inputs(B, L, DEV)
    o = _run(inp)
    assert torch.isfinite(o).all()
    rng = np.random.default_rng(B + L)
    heads = list(dict.fromkeys([(0, 0), (0, 15), (B - 1, 0), (B - 1, 15)]))
    while len(heads) < min(32, B * 16):
        bh = (int(rng.integers(B)), int(rng.integers(16)))
        if bh not in heads:
            heads.append(bh)
    got = np.stack([o[b, h].double().cpu().numpy() for b, h in heads])
    rel, mx = assert_bf16(got, _ref_heads(inp, heads), f"sweep cell B={B} L={L}")
    print(f"sweep cell B={B} L={L}: rel-L2 {rel:.3e} max-abs {mx:.3e} over {len(heads)} heads")
    del inp, o
    torch.cuda.empty_cache()


def test_ragged_workload_full_size():
    """B=512 sequences, lengths ~ U[128, 16384], cache allocated at Lmax = 16384."""
    inp = configs.decode_ragged_inputs(DEV)
    o = _run(inp)
    assert torch.isfinite(o).all()
    rng = np.random.default_rng(3)
    sl = inp.seqlens.cpu().numpy()
    order = np.argsort(sl)
    pick = list(order[:8]) + list(order[-8:]) + list(rng.integers(0, 512, 32))
    heads = [(int(b), int(rng.integers(16))) for b in pick]
    got = np.stack([o[b, h].double().cpu().numpy() for b, h in heads])
    assert_bf16(got, _ref_heads(inp, heads), "ragged decode sampled heads")
