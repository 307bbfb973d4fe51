"""Guard canaries around every output and workspace, on odd shapes.

compute-sanitizer is not available here, so overruns are caught the plain way: each
output tensor the caller passes is the middle of a larger buffer whose head and tail
(guard bands) hold a NaN bit pattern, and the interior is filled with the same pattern
before the call (an element the call should write but does not stays NaN).  After every
call the guard bands must be bit-for-bit unchanged, the interior finite, and the guard
bands around the library's own workspaces intact.  Shapes are the small odd ones where
tile tails and split-KV chunk tails sit: L = 1, 3, 127, 129; sequence lengths 1 and
lengths that are not a multiple of the chunk.
"""
import ctypes
import math

import pytest
import torch

import softmax_covariance_correction_pass_b300 as px
from softmax_covariance_correction_pass_b300 import configs

pytestmark = pytest.mark.gpu
DEV = "cuda"
GUARD = 1024  # elements on each side (4 KB of fp32, 2 KB of bf16: keeps 16-byte alignment)
PATTERN = {torch.float32: (torch.int32, 0x7FA5A5A5), torch.bfloat16: (torch.int16, 0x7FA5)}


class Guarded:
    """A tensor of `shape` inside a buffer with GUARD sentinel elements before and after."""

    def __init__(self, shape, dtype, fill_interior=True, init=None):
        n = math.prod(shape)
        itype, bits = PATTERN[dtype]
        self.raw = torch.full((n + 2 * GUARD,), bits, dtype=itype, device=DEV)
        self.buf = self.raw.view(dtype)
        self.t = self.buf[GUARD:GUARD + n].view(shape)
        if init is not None:
            self.t.copy_(init)
        elif not fill_interior:
            self.t.zero_()
        self.bits = bits

    def guards_intact(self):
        return bool((self.raw[:GUARD] == self.bits).all() and (self.raw[-GUARD:] == self.bits).all())

    def check(self, what, finite=True):
        torch.cuda.synchronize()
        assert self.guards_intact(), f"{what}: a guard band was overwritten"
        if finite:
            assert torch.isfinite(self.t.float()).all(), f"{what}: unwritten or non-finite element"


@pytest.fixture(autouse=True)
def _clean():
    px.parallax_attn_set_decode_chunk_keys(0)
    yield
    px.parallax_attn_set_decode_chunk_keys(0)
    assert px.parallax_check_device_error() == 0
    assert px.parallax_workspace_guards_intact()


ODD_L = [1, 3, 127, 129]


@pytest.mark.parametrize("L", ODD_L)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("rho", [True, False])
def test_prefill_bf16(L, d, causal, rho):
    inp = configs.prefill_inputs(2, 3, L, d, seed=L + d, device=DEV, dtype=torch.bfloat16)
    o = Guarded((2, 3, L, d), torch.float32)
    px.parallax_attn_prefill(inp.q, inp.rho if rho else None, inp.k, inp.v, o.t, causal=causal,
                             scale=inp.scale)
    o.check(f"prefill L={L} d={d}")


@pytest.mark.parametrize("L", ODD_L)
def test_prefill_f32(L):
    inp = configs.prefill_inputs(1, 2, L, 64, seed=L, device=DEV, dtype=torch.float32)
    o = Guarded((1, 2, L, 64), torch.float32)
    px.parallax_attn_prefill(inp.q, inp.rho, inp.k, inp.v, o.t, causal=True, scale=inp.scale)
    o.check(f"prefill f32 L={L}")


@pytest.mark.parametrize("L", ODD_L)
def test_prefill_train_and_backward(L):
    B, H, d = 1, 2, 128
    inp = configs.prefill_inputs(B, H, L, d, seed=3 * L, device=DEV, dtype=torch.bfloat16)
    lib = px.load_library()
    vp = ctypes.c_void_p
    o, mu = Guarded((B, H, L, d), torch.float32), Guarded((B, H, L, d), torch.float32)
    lse, rbar = Guarded((B, H, L), torch.float32), Guarded((B, H, L), torch.float32)
    stream = vp(torch.cuda.current_stream().cuda_stream)
    rc = lib.parallax_attn_prefill_train(
        vp(inp.q.data_ptr()), vp(inp.rho.data_ptr()), vp(inp.k.data_ptr()), vp(inp.v.data_ptr()),
        vp(o.t.data_ptr()), vp(lse.t.data_ptr()), vp(rbar.t.data_ptr()), vp(mu.t.data_ptr()),
        B, H, L, d, 1, ctypes.c_float(inp.scale), stream)
    assert rc == px.PARALLAX_OK, px.last_error()
    for name, g in (("o", o), ("mu", mu), ("lse", lse), ("rbar", rbar)):
        g.check(f"train {name} L={L}")
    g = torch.Generator(device=DEV).manual_seed(L)
    dout = torch.randn((B, H, L, d), generator=g, device=DEV).to(torch.bfloat16)
    grads = [Guarded((B, H, L, d), torch.float32) for _ in range(4)]
    rc = lib.parallax_attn_prefill_backward(
        vp(inp.q.data_ptr()), vp(inp.rho.data_ptr()), vp(inp.k.data_ptr()), vp(inp.v.data_ptr()),
        vp(o.t.data_ptr()), vp(mu.t.data_ptr()), vp(lse.t.data_ptr()), vp(rbar.t.data_ptr()),
        vp(dout.data_ptr()), *[vp(x.t.data_ptr()) for x in grads], B, H, L, d, 1,
        ctypes.c_float(inp.scale), stream)
    assert rc == px.PARALLAX_OK, px.last_error()
    for name, x in zip(("dq", "drho", "dk", "dv"), grads):
        x.check(f"backward {name} L={L}")


@pytest.mark.parametrize("Lq,off", [(1, 0), (3, 5), (129, 127), (127, 300)])
def test_prefill_chunk(Lq, off):
    B, H, d, Lmax = 2, 2, 128, 512
    inp = configs.prefill_inputs(B, H, Lq, d, seed=Lq + off, device=DEV, dtype=torch.bfloat16)
    base = configs.prefill_inputs(B, H, Lmax, d, seed=99, device=DEV, dtype=torch.bfloat16)
    kc = Guarded((B, H, Lmax, d), torch.bfloat16, init=base.k)
    vc = Guarded((B, H, Lmax, d), torch.bfloat16, init=base.v)
    o = Guarded((B, H, Lq, d), torch.float32)
    cl = torch.tensor([off, off // 2], dtype=torch.int32, device=DEV)
    px.parallax_attn_prefill_chunk(inp.q, inp.rho, inp.k, inp.v, kc.t, vc.t, cl, o.t)
    o.check(f"chunk o Lq={Lq}")
    kc.check("k cache")
    vc.check("v cache")


SEQS = [[1], [1, 257, 1000], [255, 0, 513]]


@pytest.mark.parametrize("seqlens", SEQS)
@pytest.mark.parametrize("chunk", [0, 256])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode(seqlens, chunk, dtype):
    px.parallax_attn_set_decode_chunk_keys(chunk)
    B, H, d = len(seqlens), 3, 128
    Lmax = max(seqlens) + 5
    inp = configs.decode_inputs(B, H, d, seqlens, Lmax, seed=B + chunk, device=DEV, dtype=dtype)
    o = Guarded((B, H, d), torch.float32)
    px.parallax_attn_decode(inp.q, inp.rho, inp.k_cache, inp.v_cache, inp.seqlens, o.t)
    o.check(f"decode {seqlens} chunk={chunk}")
    if dtype == torch.bfloat16:
        o2 = Guarded((B, H, d), torch.float32)
        px.parallax_attn_decode_noalloc(inp.q, inp.rho, inp.k_cache, inp.v_cache, inp.seqlens,
                                        o2.t)
        o2.check("decode no-alloc")


@pytest.mark.parametrize("Hkv", [1, 2, 4])
@pytest.mark.parametrize("chunk", [0, 256])
def test_decode_gqa_and_paged(Hkv, chunk):
    px.parallax_attn_set_decode_chunk_keys(chunk)
    B, H, d, P = 3, 8, 128, 64
    sl = [1, 257, 1000]
    Lmax = 1024
    inp = configs.decode_gqa_inputs(B, H, Hkv, d, sl, Lmax, seed=Hkv, device=DEV)
    o = Guarded((B, H, d), torch.float32)
    px.parallax_attn_decode_gqa(inp.q, inp.rho, inp.k_cache, inp.v_cache, inp.seqlens, o.t)
    o.check(f"gqa H_kv={Hkv}")
    pin, bt = configs.paged_decode_inputs(B, H, Hkv, d, sl, P, seed=Hkv + 1, device=DEV)
    o2 = Guarded((B, H, d), torch.float32)
    px.parallax_attn_decode_paged(pin.q, pin.rho, pin.k_cache, pin.v_cache, bt, pin.seqlens, o2.t)
    o2.check(f"paged H_kv={Hkv}")


@pytest.mark.parametrize("seqlens", [[300, 129], [1000, 257]])
def test_lla_decode(seqlens):
    B, H, d = len(seqlens), 2, 64
    inp = configs.decode_inputs(B, H, d, seqlens, max(seqlens) + 3, seed=5, device=DEV)
    o, rho = Guarded((B, H, d), torch.float32), Guarded((B, H, d), torch.float32)
    px.parallax_lla_decode(inp.q, inp.k_cache, inp.v_cache, inp.seqlens, o.t, rho.t)
    o.check("lla o")
    rho.check("lla rho")


@pytest.mark.parametrize("L", [1, 3, 129])
def test_projection(L):
    B, width, H, d = 2, 256, 2, 64
    x, w = configs.projection_inputs(B, L, width, H, d, 4, seed=L, device=DEV)
    outs = [Guarded((B, H, L, d), torch.bfloat16) for _ in range(4)]
    px.parallax_attn_qkvr_projection(x, w, H, d, *[g.t for g in outs])
    for name, g in zip("qkvr", outs):
        g.check(f"projection {name} L={L}")
