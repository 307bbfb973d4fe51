"""Host-side checks of the C-ABI library: it loads without a GPU, exports every
symbol include/parallax_attn.h declares, and rejects bad arguments before it
touches CUDA.  No kernel is launched here."""
import ctypes
import os
import re

import pytest

import softmax_covariance_correction_pass_b300 as px
from softmax_covariance_correction_pass_b300 import build as pxbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "parallax_attn.h")


@pytest.fixture(scope="module")
def lib():
    pxbuild.build()
    return px.load_library()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(parallax_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("parallax_attn_prefill", "parallax_attn_decode", "parallax_attn_prefill_f32",
                     "parallax_attn_decode_f32", "parallax_last_error",
                     "parallax_check_device_error"):
        assert required in names


def _declaration(name):
    """The declaration of `name` in the header, comments and preprocessor lines stripped,
    whitespace collapsed."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    text = "\n".join(l for l in text.splitlines() if not l.lstrip().startswith("#"))
    for stmt in re.split(r"[;{}]", text):
        if re.search(r"\b" + name + r"\s*\(", stmt):
            return " ".join(stmt.split())
    raise AssertionError(f"{name} is not declared")


# The boundary's own signatures (argument names, order and types), as the hot-path scope
# defines them: prefill(q, rho, k, v, o, B, H, L, d, causal, scale, stream),
# decode(q, rho, k_cache, v_cache, seqlens, o, B, H, Lmax, d, stream) and a device-error
# check that takes the stream alone.
BOUNDARY = {
    "parallax_attn_prefill":
        "int parallax_attn_prefill(const void* q, const void* rho, const void* k, const void* v, "
        "void* o, int B, int H, int L, int d, int causal, float scale, cudaStream_t stream)",
    "parallax_attn_decode":
        "int parallax_attn_decode(const void* q, const void* rho, const void* k_cache, "
        "const void* v_cache, const int32_t* seqlens, void* o, int B, int H, int Lmax, int d, "
        "cudaStream_t stream)",
    "parallax_attn_prefill_f32":
        "int parallax_attn_prefill_f32(const void* q, const void* rho, const void* k, "
        "const void* v, void* o, int B, int H, int L, int d, int causal, float scale, "
        "cudaStream_t stream)",
    "parallax_attn_decode_f32":
        "int parallax_attn_decode_f32(const void* q, const void* rho, const void* k_cache, "
        "const void* v_cache, const int32_t* seqlens, void* o, int B, int H, int Lmax, int d, "
        "cudaStream_t stream)",
    "parallax_last_error": "const char* parallax_last_error(void)",
    "parallax_check_device_error": "int parallax_check_device_error(cudaStream_t stream)",
}


@pytest.mark.parametrize("name", sorted(BOUNDARY))
def test_boundary_signatures(name):
    assert _declaration(name) == BOUNDARY[name]


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_version(lib):
    assert px.parallax_version() >= 100


FAKE = 0x10000  # a 16-byte aligned non-null address; never dereferenced by the checks below


def _prefill(lib, q=FAKE, rho=None, k=FAKE, v=FAKE, o=FAKE, B=1, H=1, L=8, d=64, causal=1,
             scale=0.125, f32=False):
    fn = lib.parallax_attn_prefill_f32 if f32 else lib.parallax_attn_prefill
    vp = ctypes.c_void_p
    return fn(vp(q), vp(rho), vp(k), vp(v), vp(o), B, H, L, d, causal, ctypes.c_float(scale), None)


def _decode(lib, q=FAKE, rho=None, k=FAKE, v=FAKE, sl=FAKE, o=FAKE, B=1, H=1, Lmax=8, d=128,
            f32=False):
    fn = lib.parallax_attn_decode_f32 if f32 else lib.parallax_attn_decode
    vp = ctypes.c_void_p
    return fn(vp(q), vp(rho), vp(k), vp(v), vp(sl), vp(o), B, H, Lmax, d, None)


@pytest.mark.parametrize("f32", [False, True])
def test_prefill_argument_errors(lib, f32):
    E, U = px.PARALLAX_ERR_INVALID, px.PARALLAX_ERR_UNSUPPORTED
    assert _prefill(lib, q=None, f32=f32) == E
    assert _prefill(lib, k=None, f32=f32) == E
    assert _prefill(lib, v=None, f32=f32) == E
    assert _prefill(lib, o=None, f32=f32) == E
    assert _prefill(lib, B=0, f32=f32) == E
    assert _prefill(lib, H=-1, f32=f32) == E
    assert _prefill(lib, L=0, f32=f32) == E
    assert _prefill(lib, d=96, f32=f32) == U
    assert _prefill(lib, d=256, f32=f32) == U
    assert _prefill(lib, q=FAKE + 8, f32=f32) == E
    assert _prefill(lib, rho=FAKE + 4, f32=f32) == E
    assert _prefill(lib, causal=2, f32=f32) == E
    assert _prefill(lib, scale=float("nan"), f32=f32) == E
    assert _prefill(lib, scale=float("inf"), f32=f32) == E
    assert "causal" in px.last_error() or "scale" in px.last_error()


@pytest.mark.parametrize("f32", [False, True])
def test_decode_argument_errors(lib, f32):
    E, U = px.PARALLAX_ERR_INVALID, px.PARALLAX_ERR_UNSUPPORTED
    assert _decode(lib, q=None, f32=f32) == E
    assert _decode(lib, sl=None, f32=f32) == E
    assert _decode(lib, o=None, f32=f32) == E
    assert _decode(lib, Lmax=0, f32=f32) == E
    assert _decode(lib, B=0, f32=f32) == E
    assert _decode(lib, d=32, f32=f32) == U
    assert _decode(lib, k=FAKE + 2, f32=f32) == E


def test_last_error_is_thread_local(lib):
    import threading

    assert _prefill(lib, d=96) == px.PARALLAX_ERR_UNSUPPORTED
    seen = {}

    def other():
        seen["msg"] = px.last_error()

    t = threading.Thread(target=other)
    t.start()
    t.join()
    assert seen["msg"] == ""
    assert "d=96" in px.last_error()


def test_chunk_plan(lib):
    # split-KV plan with one query head per key/value head (148 SMs, 2 CTAs each, without a
    # device): the longest chunk of 256..4096 keys that leaves at least 0.85 items per CTA;
    # heads of at most 1024 keys are never split
    f = px.parallax_attn_decode_chunk_keys
    ctas = 2 * 148
    assert f(1, 16, 128, 128, 2) == 128                      # no split: whole cache
    assert f(8, 16, 1024, 128, 2) == 1024                    # short heads: no split
    assert f(2048, 16, 1024, 128, 2) == 1024                 # many heads: no split
    assert f(1, 16, 32768, 128, 2) == 2048                   # 16 heads x 16 chunks
    assert f(8, 16, 8192, 128, 2) == 4096                    # 128 heads x 2 chunks
    assert f(1, 16, 8192, 128, 2) == 512                     # 16 heads x 16 chunks
    assert f(64, 16, 8192, 128, 2) == 4096
    assert f(512, 16, 16384, 128, 2) == 4096                 # the 4096-key cap
    for B, L in ((1, 2048), (1, 100000), (4, 5000), (32, 2049), (3, 65536)):
        c = f(B, 16, L, 128, 2)
        items = B * 16 * -(-L // c)
        assert c == L or (256 <= c <= 4096 and c & (c - 1) == 0)
        assert items >= 0.85 * ctas or c == 256
        assert c >= 4096 or c == L or B * 16 * -(-L // (2 * c)) < 0.85 * ctas
    with pytest.raises(px.ParallaxError):
        f(0, 16, 128, 128, 2)
    with pytest.raises(px.ParallaxError):
        f(1, 16, 128, 128, 3)


def test_decode_plan_by_group_size(lib):
    """The plan of the plain, grouped-query and paged decode (host logic, 148 SMs without a
    device): plain decode as above, groups of 2 aim at ~8 items per SM, groups of 4 and 8 take
    the longest chunk leaving >= 1.7 items per SM, grouped heads on a paged cache stop at 2048
    keys; chunks stay within 256..4096 keys or cover the whole cache."""
    f = px.parallax_attn_decode_plan_keys
    sms = 148
    # one query head per key/value head: the same plan as parallax_attn_decode_chunk_keys
    for B, H, L in ((64, 16, 8192), (1, 16, 32768), (512, 16, 16384), (2048, 16, 1024)):
        assert f(B, H, H, L, 128) == px.parallax_attn_decode_chunk_keys(B, H, L, 128, 2)
    # B=64, H=16, 8192 keys: H_kv = 8 / 4 / 2 (groups of 2 / 4 / 8)
    assert f(64, 16, 8, 8192, 128) == 2048
    assert f(64, 16, 4, 8192, 128) == 4096
    assert f(64, 16, 2, 8192, 128) == 4096
    assert f(8, 16, 2, 8192, 128) == 512
    for B in (1, 4, 8, 16, 32, 64, 128):
        for Hkv in (4, 2):
            c = f(B, 16, Hkv, 8192, 128)
            items = B * Hkv * -(-8192 // c)
            assert 256 <= c <= 4096
            # the longest chunk that keeps >= 1.7 items per SM (or the shortest chunk)
            assert items >= 1.7 * sms or c == 256
            assert c == 4096 or B * Hkv * -(-8192 // (2 * c)) < 1.7 * sms
    # paged: grouped heads at most 2048 keys per item, one head per group as contiguous
    assert f(512, 16, 4, 16384, 128, 256) == 2048
    assert f(512, 16, 16, 16384, 128, 256) == f(512, 16, 16, 16384, 128, 0) == 4096
    assert f(1, 16, 2, 300, 128, 16) == 256
    # a forced chunk wins, also over the paged cap
    px.parallax_attn_set_decode_chunk_keys(4096)
    try:
        assert f(512, 16, 4, 16384, 128, 256) == 4096
        assert f(64, 16, 2, 8192, 64) == 4096
        assert f(1, 16, 2, 1000, 128) == 1000  # >= Lmax: no split
    finally:
        px.parallax_attn_set_decode_chunk_keys(0)
    for args, code in (((0, 16, 2, 128, 128), px.PARALLAX_ERR_INVALID),
                       ((1, 16, 3, 128, 128), px.PARALLAX_ERR_INVALID),
                       ((1, 16, 1, 128, 128), px.PARALLAX_ERR_UNSUPPORTED),   # groups of 16
                       ((1, 16, 2, 128, 96), px.PARALLAX_ERR_UNSUPPORTED),
                       ((1, 16, 2, 128, 128, 20), px.PARALLAX_ERR_UNSUPPORTED),
                       ((1, 16, 2, 128, 128, -16), px.PARALLAX_ERR_INVALID)):
        with pytest.raises(px.ParallaxError) as ei:
            f(*args)
        assert ei.value.code == code, args


def test_decode_plan_kernel(lib):
    """Which decode kernel a bf16 shape runs (host logic, 148 SMs and 2 CTAs each without a
    device): grouped heads always take the tensor-core kernel; one head per key/value head
    takes it when every CTA gets at least two items of 512 keys or more."""
    f = px.parallax_attn_decode_plan_kernel
    assert f(64, 16, 16, 8192, 128) == "decode_mma_kernel"     # 2048 items of 4096 keys
    assert f(2048, 16, 16, 1024, 128) == "decode_mma_kernel"   # unsplit 1024-key items
    assert f(8, 16, 16, 8192, 128) == "decode_kernel"          # 256 items: too few
    assert f(256, 16, 16, 128, 128) == "decode_kernel"         # 128-key items: too short
    assert f(1, 16, 16, 32768, 128) == "decode_kernel"
    for Hkv in (8, 4, 2):
        assert f(8, 16, Hkv, 1024, 128) == "decode_mma_kernel"
    # paged: the tensor-core kernel maps a stage (64 keys at d = 128, 128 at d = 64) to a page
    assert f(512, 16, 4, 16384, 128, 256) == "decode_mma_kernel"
    assert f(512, 16, 4, 16384, 128, 48) == "decode_kernel"
    assert f(512, 16, 4, 16384, 64, 64) == "decode_kernel"
    with pytest.raises(px.ParallaxError):
        f(1, 16, 3, 128, 128)


def test_forced_chunk_validation(lib):
    with pytest.raises(px.ParallaxError):
        px.parallax_attn_set_decode_chunk_keys(100)
    px.parallax_attn_set_decode_chunk_keys(512)
    assert px.parallax_attn_decode_chunk_keys(1, 1, 4096, 128, 2) == 512
    assert px.parallax_attn_decode_chunk_keys(1, 1, 300, 128, 2) == 300  # >= Lmax: no split
    px.parallax_attn_set_decode_chunk_keys(0)


def _proj(lib, x=FAKE, w=FAKE, q=FAKE, k=FAKE, v=FAKE, rho=FAKE, B=1, L=8, width=64, H=2, d=64):
    vp = ctypes.c_void_p
    return lib.parallax_attn_qkvr_projection(vp(x), vp(w), vp(q), vp(k), vp(v), vp(rho), B, L,
                                             width, H, d, None)


@pytest.mark.parametrize("kw,code", [
    (dict(x=0), px.PARALLAX_ERR_INVALID),
    (dict(w=0), px.PARALLAX_ERR_INVALID),
    (dict(v=0), px.PARALLAX_ERR_INVALID),
    (dict(B=0), px.PARALLAX_ERR_INVALID),
    (dict(L=-1), px.PARALLAX_ERR_INVALID),
    (dict(width=0), px.PARALLAX_ERR_INVALID),
    (dict(d=96), px.PARALLAX_ERR_UNSUPPORTED),
    (dict(H=1, d=64), px.PARALLAX_ERR_UNSUPPORTED),   # H*d = 64 is not a multiple of 128
    (dict(width=60), px.PARALLAX_ERR_UNSUPPORTED),
    (dict(q=FAKE + 8), px.PARALLAX_ERR_INVALID),
    (dict(rho=FAKE + 4), px.PARALLAX_ERR_INVALID),
])
def test_projection_validation(lib, kw, code):
    assert _proj(lib, **kw) == code
    assert px.last_error() != ""


def _gqa(lib, q=FAKE, rho=None, k=FAKE, v=FAKE, sl=FAKE, o=FAKE, B=1, H=8, Hkv=2, Lmax=64,
         d=128):
    vp = ctypes.c_void_p
    return lib.parallax_attn_decode_gqa(vp(q), vp(rho), vp(k), vp(v), vp(sl), vp(o), B, H, Hkv,
                                        Lmax, d, None)


@pytest.mark.parametrize("kw,code", [
    (dict(Hkv=3), px.PARALLAX_ERR_INVALID),         # 8 is not a multiple of 3
    (dict(Hkv=0), px.PARALLAX_ERR_INVALID),
    (dict(H=16, Hkv=1), px.PARALLAX_ERR_UNSUPPORTED),  # 16 query heads per key/value head
    (dict(H=6, Hkv=2), px.PARALLAX_ERR_UNSUPPORTED),   # group of 3
    (dict(sl=0), px.PARALLAX_ERR_INVALID),
    (dict(d=32), px.PARALLAX_ERR_UNSUPPORTED),
])
def test_gqa_validation(lib, kw, code):
    assert _gqa(lib, **kw) == code


def _paged(lib, q=FAKE, rho=None, k=FAKE, v=FAKE, bt=FAKE, sl=FAKE, o=FAKE, B=1, H=4, Hkv=4,
           P=16, max_pages=4, num_pages=8, d=128):
    vp = ctypes.c_void_p
    return lib.parallax_attn_decode_paged(vp(q), vp(rho), vp(k), vp(v), vp(bt), vp(sl), vp(o), B,
                                          H, Hkv, P, max_pages, num_pages, d, None)


@pytest.mark.parametrize("kw,code", [
    (dict(bt=0), px.PARALLAX_ERR_INVALID),
    (dict(P=0), px.PARALLAX_ERR_INVALID),
    (dict(P=24), px.PARALLAX_ERR_UNSUPPORTED),      # not a multiple of 16
    (dict(max_pages=0), px.PARALLAX_ERR_INVALID),
    (dict(num_pages=0), px.PARALLAX_ERR_INVALID),
    (dict(P=1 << 20, max_pages=1 << 12), px.PARALLAX_ERR_INVALID),  # Lmax beyond int
    (dict(Hkv=3), px.PARALLAX_ERR_INVALID),
    (dict(k=FAKE + 2), px.PARALLAX_ERR_INVALID),
])
def test_paged_validation(lib, kw, code):
    assert _paged(lib, **kw) == code


def _chunk(lib, q=FAKE, rho=None, k=FAKE, v=FAKE, kc=FAKE, vc=FAKE, cl=FAKE, o=FAKE, B=1, H=1,
           Lq=8, Lmax=16, d=64, scale=0.125):
    vp = ctypes.c_void_p
    return lib.parallax_attn_prefill_chunk(vp(q), vp(rho), vp(k), vp(v), vp(kc), vp(vc), vp(cl),
                                           vp(o), B, H, Lq, Lmax, d, ctypes.c_float(scale), None)


@pytest.mark.parametrize("kw,code", [
    (dict(kc=0), px.PARALLAX_ERR_INVALID),
    (dict(cl=0), px.PARALLAX_ERR_INVALID),
    (dict(Lmax=4), px.PARALLAX_ERR_INVALID),          # chunk longer than the cache
    (dict(Lq=0), px.PARALLAX_ERR_INVALID),
    (dict(d=80), px.PARALLAX_ERR_UNSUPPORTED),
    (dict(vc=FAKE + 8), px.PARALLAX_ERR_INVALID),
    (dict(scale=float("inf")), px.PARALLAX_ERR_INVALID),
])
def test_chunk_validation(lib, kw, code):
    assert _chunk(lib, **kw) == code


def _lla(lib, q=FAKE, k=FAKE, v=FAKE, sl=FAKE, o=FAKE, rho=FAKE, B=1, H=2, Lmax=64, d=128,
         iters=0):
    vp = ctypes.c_void_p
    return lib.parallax_lla_decode(vp(q), vp(k), vp(v), vp(sl), vp(o), vp(rho), B, H, Lmax, d,
                                   iters, None)


@pytest.mark.parametrize("kw,code", [
    (dict(sl=0), px.PARALLAX_ERR_INVALID),
    (dict(rho=0), px.PARALLAX_ERR_INVALID),
    (dict(iters=-1), px.PARALLAX_ERR_INVALID),
    (dict(d=96), px.PARALLAX_ERR_UNSUPPORTED),
    (dict(B=0), px.PARALLAX_ERR_INVALID),
    (dict(v=FAKE + 4), px.PARALLAX_ERR_INVALID),   # not 16-byte aligned
])
def test_lla_validation(lib, kw, code):
    assert _lla(lib, **kw) == code
    assert px.last_error() != ""


def _train(lib, q=FAKE, rho=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, rbar=FAKE, mu=FAKE, B=1, H=1,
           L=64, d=64, causal=1, scale=0.125):
    vp = ctypes.c_void_p
    return lib.parallax_attn_prefill_train(vp(q), vp(rho), vp(k), vp(v), vp(o), vp(lse), vp(rbar),
                                           vp(mu), B, H, L, d, causal, ctypes.c_float(scale), None)


@pytest.mark.parametrize("kw,code", [
    (dict(lse=0), px.PARALLAX_ERR_INVALID),
    (dict(mu=0), px.PARALLAX_ERR_INVALID),
    (dict(rbar=FAKE + 4), px.PARALLAX_ERR_INVALID),
    (dict(causal=2), px.PARALLAX_ERR_INVALID),
    (dict(scale=float("nan")), px.PARALLAX_ERR_INVALID),
    (dict(d=48), px.PARALLAX_ERR_UNSUPPORTED),
])
def test_prefill_train_validation(lib, kw, code):
    assert _train(lib, **kw) == code


def _bwd(lib, dout=FAKE, dq=FAKE, drho=FAKE, dk=FAKE, dv=FAKE, causal=1, scale=0.125, L=64, d=64):
    vp = ctypes.c_void_p
    f = FAKE
    return lib.parallax_attn_prefill_backward(vp(f), vp(f), vp(f), vp(f), vp(f), vp(f), vp(f),
                                              vp(f), vp(dout), vp(dq), vp(drho), vp(dk), vp(dv),
                                              1, 1, L, d, causal, ctypes.c_float(scale), None)


@pytest.mark.parametrize("kw,code", [
    (dict(dout=0), px.PARALLAX_ERR_INVALID),
    (dict(dk=0), px.PARALLAX_ERR_INVALID),
    (dict(dv=FAKE + 8), px.PARALLAX_ERR_INVALID),
    (dict(causal=-1), px.PARALLAX_ERR_INVALID),
    (dict(scale=float("inf")), px.PARALLAX_ERR_INVALID),
    (dict(L=0), px.PARALLAX_ERR_INVALID),
    (dict(d=256), px.PARALLAX_ERR_UNSUPPORTED),
])
def test_prefill_backward_validation(lib, kw, code):
    assert _bwd(lib, **kw) == code


def test_no_cpu_path(lib, monkeypatch, tmp_path):
    """Nothing computes on the CPU: host tensors are refused, and without the CUDA library
    every call raises."""
    import torch

    x = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        px.parallax_attn_prefill(x, None, x, x)
    monkeypatch.setattr(px, "LIB_PATH", str(tmp_path / "libparallax_attn.so"))
    monkeypatch.setattr(px, "_lib", None)
    with pytest.raises(ImportError, match="no CPU fallback"):
        px.parallax_attn_decode_plan_keys(1, 1, 1, 128, 64)
    with pytest.raises(ImportError):
        px.parallax_version()


def test_binding_refuses_tensors_on_another_device(monkeypatch):
    """The library launches on the current device; the binding refuses a tensor or a stream of
    another device (emulated on the CPU: a tensor subclass that reports a CUDA device)."""
    import torch

    class FakeCuda(torch.Tensor):
        @property
        def is_cuda(self):
            return True

        def get_device(self):
            return self.fake_index

    def on(index):
        t = torch.zeros(2, 3).as_subclass(FakeCuda)
        t.fake_index = index
        return t

    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    px._need(on(0), "q", torch.float32, (2, 3))          # the current device: accepted
    with pytest.raises(ValueError, match="cuda:1.*current device cuda:0"):
        px._need(on(1), "q", torch.float32, (2, 3))

    class FakeStream:
        device = torch.device("cuda", 1)
        cuda_stream = 0

    with pytest.raises(ValueError, match="stream belongs to cuda:1"):
        px._stream(FakeStream())
    FakeStream.device = torch.device("cuda", 0)
    assert px._stream(FakeStream()).value is None        # the null stream handle
