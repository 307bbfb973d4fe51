"""Parallax attention forward hot path for B300 (sm_103a).

Thin ctypes binding over ``libparallax_attn.so`` (C ABI declared in
``include/parallax_attn.h``).  This module only marshals arguments: every step
of the computation runs in the library's CUDA kernels.  There is no CPU path:
the library is loaded on the first call (so that the build step can import this
package before the library exists), and if it is missing that call raises
ImportError.

Functions carry the C names (``parallax_attn_prefill``, ...), with short
aliases ``prefill`` / ``decode``.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# PARALLAX_LIBRARY=debug selects the build with device-side bounds checks
# (`python -m softmax_covariance_correction_pass_b300.build --debug`)
LIB_PATH = os.path.join(_HERE, "libparallax_attn_debug.so"
                        if os.environ.get("PARALLAX_LIBRARY") == "debug" else "libparallax_attn.so")

PARALLAX_OK = 0
PARALLAX_ERR_INVALID = -1
PARALLAX_ERR_UNSUPPORTED = -2
PARALLAX_ERR_CUDA = -3
PARALLAX_ERR_DEVICE = -4
DEVERR_SEQLEN_CLAMPED = 0x1
DEVERR_WAIT_TIMEOUT = 0x2
DEVERR_PAGE_OUT_OF_RANGE = 0x4
DEVERR_SMEM_MISALIGNED = 0x8
DEVERR_BOUNDS = 0x10

_lib = None


class ParallaxError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"parallax error {code}: {msg}")
        self.code = code


def load_library() -> ctypes.CDLL:
    """Load the in-tree CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with "
            "`python -m softmax_covariance_correction_pass_b300.build` (add --debug for the "
            "checked build; no CPU fallback exists)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.parallax_attn_prefill.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp]
    lib.parallax_attn_prefill_f32.argtypes = lib.parallax_attn_prefill.argtypes
    lib.parallax_attn_decode.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp]
    lib.parallax_attn_decode_f32.argtypes = lib.parallax_attn_decode.argtypes
    lib.parallax_attn_prefill_train.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                                i32, f32, vp]
    lib.parallax_attn_prefill_backward.argtypes = [vp] * 13 + [i32] * 5 + [f32, vp]
    lib.parallax_lla_decode.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp]
    lib.parallax_attn_prefill_chunk.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32,
                                                i32, i32, f32, vp]
    lib.parallax_attn_decode_gqa.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp]
    lib.parallax_attn_decode_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                               i32, i32, i32, vp]
    lib.parallax_attn_decode_chunk_keys.argtypes = [i32, i32, i32, i32, i32]
    lib.parallax_attn_decode_plan_keys.argtypes = [i32] * 6
    lib.parallax_attn_decode_plan_kernel.argtypes = [i32] * 6
    lib.parallax_attn_qkvr_projection.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                                  vp]
    lib.parallax_attn_set_decode_chunk_keys.argtypes = [i32]
    lib.parallax_attn_workspace_bytes.restype = ctypes.c_size_t
    lib.parallax_last_error.restype = ctypes.c_char_p
    lib.parallax_check_device_error.argtypes = [vp]
    lib.parallax_last_device_error_bits.argtypes = []
    lib.parallax_last_device_error_bits.restype = ctypes.c_uint
    lib.parallax_selftest_wait_timeout.argtypes = [i32, ctypes.c_uint, vp]
    lib.parallax_workspace_guards_intact.argtypes = []
    for name in ("parallax_attn_prefill", "parallax_attn_prefill_f32", "parallax_attn_decode",
                 "parallax_attn_qkvr_projection", "parallax_attn_decode_gqa",
                 "parallax_attn_decode_paged", "parallax_attn_prefill_chunk",
                 "parallax_attn_prefill_train", "parallax_attn_prefill_backward",
                 "parallax_lla_decode",
                 "parallax_attn_decode_f32", "parallax_attn_decode_chunk_keys",
                 "parallax_attn_decode_plan_keys", "parallax_attn_decode_plan_kernel",
                 "parallax_attn_set_decode_chunk_keys", "parallax_attn_release_workspace",
                 "parallax_check_device_error", "parallax_version",
                 "parallax_selftest_wait_timeout", "parallax_workspace_guards_intact",
                 "parallax_debug_checks"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def last_error() -> str:
    return load_library().parallax_last_error().decode()


def _check(rc: int):
    if rc != PARALLAX_OK:
        raise ParallaxError(rc, last_error())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    elif isinstance(getattr(stream, "device", None), torch.device):
        dev = torch.cuda.current_device()
        if stream.device.index != dev:
            raise ValueError(f"stream belongs to {stream.device}, but the library launches on "
                             f"the current device cuda:{dev}")
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t, name, dtype, shape):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    dev = torch.cuda.current_device()
    if t.get_device() != dev:
        # the library launches on the current device; a pointer into another device's
        # memory would be dereferenced there
        raise ValueError(f"{name} is on cuda:{t.get_device()}, but the library launches on the "
                         f"current device cuda:{dev} (use torch.cuda.device(...))")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def parallax_attn_prefill(q, rho, k, v, o=None, causal: bool = True, scale: float | None = None,
                          stream=None):
    """Prefill over [B, H, L, d] tensors (bf16 -> tensor-core kernel, fp32 -> fp32 kernel).

    ``rho=None`` is the W_R = 0 path (plain softmax attention).  Returns ``o``
    (fp32 [B, H, L, d]).
    """
    B, H, L, d = q.shape
    dt = q.dtype
    if dt not in (torch.bfloat16, torch.float32):
        raise ValueError("q must be bf16 or fp32")
    for name, t in (("q", q), ("k", k), ("v", v)) + ((("rho", rho),) if rho is not None else ()):
        _need(t, name, dt, (B, H, L, d))
    if o is None:
        o = torch.empty((B, H, L, d), dtype=torch.float32, device=q.device)
    _need(o, "o", torch.float32, (B, H, L, d))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    fn = load_library().parallax_attn_prefill if dt == torch.bfloat16 else \
        load_library().parallax_attn_prefill_f32
    _check(fn(_ptr(q), _ptr(rho), _ptr(k), _ptr(v), _ptr(o), B, H, L, d, 1 if causal else 0,
              float(scale), _stream(stream)))
    return o


def parallax_attn_prefill_train(q, rho, k, v, causal: bool = True, scale: float | None = None,
                                stream=None):
    """Training forward (bf16 [B, H, L, d] inputs): returns (o, lse, rbar, mu_v), fp32;
    lse/rbar [B, H, L] and mu_v [B, H, L, d] are what the backward pass needs."""
    B, H, L, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v)) + ((("rho", rho),) if rho is not None else ()):
        _need(t, name, torch.bfloat16, (B, H, L, d))
    o = torch.empty((B, H, L, d), dtype=torch.float32, device=q.device)
    mu = torch.empty_like(o)
    lse = torch.empty((B, H, L), dtype=torch.float32, device=q.device)
    rbar = torch.empty_like(lse)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _check(load_library().parallax_attn_prefill_train(
        _ptr(q), _ptr(rho), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(rbar), _ptr(mu), B, H, L,
        d, 1 if causal else 0, float(scale), _stream(stream)))
    return o, lse, rbar, mu


def parallax_attn_prefill_backward(q, rho, k, v, o, mu_v, lse, rbar, dout, causal: bool = True,
                                   scale: float | None = None, stream=None):
    """Gradients (dq, drho, dk, dv), fp32 [B, H, L, d], of sum(dout * o) for the prefill;
    o, mu_v, lse, rbar come from parallax_attn_prefill_train, dout is bf16.  drho is
    None when rho is None."""
    B, H, L, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v), ("dout", dout)) + \
            ((("rho", rho),) if rho is not None else ()):
        _need(t, name, torch.bfloat16, (B, H, L, d))
    _need(o, "o", torch.float32, (B, H, L, d))
    _need(mu_v, "mu_v", torch.float32, (B, H, L, d))
    _need(lse, "lse", torch.float32, (B, H, L))
    _need(rbar, "rbar", torch.float32, (B, H, L))
    dq, dk, dv = (torch.empty((B, H, L, d), dtype=torch.float32, device=q.device)
                  for _ in range(3))
    drho = None if rho is None else torch.empty_like(dq)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _check(load_library().parallax_attn_prefill_backward(
        _ptr(q), _ptr(rho), _ptr(k), _ptr(v), _ptr(o), _ptr(mu_v), _ptr(lse), _ptr(rbar),
        _ptr(dout), _ptr(dq), _ptr(drho), _ptr(dk), _ptr(dv), B, H, L, d, 1 if causal else 0,
        float(scale), _stream(stream)))
    return dq, drho, dk, dv


def parallax_attn_prefill_chunk(q, rho, k_new, v_new, k_cache, v_cache, cache_lens, o=None,
                                scale: float | None = None, stream=None):
    """Causal prefill of a chunk that continues cached sequences (bf16).

    q, rho, k_new, v_new [B, H, Lq, d]; caches [B, H, Lmax, d] holding cache_lens[b]
    tokens (int32 [B] on the device).  Writes the chunk's keys and values into the
    caches, then returns o (fp32 [B, H, Lq, d]): chunk token i attends to the cached
    tokens and to chunk tokens 0..i.  cache_lens is not advanced.
    """
    B, H, Lq, d = q.shape
    Lmax = k_cache.shape[2]
    for name, t in (("q", q), ("k_new", k_new), ("v_new", v_new)) + \
            ((("rho", rho),) if rho is not None else ()):
        _need(t, name, torch.bfloat16, (B, H, Lq, d))
    _need(k_cache, "k_cache", torch.bfloat16, (B, H, Lmax, d))
    _need(v_cache, "v_cache", torch.bfloat16, (B, H, Lmax, d))
    _need(cache_lens, "cache_lens", torch.int32, (B,))
    if o is None:
        o = torch.empty((B, H, Lq, d), dtype=torch.float32, device=q.device)
    _need(o, "o", torch.float32, (B, H, Lq, d))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _check(load_library().parallax_attn_prefill_chunk(
        _ptr(q), _ptr(rho), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
        _ptr(cache_lens), _ptr(o), B, H, Lq, Lmax, d, float(scale), _stream(stream)))
    return o


def parallax_attn_decode(q, rho, k_cache, v_cache, seqlens, o=None, stream=None):
    """Single-token decode; q/rho [B, H, d], caches [B, H, Lmax, d], seqlens int32 [B].

    Returns ``o`` (fp32 [B, H, d]).  The softmax scale is 1/sqrt(d).
    """
    B, H, Lmax, d = k_cache.shape
    dt = k_cache.dtype
    if dt not in (torch.bfloat16, torch.float32):
        raise ValueError("caches must be bf16 or fp32")
    _need(q, "q", dt, (B, H, d))
    if rho is not None:
        _need(rho, "rho", dt, (B, H, d))
    _need(k_cache, "k_cache", dt, (B, H, Lmax, d))
    _need(v_cache, "v_cache", dt, (B, H, Lmax, d))
    _need(seqlens, "seqlens", torch.int32, (B,))
    if o is None:
        o = torch.empty((B, H, d), dtype=torch.float32, device=q.device)
    _need(o, "o", torch.float32, (B, H, d))
    fn = load_library().parallax_attn_decode if dt == torch.bfloat16 else \
        load_library().parallax_attn_decode_f32
    _check(fn(_ptr(q), _ptr(rho), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens), _ptr(o), B, H,
              Lmax, d, _stream(stream)))
    return o


def parallax_attn_decode_gqa(q, rho, k_cache, v_cache, seqlens, o=None, stream=None):
    """Decode with shared key/value heads: q/rho bf16 [B, H, d], caches bf16
    [B, H_kv, Lmax, d] (H / H_kv in {1, 2, 4, 8}), seqlens int32 [B].  Returns o fp32
    [B, H, d]; query head h reads key/value head h // (H // H_kv)."""
    B, Hkv, Lmax, d = k_cache.shape
    H = q.shape[1]
    _need(q, "q", torch.bfloat16, (B, H, d))
    if rho is not None:
        _need(rho, "rho", torch.bfloat16, (B, H, d))
    _need(k_cache, "k_cache", torch.bfloat16, (B, Hkv, Lmax, d))
    _need(v_cache, "v_cache", torch.bfloat16, (B, Hkv, Lmax, d))
    _need(seqlens, "seqlens", torch.int32, (B,))
    if o is None:
        o = torch.empty((B, H, d), dtype=torch.float32, device=q.device)
    _need(o, "o", torch.float32, (B, H, d))
    _check(load_library().parallax_attn_decode_gqa(
        _ptr(q), _ptr(rho), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens), _ptr(o), B, H, Hkv, Lmax,
        d, _stream(stream)))
    return o


def parallax_attn_decode_paged(q, rho, k_pages, v_pages, block_table, seqlens, o=None,
                               stream=None):
    """Decode against a paged cache: pages bf16 [num_pages, H_kv, page_size, d], block_table
    int32 [B, max_pages] (key t of sequence b is row t % page_size of page
    block_table[b, t // page_size]), seqlens int32 [B].  Returns o fp32 [B, H, d]."""
    num_pages, Hkv, P, d = k_pages.shape
    B, H = q.shape[0], q.shape[1]
    max_pages = block_table.shape[1]
    _need(q, "q", torch.bfloat16, (B, H, d))
    if rho is not None:
        _need(rho, "rho", torch.bfloat16, (B, H, d))
    _need(k_pages, "k_pages", torch.bfloat16, (num_pages, Hkv, P, d))
    _need(v_pages, "v_pages", torch.bfloat16, (num_pages, Hkv, P, d))
    _need(block_table, "block_table", torch.int32, (B, max_pages))
    _need(seqlens, "seqlens", torch.int32, (B,))
    if o is None:
        o = torch.empty((B, H, d), dtype=torch.float32, device=q.device)
    _need(o, "o", torch.float32, (B, H, d))
    _check(load_library().parallax_attn_decode_paged(
        _ptr(q), _ptr(rho), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(seqlens),
        _ptr(o), B, H, Hkv, P, max_pages, num_pages, d, _stream(stream)))
    return o


def parallax_lla_decode(q, k_cache, v_cache, seqlens, o=None, rho=None, cg_iters: int = 0,
                        stream=None):
    """Exact local linear attention decode (the per-query solve the Parallax probe replaces):
    q bf16 [B, H, d], caches bf16 [B, H, Lmax, d], seqlens int32 [B].  Returns (o, rho),
    fp32 [B, H, d]: rho = Sigma_kk^-1 (mu_k - q) by conjugate gradient (cg_iters steps,
    0 = d), o = mu_v - C^T rho (the Parallax output with that probe), one pass over K and V."""
    B, H, Lmax, d = k_cache.shape
    _need(q, "q", torch.bfloat16, (B, H, d))
    _need(k_cache, "k_cache", torch.bfloat16, (B, H, Lmax, d))
    _need(v_cache, "v_cache", torch.bfloat16, (B, H, Lmax, d))
    _need(seqlens, "seqlens", torch.int32, (B,))
    if o is None:
        o = torch.empty((B, H, d), dtype=torch.float32, device=q.device)
    if rho is None:
        rho = torch.empty((B, H, d), dtype=torch.float32, device=q.device)
    _need(o, "o", torch.float32, (B, H, d))
    _need(rho, "rho", torch.float32, (B, H, d))
    _check(load_library().parallax_lla_decode(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens), _ptr(o), _ptr(rho), B, H, Lmax, d,
        int(cg_iters), _stream(stream)))
    return o, rho


def parallax_attn_decode_noalloc(q, rho, k_cache, v_cache, seqlens, o, stream=None):
    """parallax_attn_decode (bf16) with the split-KV partials in the library's fixed
    device array: the call allocates nothing (``o`` must be supplied)."""
    B, H, Lmax, d = k_cache.shape
    _need(q, "q", torch.bfloat16, (B, H, d))
    if rho is not None:
        _need(rho, "rho", torch.bfloat16, (B, H, d))
    _need(k_cache, "k_cache", torch.bfloat16, (B, H, Lmax, d))
    _need(v_cache, "v_cache", torch.bfloat16, (B, H, Lmax, d))
    _need(seqlens, "seqlens", torch.int32, (B,))
    _need(o, "o", torch.float32, (B, H, d))
    lib = load_library()
    fn = lib.parallax_attn_decode_noalloc
    fn.argtypes = lib.parallax_attn_decode.argtypes
    fn.restype = ctypes.c_int
    _check(fn(_ptr(q), _ptr(rho), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens), _ptr(o), B, H,
              Lmax, d, _stream(stream)))
    return o


def parallax_attn_qkvr_projection(x, w, H: int, d: int, q=None, k=None, v=None, rho=None,
                                  with_rho: bool = True, stream=None):
    """q, k, v and the probe rho = W_R x of a layer in one tensor-core product.

    ``x`` bf16 [B, L, width]; ``w`` bf16 [n_out*H*d, width], the stacked weight
    W_q; W_k; W_v; W_R (rows = output features), n_out = 4, or 3 with
    ``with_rho=False`` (W_R = 0: no probe is computed).  Returns
    ``(q, k, v, rho)`` as bf16 [B, H, L, d] (``rho`` is None without the probe).
    """
    B, L, width = x.shape
    n_out = 4 if with_rho else 3
    _need(x, "x", torch.bfloat16, (B, L, width))
    _need(w, "w", torch.bfloat16, (n_out * H * d, width))
    outs = []
    for name, t in (("q", q), ("k", k), ("v", v)) + ((("rho", rho),) if with_rho else ()):
        if t is None:
            t = torch.empty((B, H, L, d), dtype=torch.bfloat16, device=x.device)
        _need(t, name, torch.bfloat16, (B, H, L, d))
        outs.append(t)
    if not with_rho:
        outs.append(None)
    lib = load_library()
    _check(lib.parallax_attn_qkvr_projection(_ptr(x), _ptr(w), *[_ptr(t) for t in outs], B, L,
                                             width, H, d, _stream(stream)))
    return tuple(outs)


def parallax_attn_decode_chunk_keys(B: int, H: int, Lmax: int, d: int, elem_bytes: int) -> int:
    rc = load_library().parallax_attn_decode_chunk_keys(B, H, Lmax, d, elem_bytes)
    if rc < 0:
        raise ParallaxError(rc, last_error())
    return rc


def parallax_attn_decode_plan_keys(B: int, H: int, H_kv: int, Lmax: int, d: int,
                                   page_size: int = 0) -> int:
    """Keys per work item of the decode plan (plain, grouped-query or paged decode)."""
    rc = load_library().parallax_attn_decode_plan_keys(B, H, H_kv, Lmax, d, page_size)
    if rc < 0:
        raise ParallaxError(rc, last_error())
    return rc


def parallax_attn_decode_plan_kernel(B: int, H: int, H_kv: int, Lmax: int, d: int,
                                     page_size: int = 0) -> str:
    """The decode kernel the bf16 entry points run for this shape: "decode_mma_kernel" (tensor
    cores) or "decode_kernel" (SIMT).  Host-only."""
    rc = load_library().parallax_attn_decode_plan_kernel(B, H, H_kv, Lmax, d, page_size)
    if rc < 0:
        raise ParallaxError(rc, last_error())
    return "decode_mma_kernel" if rc == 1 else "decode_kernel"


def parallax_attn_set_decode_chunk_keys(keys: int) -> None:
    _check(load_library().parallax_attn_set_decode_chunk_keys(int(keys)))


def parallax_attn_workspace_bytes() -> int:
    return int(load_library().parallax_attn_workspace_bytes())


def parallax_attn_release_workspace() -> None:
    _check(load_library().parallax_attn_release_workspace())


def parallax_check_device_error(stream=None) -> int:
    """Synchronise ``stream`` and return (and clear) the device error bits (0 = none)."""
    lib = load_library()
    rc = lib.parallax_check_device_error(_stream(stream))
    if rc not in (PARALLAX_OK, PARALLAX_ERR_DEVICE):
        raise ParallaxError(rc, last_error())
    return int(lib.parallax_last_device_error_bits())


def parallax_workspace_guards_intact() -> bool:
    """Synchronise the device and report whether the guard bands around the library's own
    workspaces are intact (no kernel wrote past either end of its workspace)."""
    rc = load_library().parallax_workspace_guards_intact()
    if rc < 0:
        raise ParallaxError(rc, last_error())
    return rc == 1


SELFTEST_DECODE = 0
SELFTEST_PREFILL = 1


def parallax_selftest_wait_timeout(family: int, limit_us: int, stream=None) -> None:
    """Launch one thread that waits, with a limit of ``limit_us`` microseconds, on a barrier
    nothing arrives on, in the error word of ``family`` (SELFTEST_DECODE or
    SELFTEST_PREFILL); the wait gives up and raises DEVERR_WAIT_TIMEOUT there."""
    _check(load_library().parallax_selftest_wait_timeout(int(family), int(limit_us),
                                                          _stream(stream)))


def parallax_version() -> int:
    return int(load_library().parallax_version())


def parallax_debug_checks() -> bool:
    """True if the loaded library is the build with device-side bounds checks."""
    return bool(load_library().parallax_debug_checks())


prefill = parallax_attn_prefill
decode = parallax_attn_decode
qkvr_projection = parallax_attn_qkvr_projection
decode_gqa = parallax_attn_decode_gqa
prefill_chunk = parallax_attn_prefill_chunk
prefill_train = parallax_attn_prefill_train
prefill_backward = parallax_attn_prefill_backward
lla_decode = parallax_lla_decode
decode_paged = parallax_attn_decode_paged
