"""fp64 CPU oracle for Parallax attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference arm may import this package.  The CUDA product path never imports
it, and it imports nothing from the product package.

The arithmetic lives in ``parallax_oracle.c`` (plain loops, fp64, OpenMP over
rows); this module only marshals numpy arrays.  Each function follows the
definition in the Parallax news pages ("Parallax mantem softmax ...",
paragraph 2; "Parallax garde softmax ...", paragraph 2): the output is softmax
attention minus the key/value covariance multiplied by the probe
``rho_i = W_R x_i``; ``W_R = 0`` (``rho=None``) gives plain softmax attention.

Forms: ``"explicit"`` (d x d covariance, centered two-pass), ``"contracted"``
(rho contracted into the centered key side first, O(n d) per row) and
``"uncentered"`` (one pass of raw moments).  All three are the same function
of the inputs up to rounding.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "parallax_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

FORMS = {"explicit": 0, "contracted": 1, "uncentered": 2}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``parallax_oracle.c`` into ``liboracle.so`` (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            dp = ctypes.POINTER(ctypes.c_double)
            i64 = ctypes.c_int64
            lib.oracle_rows.argtypes = [dp, dp, dp, dp, ctypes.POINTER(i64), i64, i64, i64,
                                        ctypes.c_double, ctypes.c_int, dp]
            lib.oracle_prefill.argtypes = [dp, dp, dp, dp, i64, i64, i64, i64, ctypes.c_int,
                                           ctypes.c_double, ctypes.c_int, dp]
            lib.oracle_decode.argtypes = [dp, dp, dp, dp, ctypes.POINTER(ctypes.c_int32), i64,
                                          i64, i64, i64, ctypes.c_double, ctypes.c_int, dp]
            for f in (lib.oracle_rows, lib.oracle_prefill, lib.oracle_decode):
                f.restype = ctypes.c_int
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x):
    """Widen to a contiguous float64 numpy array (torch tensors are moved to the CPU)."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: widen exactly on the host
        import torch

        x = x.detach().to("cpu", torch.float64).contiguous().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use on this host."""
    return int(_load().oracle_num_threads())


def prefill(q, rho, k, v, causal: bool = True, scale: float | None = None,
            form: str = "explicit") -> np.ndarray:
    """Parallax prefill rows; q, rho, k, v are [B, H, L, d]; rho=None means W_R = 0."""
    q, rho, k, v = _f64(q), _f64(rho), _f64(k), _f64(v)
    B, H, L, d = q.shape
    assert k.shape == v.shape == q.shape and (rho is None or rho.shape == q.shape)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.empty_like(q)
    rc = _load().oracle_prefill(_ptr(q), _ptr(rho), _ptr(k), _ptr(v), B, H, L, d,
                                1 if causal else 0, float(scale), FORMS[form], _ptr(o))
    if rc != 0:
        raise RuntimeError(f"oracle_prefill failed ({rc})")
    return o


def decode(q, rho, k_cache, v_cache, seqlens, scale: float | None = None,
           form: str = "explicit") -> np.ndarray:
    """Parallax single-token decode; q, rho [B, H, d], caches [B, H, Lmax, d], seqlens [B]."""
    q, rho, kc, vc = _f64(q), _f64(rho), _f64(k_cache), _f64(v_cache)
    if hasattr(seqlens, "detach"):
        seqlens = seqlens.detach().cpu().numpy()
    sl = np.ascontiguousarray(seqlens, dtype=np.int32)
    B, H, Lmax, d = kc.shape
    assert q.shape == (B, H, d) and vc.shape == kc.shape and sl.shape == (B,)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.empty_like(q)
    rc = _load().oracle_decode(_ptr(q), _ptr(rho), _ptr(kc), _ptr(vc),
                               sl.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), B, H, Lmax, d,
                               float(scale), FORMS[form], _ptr(o))
    if rc != 0:
        raise RuntimeError(f"oracle_decode failed ({rc})")
    return o


def rows(q, rho, k, v, nkeys, scale: float, form: str = "explicit") -> np.ndarray:
    """Rows that share one key set: q, rho [nq, d]; k, v [nk, d]; row i uses keys < nkeys[i]."""
    q, rho, k, v = _f64(q), _f64(rho), _f64(k), _f64(v)
    nq, d = q.shape
    nk = k.shape[0]
    nkeys = np.ascontiguousarray(nkeys, dtype=np.int64)
    assert nkeys.shape == (nq,) and k.shape == v.shape == (nk, d)
    o = np.empty_like(q)
    rc = _load().oracle_rows(_ptr(q), _ptr(rho), _ptr(k), _ptr(v),
                             nkeys.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), nq, nk, d,
                             float(scale), FORMS[form], _ptr(o))
    if rc != 0:
        raise RuntimeError(f"oracle_rows failed ({rc})")
    return o


def qkvr_projection(x, w, H: int, d: int) -> list:
    """The layer's input projections: q, k, v and the probe rho = W_R x.

    The probe is a learned linear map of the layer input x_i ("Parallax mantem
    softmax ...", paragraph 2: rho_i = W_R x_i); q, k and v are the usual
    attention projections of the same x_i.  Here they are one product with the
    stacked weight:

      x : [B, L, width]            (one row per token)
      w : [n_out * H * d, width]   rows = output features, blocks W_q; W_k; W_v; (W_R)
      y = x w^T                    [B, L, n_out * H * d]      (fp64, numpy matmul)
      out[t][b, h, l, c] = y[b, l, t*H*d + h*d + c]           (t = 0: q, 1: k, 2: v, 3: rho)

    Returns the n_out arrays [B, H, L, d] in fp64 (n_out = rows of w / (H*d)).
    """
    x, w = _f64(x), _f64(w)
    B, L, width = x.shape
    n_out, rem = divmod(w.shape[0], H * d)
    assert rem == 0 and w.shape[1] == width
    y = x.reshape(B * L, width) @ w.T
    y = y.reshape(B, L, n_out, H, d)
    return [np.ascontiguousarray(y[:, :, t].transpose(0, 2, 1, 3)) for t in range(n_out)]


def decode_gqa(q, rho, k_cache, v_cache, seqlens, scale: float | None = None,
               form: str = "explicit") -> np.ndarray:
    """Decode with key/value heads shared by groups of query heads (grouped-query
    attention): q, rho [B, H, d]; caches [B, H_kv, Lmax, d] with H a multiple of
    H_kv; query head h reads key/value head h // (H // H_kv).  Each query head's
    output is the Parallax decode of its own q and rho against that cache."""
    q, rho, kc, vc = _f64(q), _f64(rho), _f64(k_cache), _f64(v_cache)
    B, H, d = q.shape
    Hkv = kc.shape[1]
    G, rem = divmod(H, Hkv)
    assert rem == 0
    heads = [h // G for h in range(H)]
    return decode(q, rho, kc[:, heads], vc[:, heads], seqlens, scale=scale, form=form)


def gather_pages(pages, block_table, seqlens, page_size: int) -> np.ndarray:
    """The contiguous cache [B, H_kv, Lmax, d] that a paged cache stands for:
    key t of sequence b lives in page block_table[b, t // page_size], row
    t % page_size, of pages [num_pages, H_kv, page_size, d].  Rows at or past
    seqlens[b] are left zero; Lmax = block_table.shape[1] * page_size."""
    pages = _f64(pages)
    if hasattr(block_table, "detach"):
        block_table = block_table.detach().cpu().numpy()
    if hasattr(seqlens, "detach"):
        seqlens = seqlens.detach().cpu().numpy()
    bt = np.asarray(block_table)
    B, max_pages = bt.shape
    _, Hkv, P, d = pages.shape
    assert P == page_size
    out = np.zeros((B, Hkv, max_pages * P, d))
    for b in range(B):
        for t in range(int(seqlens[b])):
            out[b, :, t] = pages[bt[b, t // P], :, t % P]
    return out


def decode_paged(q, rho, k_pages, v_pages, block_table, seqlens, page_size: int,
                 scale: float | None = None, form: str = "explicit") -> np.ndarray:
    """Decode against a paged key/value cache (see gather_pages), with grouped
    query heads when the pages hold fewer heads than q (see decode_gqa)."""
    kc = gather_pages(k_pages, block_table, seqlens, page_size)
    vc = gather_pages(v_pages, block_table, seqlens, page_size)
    return decode_gqa(q, rho, kc, vc, seqlens, scale=scale, form=form)


def prefill_chunk(q, rho, k_new, v_new, k_cache, v_cache, cache_lens, scale: float | None = None,
                  form: str = "explicit") -> np.ndarray:
    """Causal prefill of a chunk of new tokens that continues cached sequences.

    q, rho, k_new, v_new : [B, H, Lq, d]   the chunk (Lq new tokens per sequence)
    k_cache, v_cache     : [B, H, Lmax, d] sequence b holds cache_lens[b] earlier tokens
    Token i of the chunk sits at position p = cache_lens[b] + i of its sequence; its
    key set is the sequence's keys at positions 0..p: the cached rows 0..cache_lens[b]-1
    followed by the chunk's rows 0..i.  Returns o [B, H, Lq, d].
    """
    q, rho, kn, vn = _f64(q), _f64(rho), _f64(k_new), _f64(v_new)
    kc, vc = _f64(k_cache), _f64(v_cache)
    if hasattr(cache_lens, "detach"):
        cache_lens = cache_lens.detach().cpu().numpy()
    B, H, Lq, d = q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.empty_like(q)
    for b in range(B):
        off = int(cache_lens[b])
        nkeys = off + 1 + np.arange(Lq)
        for h in range(H):
            K = np.concatenate([kc[b, h, :off], kn[b, h]])
            V = np.concatenate([vc[b, h, :off], vn[b, h]])
            o[b, h] = rows(q[b, h], None if rho is None else rho[b, h], K, V, nkeys, scale,
                           form=form)
    return o


def _head_terms(q, rho, k, v, causal: bool, scale: float):
    """Per-head quantities of the forward pass (fp64, one head [L, d] at a time):
    softmax weights P, probe scores R = rho k^T, rbar = sum_j p_j r_j, and the output
    weights Wt = P (1 + rbar - R), so that o = Wt v (the output written as one
    weighted sum: o_i = mu_v - sum_j p_j (r_j - rbar)(v_j - mu_v) = sum_j w_j v_j)."""
    L = q.shape[0]
    S = scale * (q @ k.T)
    if causal:
        S = np.where(np.tril(np.ones((L, k.shape[0]), dtype=bool)), S, -np.inf)
    m = S.max(axis=1, keepdims=True)
    E = np.exp(S - m)
    Z = E.sum(axis=1, keepdims=True)
    P = E / Z
    lse = (m + np.log(Z))[:, 0]
    R = np.zeros_like(S) if rho is None else rho @ k.T
    rbar = (P * R).sum(axis=1)
    Wt = P * (1.0 + rbar[:, None] - R)
    return P, R, rbar, Wt, lse


def prefill_stats(q, rho, k, v, causal: bool = True, scale: float | None = None):
    """Per-row quantities a training forward keeps for the backward pass:
    lse_i = log sum_j exp(s_ij) (natural log, s = scale q.k), rbar_i = sum_j p_ij r_ij
    and mu_v,i = sum_j p_ij v_j.  Returns (lse [B,H,L], rbar [B,H,L], mu_v [B,H,L,d])."""
    q, rho, k, v = _f64(q), _f64(rho), _f64(k), _f64(v)
    B, H, L, d = q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    lse = np.empty((B, H, L))
    rbar = np.empty((B, H, L))
    mu = np.empty((B, H, L, d))
    for b in range(B):
        for h in range(H):
            P, _, rb, _, ls = _head_terms(q[b, h], None if rho is None else rho[b, h], k[b, h],
                                          v[b, h], causal, scale)
            lse[b, h], rbar[b, h], mu[b, h] = ls, rb, P @ v[b, h]
    return lse, rbar, mu


def prefill_backward(q, rho, k, v, do, causal: bool = True, scale: float | None = None):
    """Gradients of sum(do * o) for the Parallax prefill o = prefill(q, rho, k, v).

    With o_i = sum_j w_ij v_j, w_ij = p_ij (1 + rbar_i - r_ij) (see _head_terms),
    D_ij = do_i . v_j, abar_i = sum_j p_ij D_ij (= do_i . mu_v,i), delta_i = do_i . o_i:
      dv_j   = sum_i w_ij do_i
      dr_ij  = p_ij (abar_i - D_ij)                      (r_ij = rho_i . k_j)
      ds_ij  = p_ij ((D_ij - abar_i)(rbar_i - r_ij) + D_ij - delta_i)   (s_ij = scale q_i.k_j)
      dq_i   = scale sum_j ds_ij k_j,     drho_i = sum_j dr_ij k_j
      dk_j   = scale sum_i ds_ij q_i + sum_i dr_ij rho_i
    Returns (dq, drho, dk, dv), each [B, H, L, d] in fp64 (drho is the gradient at the
    given rho, zeros included: rho=None is treated as rho = 0)."""
    q, rho, k, v, do = _f64(q), _f64(rho), _f64(k), _f64(v), _f64(do)
    B, H, L, d = q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    if rho is None:
        rho = np.zeros_like(q)
    dq, drho, dk, dv = (np.zeros_like(q) for _ in range(4))
    for b in range(B):
        for h in range(H):
            qh, rh, kh, vh, doh = q[b, h], rho[b, h], k[b, h], v[b, h], do[b, h]
            P, R, rbar, Wt, _ = _head_terms(qh, rh, kh, vh, causal, scale)
            o = Wt @ vh
            Dm = doh @ vh.T
            abar = (P * Dm).sum(axis=1)
            delta = (doh * o).sum(axis=1)
            dR = P * (abar[:, None] - Dm)
            dS = P * ((Dm - abar[:, None]) * (rbar[:, None] - R) + Dm - delta[:, None])
            dv[b, h] = Wt.T @ doh
            dq[b, h] = scale * (dS @ kh)
            drho[b, h] = dR @ kh
            dk[b, h] = scale * (dS.T @ qh) + dR.T @ rh
    return dq, drho, dk, dv


def conjugate_gradient(A, b, iters: int, tol: float = 0.0):
    """Plain conjugate gradient for a symmetric positive (semi)definite A, from x = 0:
    r = b, p = r; each step a = (r.r)/(p.A p), x += a p, r -= a A p, p = r + (r'.r')/(r.r) p.
    Stops after `iters` steps or once |r| <= tol |b|."""
    x = np.zeros_like(b)
    r = b.copy()
    p = r.copy()
    rs = float(r @ r)
    stop = (tol * float(np.sqrt(b @ b))) ** 2
    for _ in range(iters):
        if rs <= stop or rs == 0.0:
            break
        Ap = A @ p
        alpha = rs / float(p @ Ap)
        x += alpha * p
        r -= alpha * Ap
        rs_new = float(r @ r)
        p = r + (rs_new / rs) * p
        rs = rs_new
    return x


def lla_decode(q, k_cache, v_cache, seqlens, scale: float | None = None, iters: int | None = None,
               tol: float = 0.0):
    """Exact local linear attention for one query token per (b, h), the method the Parallax
    probe replaces (the pages: Parallax keeps LLA's covariance correction but swaps its
    per-query solve for the learned probe W_R x).

    With softmax weights p_j over the sequence's keys, mu_k = sum p k, mu_v = sum p v and
    Sigma_kk = sum_j p_j (k_j - mu_k)(k_j - mu_k)^T, the probe is the solution of
    Sigma_kk rho = mu_k - q, found by conjugate gradient (conjugate_gradient, `iters`
    steps, default d: exact in exact arithmetic); the output is the Parallax output with
    that probe, o = mu_v - C^T rho.  Returns (o [B, H, d], rho [B, H, d]).  A sequence
    with no keys gives o = 0 and rho = 0."""
    q, kc, vc = _f64(q), _f64(k_cache), _f64(v_cache)
    if hasattr(seqlens, "detach"):
        seqlens = seqlens.detach().cpu().numpy()
    B, H, Lmax, d = kc.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    if iters is None:
        iters = d
    rho = np.zeros((B, H, d))
    for b in range(B):
        n = int(seqlens[b])
        if n == 0:
            continue
        for h in range(H):
            K = kc[b, h, :n]
            s = scale * (K @ q[b, h])
            p = np.exp(s - s.max())
            p /= p.sum()
            mu_k = p @ K
            Kc = K - mu_k
            sigma = (Kc * p[:, None]).T @ Kc
            rho[b, h] = conjugate_gradient(sigma, mu_k - q[b, h], iters, tol)
    o = decode(q, rho, kc, vc, seqlens, scale=scale)
    return o, rho
