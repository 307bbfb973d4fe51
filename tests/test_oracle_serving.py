"""Pins for the oracle's serving variants of decode: grouped-query heads (a
key/value head shared by several query heads) and a paged key/value cache
(rows looked up through a block table).

Each is pinned to a brute force that indexes the shared head and the page by
hand and evaluates the row in 50-digit decimal arithmetic with the uncentered
covariance algebra (the brute force of the base pins), plus identities that do
not use the oracle's own gather: one query head per key/value head is plain
decode, an identity block table over a reshaped cache is the cache itself, and
permuting the physical pages (with the table permuted alike) changes nothing.
Planted mistakes in the head mapping or the page lookup fail the brute force.
"""
import inspect
import textwrap

import numpy as np
import pytest

import oracle
from test_oracle_pins import _brute_row


def _brute_gqa(q, rho, kc, vc, seqlens):
    B, H, d = q.shape
    G = H // kc.shape[1]
    o = np.zeros((B, H, d))
    for b in range(B):
        n = int(seqlens[b])
        for h in range(H):
            hk = h // G
            o[b, h] = _brute_row(q[b, h], rho[b, h], kc[b, hk, :n], vc[b, hk, :n],
                                 1.0 / np.sqrt(d))
    return o


def _brute_paged(q, rho, kp, vp, bt, seqlens, P):
    B, H, d = q.shape
    G = H // kp.shape[1]
    o = np.zeros((B, H, d))
    for b in range(B):
        n = int(seqlens[b])
        for h in range(H):
            K = [kp[bt[b][t // P], h // G, t % P] for t in range(n)]
            V = [vp[bt[b][t // P], h // G, t % P] for t in range(n)]
            o[b, h] = _brute_row(q[b, h], rho[b, h], K, V, 1.0 / np.sqrt(d))
    return o


def _draw(rng, B, H, Hkv, L, d):
    q = rng.standard_normal((B, H, d))
    rho = 0.5 * rng.standard_normal((B, H, d))
    kc = 1.3 * rng.standard_normal((B, Hkv, L, d))
    vc = rng.standard_normal((B, Hkv, L, d))
    return q, rho, kc, vc


@pytest.mark.parametrize("B,H,Hkv,L,d,seqlens", [(2, 4, 2, 5, 3, [5, 2]), (1, 6, 3, 4, 2, [4]),
                                                  (3, 4, 1, 3, 2, [3, 0, 1])])
def test_gqa_brute_force(B, H, Hkv, L, d, seqlens):
    rng = np.random.default_rng(B * 10 + H)
    q, rho, kc, vc = _draw(rng, B, H, Hkv, L, d)
    sl = np.array(seqlens, dtype=np.int32)
    ref = _brute_gqa(q, rho, kc, vc, sl)
    got = oracle.decode_gqa(q, rho, kc, vc, sl)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13 * max(1.0, np.abs(ref).max()))


def test_gqa_one_query_head_per_kv_head_is_decode():
    rng = np.random.default_rng(1)
    q, rho, kc, vc = _draw(rng, 2, 3, 3, 6, 4)
    sl = np.array([6, 4], dtype=np.int32)
    np.testing.assert_array_equal(oracle.decode_gqa(q, rho, kc, vc, sl),
                                  oracle.decode(q, rho, kc, vc, sl))


@pytest.mark.parametrize("P", [1, 2, 3])
def test_paged_brute_force(P):
    rng = np.random.default_rng(P)
    B, H, Hkv, d = 2, 4, 2, 3
    seqlens = np.array([5, 3], dtype=np.int32)
    max_pages = -(-5 // P)
    num_pages = B * max_pages + 2
    kp = 1.3 * rng.standard_normal((num_pages, Hkv, P, d))
    vp = rng.standard_normal((num_pages, Hkv, P, d))
    bt = rng.permutation(num_pages)[:B * max_pages].reshape(B, max_pages).astype(np.int32)
    q = rng.standard_normal((B, H, d))
    rho = 0.5 * rng.standard_normal((B, H, d))
    ref = _brute_paged(q, rho, kp, vp, bt, seqlens, P)
    got = oracle.decode_paged(q, rho, kp, vp, bt, seqlens, P)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13 * max(1.0, np.abs(ref).max()))


def test_identity_block_table_is_the_contiguous_cache():
    """Pages cut from a contiguous cache [B, H_kv, Lmax, d] in order, with
    block_table[b, i] = b * max_pages + i, give the cache back."""
    rng = np.random.default_rng(2)
    B, H, Hkv, L, d, P = 2, 2, 2, 8, 4, 4
    q, rho, kc, vc = _draw(rng, B, H, Hkv, L, d)
    sl = np.array([8, 7], dtype=np.int32)
    mp = L // P
    # page (b, i) = rows i*P..(i+1)*P-1 of every head of sequence b
    kp = kc.reshape(B, Hkv, mp, P, d).transpose(0, 2, 1, 3, 4).reshape(B * mp, Hkv, P, d)
    vp = vc.reshape(B, Hkv, mp, P, d).transpose(0, 2, 1, 3, 4).reshape(B * mp, Hkv, P, d)
    bt = np.arange(B * mp, dtype=np.int32).reshape(B, mp)
    np.testing.assert_allclose(oracle.decode_paged(q, rho, kp, vp, bt, sl, P),
                               oracle.decode(q, rho, kc, vc, sl), rtol=1e-14, atol=1e-14)


def test_page_permutation_invariance():
    rng = np.random.default_rng(3)
    B, H, Hkv, d, P, mp = 2, 4, 1, 3, 2, 3
    n_pages = B * mp
    kp = rng.standard_normal((n_pages, Hkv, P, d))
    vp = rng.standard_normal((n_pages, Hkv, P, d))
    bt = np.arange(n_pages, dtype=np.int32).reshape(B, mp)
    q = rng.standard_normal((B, H, d))
    rho = rng.standard_normal((B, H, d))
    sl = np.array([6, 5], dtype=np.int32)
    perm = rng.permutation(n_pages)
    inv = np.argsort(perm)
    # physical page j of the permuted pool holds logical page perm[j]
    got = oracle.decode_paged(q, rho, kp[perm], vp[perm], inv[bt].astype(np.int32), sl, P)
    ref = oracle.decode_paged(q, rho, kp, vp, bt, sl, P)
    np.testing.assert_allclose(got, ref, rtol=1e-14, atol=1e-14)


# planted mistakes in the head mapping and the page lookup
MUTANTS = {
    "kv head h % H_kv": (oracle.decode_gqa, "heads = [h // G for h in range(H)]",
                         "heads = [h % Hkv for h in range(H)]"),
    "page row t // P": (oracle.gather_pages, "pages[bt[b, t // P], :, t % P]",
                        "pages[bt[b, t % P], :, t // P]"),
    "block table transposed": (oracle.gather_pages, "bt = np.asarray(block_table)",
                               "bt = np.asarray(block_table).T.copy().reshape(np.asarray(block_table).shape)"),
}


def _mutant(fn, old, new):
    src = textwrap.dedent(inspect.getsource(fn))
    assert old in src, old
    ns = dict(vars(oracle))
    exec(src.replace(old, new), ns)
    return ns


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_planted_mistake(name):
    fn, old, new = MUTANTS[name]
    ns = _mutant(fn, old, new)
    rng = np.random.default_rng(4)
    B, H, Hkv, d, P = 2, 4, 2, 3, 2
    sl = np.array([5, 3], dtype=np.int32)
    mp = 3
    kp = 1.3 * rng.standard_normal((B * mp + 1, Hkv, P, d))
    vp = rng.standard_normal((B * mp + 1, Hkv, P, d))
    bt = rng.permutation(B * mp + 1)[:B * mp].reshape(B, mp).astype(np.int32)
    q = rng.standard_normal((B, H, d))
    rho = 0.5 * rng.standard_normal((B, H, d))
    ref = _brute_paged(q, rho, kp, vp, bt, sl, P)
    try:
        if fn is oracle.decode_gqa:
            kc = oracle.gather_pages(kp, bt, sl, P)
            vc = oracle.gather_pages(vp, bt, sl, P)
            got = ns["decode_gqa"](q, rho, kc, vc, sl)
        else:
            kc = ns["gather_pages"](kp, bt, sl, P)
            vc = ns["gather_pages"](vp, bt, sl, P)
            got = oracle.decode_gqa(q, rho, kc, vc, sl)
    except (IndexError, ValueError):
        return  # the mistake breaks the lookup outright
    assert not np.allclose(got, ref, rtol=0, atol=1e-9), f"mutant survived: {name}"


# ----------------------------------------------------------------------------
# chunked prefill that continues a cached sequence
# ----------------------------------------------------------------------------
def _brute_chunk(q, rho, kn, vn, kc, vc, cache_lens):
    B, H, Lq, d = q.shape
    o = np.zeros((B, H, Lq, d))
    for b in range(B):
        off = int(cache_lens[b])
        for h in range(H):
            for i in range(Lq):
                K = [kc[b, h, t] for t in range(off)] + [kn[b, h, t] for t in range(i + 1)]
                V = [vc[b, h, t] for t in range(off)] + [vn[b, h, t] for t in range(i + 1)]
                o[b, h, i] = _brute_row(q[b, h, i], None if rho is None else rho[b, h, i], K, V,
                                        1.0 / np.sqrt(d))
    return o


@pytest.mark.parametrize("with_rho", [True, False])
def test_chunk_brute_force(with_rho):
    rng = np.random.default_rng(12)
    B, H, Lq, Lmax, d = 2, 2, 3, 6, 3
    q = rng.standard_normal((B, H, Lq, d))
    rho = 0.7 * rng.standard_normal((B, H, Lq, d)) if with_rho else None
    kn, vn = 1.2 * rng.standard_normal((2, B, H, Lq, d))
    kc, vc = 1.2 * rng.standard_normal((2, B, H, Lmax, d))
    cl = np.array([3, 0])
    ref = _brute_chunk(q, rho, kn, vn, kc, vc, cl)
    got = oracle.prefill_chunk(q, rho, kn, vn, kc, vc, cl)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13 * max(1.0, np.abs(ref).max()))


@pytest.mark.parametrize("off", [0, 1, 5, 9])
def test_chunks_compose_to_one_prefill(off):
    """Rows off..L-1 of one causal prefill of L tokens equal the chunk prefill of
    those rows over a cache holding tokens 0..off-1 (whatever the cache holds
    past off is never read)."""
    rng = np.random.default_rng(off)
    B, H, L, d = 2, 2, 10, 4
    q, rho, k, v = (rng.standard_normal((B, H, L, d)) for _ in range(4))
    full = oracle.prefill(q, rho, k, v, causal=True)
    kc, vc = 99.0 * rng.standard_normal((2, B, H, L + 3, d))  # garbage past off
    kc[:, :, :off], vc[:, :, :off] = k[:, :, :off], v[:, :, :off]
    got = oracle.prefill_chunk(q[:, :, off:], rho[:, :, off:], k[:, :, off:], v[:, :, off:], kc,
                               vc, np.array([off, off]))
    np.testing.assert_allclose(got, full[:, :, off:], rtol=1e-13, atol=1e-13)


CHUNK_MUTANTS = {
    "diagonal excluded": ("nkeys = off + 1 + np.arange(Lq)", "nkeys = off + np.arange(Lq) + (off == 0)"),
    "cache ignored": ("K = np.concatenate([kc[b, h, :off], kn[b, h]])",
                      "K = np.concatenate([kn[b, h, :1].repeat(off, 0), kn[b, h]])"),
    "cache one row short": ("V = np.concatenate([vc[b, h, :off], vn[b, h]])",
                            "V = np.concatenate([vc[b, h, 1:off + 1], vn[b, h]])"),
}


@pytest.mark.parametrize("name", sorted(CHUNK_MUTANTS))
def test_chunk_pins_reject_planted_mistake(name):
    old, new = CHUNK_MUTANTS[name]
    ns = _mutant(oracle.prefill_chunk, old, new)
    rng = np.random.default_rng(13)
    B, H, Lq, Lmax, d = 2, 2, 3, 6, 3
    q, rho, kn, vn = (rng.standard_normal((B, H, Lq, d)) for _ in range(4))
    kc, vc = rng.standard_normal((2, B, H, Lmax, d))
    cl = np.array([3, 2])
    ref = _brute_chunk(q, rho, kn, vn, kc, vc, cl)
    got = ns["prefill_chunk"](q, rho, kn, vn, kc, vc, cl)
    assert not np.allclose(got, ref, rtol=0, atol=1e-9), f"mutant survived: {name}"
