"""Pins for the CPU oracle: each check compares it with something other than itself.

Each ``check_*`` takes a loaded oracle library and raises AssertionError when the
oracle disagrees with what the pages or the mathematics fix.  The tests run
them on the real oracle (must pass) and on deliberately broken copies of the
oracle source (must fail), which shows each pin can see the mistake it guards.

Sources of truth used here, none of them the oracle's own code:
  * a library routine: torch's CPU ``scaled_dot_product_attention`` in float64,
    which for G = H is multi-head attention and for G = 1 is multi-query
    attention ("Grouped-query attention (GQA)" concept page, "Choosing the group
    count G": G = H is MHA, G = 1 is MQA; arxiv:2305.13245 §2.2);
  * the definition's consequence that replicating each K/V head H/G times
    turns GQA into MHA (same page, "Overview": every query head in a group
    attends with that group's single key and value head);
  * closed forms (one token, two tokens, constant keys) and invariances
    (shifting every key by the same vector, permuting cache positions);
  * brute force on tiny integer inputs with 50-digit arithmetic and no
    maximum subtraction;
  * for the variants (cross-attention over all positions, sliding window,
    paged cache, fused append): the library's attention with an explicit
    position mask, a numpy scatter of the cache into pages that the gather
    must invert, the newest-position closed form (window 1) and a numpy
    assignment of the appended row;
  * for the mean-pool conversion (same page, "Converted and uptrained
    checkpoints" and the conversion pseudocode; arxiv:2305.13245 §2.1):
    identical heads, the identity at G = H, the column mean at G = 1, exact
    small-integer means, and the pages' [d_model, H*h] layout.
"""
from __future__ import annotations

import itertools
import math

import mpmath
import numpy as np
import torch
import torch.nn.functional as F

import oracle
from kv_cache_decode_06_b300.inputs import (
    DecodeConfig, bf16_bits_to_f32, f32_to_bf16_bits, make_decode_inputs, make_meanpool_input,
)


def _f64(bits):
    return bf16_bits_to_f32(bits).astype(np.float64)


def _small_cfg(G, H=8, d=16, L=37, B=3, seq=(5, 37)):
    return DecodeConfig("pin", 90 + G, B=B, H=H, G=G, d=d, Lmax=L, seq_lo=seq[0], seq_hi=seq[1])


def sdpa_reference(inp) -> np.ndarray:
    """torch CPU scaled_dot_product_attention (float64), one batch entry at a time."""
    cfg = inp.cfg
    q = torch.from_numpy(_f64(inp.q))
    k = torch.from_numpy(_f64(inp.k))
    v = torch.from_numpy(_f64(inp.v))
    out = np.zeros((cfg.B, cfg.H, cfg.d))
    for b in range(cfg.B):
        T = int(inp.seq_lens[b])
        if T == 0:
            continue
        o = F.scaled_dot_product_attention(
            q[b][None, :, None, :], k[b, :, :T][None], v[b, :, :T][None],
            scale=float(inp.scale), enable_gqa=True)
        out[b] = o[0, :, 0, :].numpy()
    return out


def check_mha_matches_library(lib):
    """G = H: the oracle equals the library's multi-head attention."""
    inp = make_decode_inputs(_small_cfg(G=8))
    got = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale, lib=lib)
    ref = sdpa_reference(inp)
    assert np.max(np.abs(got - ref)) <= 1e-12, np.max(np.abs(got - ref))


def check_mqa_matches_library(lib):
    """G = 1: every head attends with the single K/V head."""
    inp = make_decode_inputs(_small_cfg(G=1))
    got = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale, lib=lib)
    q = torch.from_numpy(_f64(inp.q))
    k = torch.from_numpy(_f64(inp.k))
    v = torch.from_numpy(_f64(inp.v))
    for b in range(inp.cfg.B):
        T = int(inp.seq_lens[b])
        kb = k[b, 0, :T]
        vb = v[b, 0, :T]
        ref = F.scaled_dot_product_attention(q[b][:, None, :], kb.expand(inp.cfg.H, T, -1),
                                             vb.expand(inp.cfg.H, T, -1), scale=float(inp.scale))
        assert np.max(np.abs(got[b] - ref[:, 0, :].numpy())) <= 1e-12


def check_gqa_matches_library(lib, G=2):
    """1 < G < H: the library's grouped attention maps head i to K/V head i // (H/G)."""
    inp = make_decode_inputs(_small_cfg(G=G))
    got = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale, lib=lib)
    ref = sdpa_reference(inp)
    assert np.max(np.abs(got - ref)) <= 1e-12


def check_replication_turns_gqa_into_mha(lib):
    """Repeating each K/V head H/G times and running with G' = H gives the same result.

    The oracle evaluates each head from the same widened numbers in the same
    order either way, so equality is bitwise.
    """
    inp = make_decode_inputs(_small_cfg(G=2))
    n = inp.cfg.n
    got = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale, lib=lib)
    k_rep = np.repeat(inp.k, n, axis=1)
    v_rep = np.repeat(inp.v, n, axis=1)
    mha = oracle.gqa_decode_f64(inp.q, k_rep, v_rep, inp.seq_lens, inp.scale, lib=lib)
    assert np.array_equal(got, mha)


def check_constant_keys_give_mean_of_v(lib):
    """All keys equal: the softmax is uniform, so out is the mean of the valid values."""
    inp = make_decode_inputs(_small_cfg(G=4))
    k = inp.k.copy()
    k[:, :, :, :] = k[:, :, :1, :]
    got = oracle.gqa_decode_f64(inp.q, k, inp.v, inp.seq_lens, inp.scale, lib=lib)
    v = _f64(inp.v)
    n = inp.cfg.n
    for b in range(inp.cfg.B):
        T = int(inp.seq_lens[b])
        for i in range(inp.cfg.H):
            ref = v[b, i // n, :T].mean(axis=0)
            assert np.max(np.abs(got[b, i] - ref)) <= 1e-13


def check_single_token_returns_v0(lib):
    """One cached token: the softmax weight is exactly 1, so out equals v_0 bit for bit."""
    cfg = _small_cfg(G=2)
    inp = make_decode_inputs(cfg, seq_lens=[1] * cfg.B)
    got = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale, lib=lib)
    v = _f64(inp.v)
    for i in range(cfg.H):
        assert np.array_equal(got[:, i], v[:, i // cfg.n, 0])


def check_two_token_closed_form(lib):
    """Two tokens: out = sigmoid(s0 - s1) v0 + sigmoid(s1 - s0) v1."""
    cfg = _small_cfg(G=2)
    inp = make_decode_inputs(cfg, seq_lens=[2] * cfg.B)
    got = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale, lib=lib)
    q, k, v = _f64(inp.q), _f64(inp.k), _f64(inp.v)
    sc = float(inp.scale)
    for b in range(cfg.B):
        for i in range(cfg.H):
            g = i // cfg.n
            s0 = sc * math.fsum(q[b, i] * k[b, g, 0])
            s1 = sc * math.fsum(q[b, i] * k[b, g, 1])
            w0 = 1.0 / (1.0 + math.exp(s1 - s0))
            w1 = 1.0 / (1.0 + math.exp(s0 - s1))
            ref = w0 * v[b, g, 0] + w1 * v[b, g, 1]
            assert np.max(np.abs(got[b, i] - ref)) <= 1e-14


def _integer_inputs(cfg, lo=-4, hi=4, seed=7):
    """Small-integer bf16 data (exact in bf16 and in every sum here)."""
    inp = make_decode_inputs(cfg)
    rng = np.random.default_rng(seed)
    q = f32_to_bf16_bits(rng.integers(lo, hi + 1, size=inp.q.shape).astype(np.float32))
    k = inp.k.copy()
    v = inp.v.copy()
    for b in range(cfg.B):
        T = int(inp.seq_lens[b])
        k[b, :, :T] = f32_to_bf16_bits(rng.integers(lo, hi + 1, size=(cfg.G, T, cfg.d)).astype(np.float32))
        v[b, :, :T] = f32_to_bf16_bits(rng.integers(lo, hi + 1, size=(cfg.G, T, cfg.d)).astype(np.float32))
    return inp, q, k, v


def check_key_shift_invariance(lib):
    """k_t += u for every valid t adds q.u to every score of a row: out is unchanged."""
    cfg = _small_cfg(G=2)
    inp, q, k, v = _integer_inputs(cfg)
    rng = np.random.default_rng(11)
    u = rng.integers(-3, 4, size=(cfg.B, cfg.G, 1, cfg.d)).astype(np.float32)
    kf = bf16_bits_to_f32(k).copy()
    for b in range(cfg.B):
        T = int(inp.seq_lens[b])
        kf[b, :, :T] += u[b]
    k2 = f32_to_bf16_bits(kf)
    assert np.array_equal(bf16_bits_to_f32(k2)[:, :, :5], kf[:, :, :5])  # exact shift
    a = oracle.gqa_decode_f64(q, k, v, inp.seq_lens, inp.scale, lib=lib)
    c = oracle.gqa_decode_f64(q, k2, v, inp.seq_lens, inp.scale, lib=lib)
    assert np.max(np.abs(a - c)) <= 1e-12


def check_permutation_invariance(lib):
    """Reordering the valid cache positions (same permutation for K and V) changes nothing."""
    cfg = _small_cfg(G=4)
    inp = make_decode_inputs(cfg)
    k = inp.k.copy()
    v = inp.v.copy()
    rng = np.random.default_rng(3)
    for b in range(cfg.B):
        T = int(inp.seq_lens[b])
        perm = rng.permutation(T)
        k[b, :, :T] = inp.k[b, :, perm].transpose(1, 0, 2)
        v[b, :, :T] = inp.v[b, :, perm].transpose(1, 0, 2)
    a = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale, lib=lib)
    c = oracle.gqa_decode_f64(inp.q, k, v, inp.seq_lens, inp.scale, lib=lib)
    assert np.max(np.abs(a - c)) <= 1e-13


def _mp_attention(qv, K, V, scale):
    """Softmax attention in 50-digit arithmetic, straight from the definition (no max shift)."""
    with mpmath.workdps(50):
        sc = mpmath.mpf(float(scale))
        s = [sc * mpmath.fsum(mpmath.mpf(float(a)) * mpmath.mpf(float(b)) for a, b in zip(qv, kt)) for kt in K]
        e = [mpmath.e ** x for x in s]
        z = mpmath.fsum(e)
        return [float(mpmath.fsum(e[t] * mpmath.mpf(float(V[t][j])) for t in range(len(K))) / z)
                for j in range(len(V[0]))]


def check_bruteforce_high_precision(lib):
    """Every q, k, v in {-1, 0, 1} on tiny shapes against 50-digit arithmetic."""
    vals = (-1.0, 0.0, 1.0)
    H, G, d, L = 2, 1, 2, 2
    scale = np.float32(0.75)
    kvs = list(itertools.product(vals, repeat=L * d))
    qs = list(itertools.product(vals, repeat=d))
    rng = np.random.default_rng(5)
    # every (q, K) pair with a fixed random V, plus every V with a random (q, K)
    cases = [(qq, kk, tuple(rng.choice(vals, size=L * d))) for qq in qs for kk in kvs]
    cases += [(tuple(rng.choice(vals, size=d)), tuple(rng.choice(vals, size=L * d)), vv) for vv in kvs]
    for T in (1, 2):
        qb = np.zeros((len(cases), H, d), dtype=np.float32)
        kb = np.zeros((len(cases), G, L, d), dtype=np.float32)
        vb = np.zeros((len(cases), G, L, d), dtype=np.float32)
        for c, (qq, kk, vv) in enumerate(cases):
            qb[c, 0] = qq
            qb[c, 1] = [-x for x in qq]
            kb[c, 0] = np.reshape(kk, (L, d))
            vb[c, 0] = np.reshape(vv, (L, d))
        sl = np.full(len(cases), T, dtype=np.int32)
        got = oracle.gqa_decode_f64(f32_to_bf16_bits(qb), f32_to_bf16_bits(kb), f32_to_bf16_bits(vb),
                                    sl, scale, lib=lib)
        for c in range(len(cases)):
            for i in range(H):
                ref = _mp_attention(qb[c, i], kb[c, 0, :T], vb[c, 0, :T], scale)
                assert np.max(np.abs(got[c, i] - np.asarray(ref))) <= 1e-15


def check_tail_is_never_read(lib):
    """NaN in every position t >= seq_len does not reach the output; row subsets agree."""
    cfg = _small_cfg(G=2)
    inp = make_decode_inputs(cfg, poison_tail=True)
    got = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale, lib=lib)
    assert np.isfinite(got).all()
    clean = make_decode_inputs(cfg, poison_tail=False)
    ref = oracle.gqa_decode_f64(clean.q, clean.k, clean.v, clean.seq_lens, clean.scale, lib=lib)
    assert np.array_equal(got, ref)
    rows = np.array([0, 5, cfg.H + 3, cfg.B * cfg.H - 1])
    sub = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale, rows=rows, lib=lib)
    assert np.array_equal(sub.reshape(-1, cfg.d)[rows], got.reshape(-1, cfg.d)[rows])


def check_empty_sequence_gives_zero(lib):
    cfg = _small_cfg(G=2)
    inp = make_decode_inputs(cfg, seq_lens=[0, 3, 0])
    got = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale, lib=lib)
    assert np.array_equal(got[0], np.zeros_like(got[0])) and np.array_equal(got[2], np.zeros_like(got[2]))
    assert np.isfinite(got[1]).all() and np.abs(got[1]).max() > 0


# ------------------------------------------------ variants of the decode step

def _sdpa_masked(inp, allowed) -> np.ndarray:
    """torch CPU attention (float64) with an explicit boolean mask allowed[b][t] over the Lmax positions."""
    cfg = inp.cfg
    q = torch.from_numpy(_f64(inp.q))
    k = torch.from_numpy(np.nan_to_num(_f64(inp.k)))
    v = torch.from_numpy(np.nan_to_num(_f64(inp.v)))
    out = np.zeros((cfg.B, cfg.H, cfg.d))
    for b in range(cfg.B):
        m = torch.from_numpy(np.asarray(allowed[b], dtype=bool))
        if not m.any():
            continue
        o = F.scaled_dot_product_attention(q[b][None, :, None, :], k[b][None], v[b][None],
                                           attn_mask=m[None, None, None, :], scale=float(inp.scale),
                                           enable_gqa=True)
        out[b] = o[0, :, 0, :].numpy()
    return out


def check_cross_attention_matches_library(lib):
    """seq_lens = NULL: every one of the Lmax positions is attended (an encoder cache of fixed length)."""
    cfg = _small_cfg(G=2, L=29, seq=(29, 29))
    inp = make_decode_inputs(cfg)
    got = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, None, inp.scale, lib=lib)
    ref = _sdpa_masked(inp, np.ones((cfg.B, cfg.Lmax), dtype=bool))
    assert np.max(np.abs(got - ref)) <= 1e-12


def check_window_matches_library_mask(lib):
    """A window W attends to positions max(0, T - W) <= t < T: the library with that mask agrees."""
    cfg = _small_cfg(G=4, L=41, B=4, seq=(1, 41))
    inp = make_decode_inputs(cfg, seq_lens=[41, 17, 1, 30], poison_tail=True)
    for W in (1, 2, 7, 16, 30, 41, 100):
        got = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale, window=W, lib=lib)
        allowed = np.zeros((cfg.B, cfg.Lmax), dtype=bool)
        for b, T in enumerate(inp.seq_lens):
            allowed[b, max(0, int(T) - W):int(T)] = True
        ref = _sdpa_masked(inp, allowed)
        assert np.max(np.abs(got - ref)) <= 1e-12, W
    # positions before the window may hold anything: they are never read
    k, v = inp.k.copy(), inp.v.copy()
    for b, T in enumerate(inp.seq_lens):
        k[b, :, :max(0, int(T) - 7)] = 0x7FC0   # bf16 NaN
        v[b, :, :max(0, int(T) - 7)] = 0x7FC0
    got = oracle.gqa_decode_f64(inp.q, k, v, inp.seq_lens, inp.scale, window=7, lib=lib)
    ref = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale, window=7, lib=lib)
    assert np.array_equal(got, ref)


def check_window_of_one_returns_last_value(lib):
    """W = 1: the only attended position is the newest, so out = v[T-1] bit for bit."""
    cfg = _small_cfg(G=2)
    inp = make_decode_inputs(cfg)
    got = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale, window=1, lib=lib)
    v = _f64(inp.v)
    for b, T in enumerate(inp.seq_lens):
        for i in range(cfg.H):
            assert np.array_equal(got[b, i], v[b, i // cfg.n, int(T) - 1])


def scatter_to_pages(caches, seq_lens, page_size, rng, extra_pages=3):
    """Numpy: contiguous caches [B,G,L,d] (K and V) cut into pages at random places of a pool.

    Returns one page pool per cache and the shared block table.  Unused pool
    pages and table entries past a sequence's pages are garbage (NaN bits and
    -1), which nothing may read.
    """
    B, G, L, d = caches[0].shape
    max_pages = -(-L // page_size)
    need = [-(-int(T) // page_size) for T in seq_lens]
    num_pages = sum(need) + extra_pages
    order = rng.permutation(num_pages)
    pools = [np.full((num_pages, G, page_size, d), 0x7FC0, dtype=np.uint16) for _ in caches]
    table = np.full((B, max_pages), -1, dtype=np.int32)
    nxt = 0
    for b in range(B):
        for p in range(need[b]):
            page = int(order[nxt])
            nxt += 1
            table[b, p] = page
            for pool, cache in zip(pools, caches):
                rows = cache[b, :, p * page_size:(p + 1) * page_size]
                pool[page, :, :rows.shape[1]] = rows
    return pools, table


def check_gather_inverts_scatter(lib):
    """Pages gathered through the block table give back the contiguous cache on every valid
    position, whatever the page size and the order of the pages in the pool; the paged
    decode (decode of the gathered cache) matches the library on the contiguous cache."""
    rng = np.random.default_rng(21)
    for page_size in (1, 4, 16, 64):
        cfg = _small_cfg(G=2, L=70, B=3, seq=(1, 70))
        inp = make_decode_inputs(cfg, seq_lens=[70, 33, 0], poison_tail=True)
        (kp, vp), table = scatter_to_pages([inp.k, inp.v], inp.seq_lens, page_size, rng)
        kg = oracle.gather_pages(kp, table, inp.seq_lens, cfg.Lmax, lib=lib)
        vg = oracle.gather_pages(vp, table, inp.seq_lens, cfg.Lmax, lib=lib)
        for b, T in enumerate(inp.seq_lens):
            assert np.array_equal(kg[b, :, :T], inp.k[b, :, :T]), (page_size, b)
            assert np.array_equal(vg[b, :, :T], inp.v[b, :, :T]), (page_size, b)
        a = oracle.gqa_decode_f64(inp.q, kg, vg, inp.seq_lens, inp.scale, lib=lib)
        ref = sdpa_reference(inp)
        assert np.max(np.abs(a - ref)) <= 1e-12
    bad = table.copy()
    bad[0, 0] = kp.shape[0]
    try:
        oracle.gather_pages(kp, bad, inp.seq_lens, cfg.Lmax, lib=lib)
    except ValueError:
        pass
    else:
        raise AssertionError("a table entry outside the pool was accepted")


def check_append_writes_one_row(lib):
    """The appended row lands at position T-1 of every K/V head of its sequence and nowhere
    else; the decode that follows attends to it as the newest position."""
    cfg = _small_cfg(G=2, L=23, B=4, seq=(1, 23))
    inp = make_decode_inputs(cfg, seq_lens=[23, 1, 0, 9], poison_tail=False)
    rng = np.random.default_rng(8)
    new = f32_to_bf16_bits(rng.standard_normal((cfg.B, cfg.G, cfg.d)).astype(np.float32))
    got = oracle.append_row(inp.k, new, inp.seq_lens, lib=lib)
    expect = inp.k.copy()
    for b, T in enumerate(inp.seq_lens):
        if T > 0:
            expect[b, :, T - 1] = new[b]
    assert np.array_equal(got, expect)
    # W = 1 after the append returns the appended value row exactly
    vnew = oracle.append_row(inp.v, new, inp.seq_lens, lib=lib)
    out = oracle.gqa_decode_f64(inp.q, got, vnew, inp.seq_lens, inp.scale, window=1, lib=lib)
    for b, T in enumerate(inp.seq_lens):
        for i in range(cfg.H):
            ref = _f64(new[b, i // cfg.n]) if T > 0 else np.zeros(cfg.d)
            assert np.array_equal(out[b, i], ref)


# ---------------------------------------------------------------- mean-pool

def check_meanpool_identical_heads(lib):
    """Mean-pooling G groups of identical heads returns that head.

    With 8 significant bits per value every partial sum j*x (j <= 16) is exact in
    fp32, so the result is exact; with full 24-bit values the running sum rounds
    and the result is within a few ulps.
    """
    for H, G in ((8, 2), (8, 4), (8, 1), (16, 2), (12, 4)):
        w1 = make_meanpool_input(G, G, 4, 32)
        short = bf16_bits_to_f32(f32_to_bf16_bits(w1))
        out = oracle.meanpool_f32(np.repeat(short, H // G, axis=0), H, G, lib=lib)
        assert np.array_equal(out, short)
        out = oracle.meanpool_f32(np.repeat(w1, H // G, axis=0), H, G, lib=lib)
        assert np.all(np.abs(out - w1) <= 4 * np.spacing(np.abs(w1)))


def check_meanpool_identity_and_mean(lib):
    """G = H is the identity; G = 1 is the head mean (within fp32 rounding of the sum)."""
    w = make_meanpool_input(8, 2, 64, 512)
    assert np.array_equal(oracle.meanpool_f32(w, 8, 8, lib=lib), w)
    m = oracle.meanpool_f64(w, 8, 1, lib=lib)[0]
    ref = w.astype(np.float64).mean(axis=0)
    assert np.max(np.abs(m - ref)) <= 1e-14
    m32 = oracle.meanpool_f32(w, 8, 1, lib=lib)[0]
    assert np.max(np.abs(m32 - ref)) <= 8 * np.finfo(np.float32).eps * np.max(np.abs(w))


def check_meanpool_small_integers(lib):
    """Hand-checkable: heads holding 1, 2, 3, 4 pool to 1.5 and 3.5 (G = 2) and 2.5 (G = 1)."""
    w = np.stack([np.full((2, 3), float(i + 1), dtype=np.float32) for i in range(4)])
    assert np.array_equal(oracle.meanpool_f32(w, 4, 2, lib=lib),
                          np.stack([np.full((2, 3), 1.5, np.float32), np.full((2, 3), 3.5, np.float32)]))
    assert np.array_equal(oracle.meanpool_f32(w, 4, 1, lib=lib), np.full((1, 2, 3), 2.5, np.float32))
    # three heads: (1 + 2) + 4 = 7, 7 / 3 rounded once in fp32
    w3 = np.stack([np.full((1, 1), x, np.float32) for x in (1.0, 2.0, 4.0)])
    assert oracle.meanpool_f32(w3, 3, 1, lib=lib)[0, 0, 0] == np.float32(7.0) / np.float32(3.0)


def check_meanpool_fp32_head_order(lib):
    """The fp32 sum runs in increasing head order, rounding after every addition.

    Heads holding 1e8, 1, -1e8, 1 (all exact in fp32; the spacing of fp32 values
    near 1e8 is 8): in head order 1e8 + 1 rounds to 1e8, + (-1e8) gives 0, + 1
    gives 1, and 1 / 4 = 0.25.  Summing in reverse gives 0 (1 - 1e8 rounds to
    -1e8), summing in pairs gives 0, and an exact (or float64) sum gives 0.5, so
    only the stated order reaches 0.25.  The float64 twin gives the exact 0.5.
    """
    w = np.array([1e8, 1.0, -1e8, 1.0], dtype=np.float32).reshape(4, 1, 1)
    assert oracle.meanpool_f32(w, 4, 1, lib=lib)[0, 0, 0] == np.float32(0.25)
    assert oracle.meanpool_f64(w, 4, 1, lib=lib)[0, 0, 0] == 0.5
    # the same four heads as the second group of two, behind a group of zeros
    w2 = np.concatenate([np.zeros((4, 1, 1), np.float32), w])
    got = oracle.meanpool_f32(w2, 8, 2, lib=lib)[:, 0, 0]
    assert got[0] == 0.0 and got[1] == np.float32(0.25)


def check_meanpool_pages_layout(lib):
    """The pages' [d_model, H*h] layout (head i = columns i*h..(i+1)*h-1) pools to
    [d_model, G*h], the transpose of the head-major result."""
    H, G, h, dm = 8, 2, 16, 48
    w_hm = make_meanpool_input(H, G, h, dm)               # [H, h, d_model]
    w_pages = np.ascontiguousarray(w_hm.transpose(2, 0, 1).reshape(dm, H * h))
    pooled_pages = oracle.meanpool_f32(w_pages.reshape(dm, H, h), H, G, head_axis=1, lib=lib)
    pooled_hm = oracle.meanpool_f32(w_hm, H, G, lib=lib)   # [G, h, d_model]
    assert np.array_equal(pooled_pages, pooled_hm.transpose(2, 0, 1))
    # pages' pseudocode: W_K_g = mean over members of the column block (float64 twin)
    ref = np.stack([w_pages[:, g * (H // G) * h:(g + 1) * (H // G) * h].reshape(dm, H // G, h)
                    .astype(np.float64).mean(axis=1) for g in range(G)], axis=1)
    got64 = oracle.meanpool_f64(w_pages.reshape(dm, H, h), H, G, head_axis=1, lib=lib)
    assert np.max(np.abs(got64 - ref)) <= 1e-14


DECODE_CHECKS = [
    check_mha_matches_library, check_mqa_matches_library, check_gqa_matches_library,
    check_replication_turns_gqa_into_mha, check_constant_keys_give_mean_of_v,
    check_single_token_returns_v0, check_two_token_closed_form, check_key_shift_invariance,
    check_permutation_invariance, check_bruteforce_high_precision, check_tail_is_never_read,
    check_empty_sequence_gives_zero,
]
VARIANT_CHECKS = [
    check_cross_attention_matches_library, check_window_matches_library_mask,
    check_window_of_one_returns_last_value, check_gather_inverts_scatter, check_append_writes_one_row,
]
MEANPOOL_CHECKS = [
    check_meanpool_identical_heads, check_meanpool_identity_and_mean,
    check_meanpool_small_integers, check_meanpool_pages_layout, check_meanpool_fp32_head_order,
]
