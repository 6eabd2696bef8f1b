"""CPU check of the decode kernels' work split, written from the same rules.

The kernels give CTA c of P the tiles [c*W/P, (c+1)*W/P) of the (b, g, j)-ordered
tile list, cut segments into pieces and store a piece's partial state in slot
c + (b*G + g); the split-combine kernel's CTA c merges the segment cut at the
start of decode CTA c's range when that is the segment's first cut.  This test
replays those rules in Python for many shapes and checks that every tile is
processed exactly once, slots are distinct and inside the workspace, every
split segment is merged exactly once from exactly its pieces, and TMA
coordinates stay within the tensor map.
"""
import random

import pytest

TILE = 128
MAX_CTAS = 1024


def tiles_of(s):
    return (s + TILE - 1) // TILE


def schedule(seq, G, P, Lmax):
    B = len(seq)
    tiles = [tiles_of(min(max(s, 0), Lmax)) for s in seq]
    prefix = [0]
    for t in tiles:
        prefix.append(prefix[-1] + t)
    W = G * prefix[B]
    P = min(P, W)       # only the first W CTAs take tiles

    def cta_of_tile(t):
        return ((t + 1) * P - 1) // W

    def cursor_at(u):
        lo, hi = 0, B - 1
        while lo < hi:
            mid = (lo + hi + 1) >> 1
            if G * prefix[mid] <= u:
                lo = mid
            else:
                hi = mid - 1
        tb = prefix[lo + 1] - prefix[lo]
        r = u - G * prefix[lo]
        return [lo, r // tb, r % tb, tb]

    def cursor_next(c):
        c[2] += 1
        if c[2] < c[3]:
            return
        c[2] = 0
        c[1] += 1
        if c[1] < G:
            return
        c[1] = 0
        c[0] += 1
        while c[0] < B and prefix[c[0] + 1] == prefix[c[0]]:
            c[0] += 1
        if c[0] < B:
            c[3] = prefix[c[0] + 1] - prefix[c[0]]

    seen = {}
    slots = {}
    pieces = {}
    for c in range(P):
        u0, u1 = c * W // P, (c + 1) * W // P
        if u0 >= u1:
            continue
        cur = cursor_at(u0)
        piece_u0 = u0
        for u in range(u0, u1):
            b, g, j, tb = cur
            assert 0 <= b < B and 0 <= g < G and 0 <= j < tb
            key = (b, g, j)
            assert key not in seen
            seen[key] = c
            # TMA box: y = j*128 in [0, Lmax), z = b*G+g in [0, B*G)
            assert 0 <= j * TILE < Lmax and 0 <= b * G + g < B * G
            first = (u == u0) or j == 0
            last = (u + 1 == u1) or (j + 1 == tb)
            if first:
                piece_u0 = u
            if last:
                seg = b * G + g
                seg_a = G * prefix[b] + g * tb
                owned = piece_u0 == seg_a and j + 1 == tb
                if not owned:
                    slot = c + seg
                    assert slot not in slots and slot < MAX_CTAS + B * G
                    slots[slot] = (c, seg)
                    pieces.setdefault(seg, []).append(c)
                    c_lo, c_hi = cta_of_tile(seg_a), cta_of_tile(seg_a + tb - 1)
                    assert c_lo <= c <= c_hi
            cursor_next(cur)
    # every tile of every segment exactly once
    expect = {(b, g, j) for b in range(B) for g in range(G) for j in range(tiles[b])}
    assert set(seen) == expect
    # shared segments: the pieces are exactly CTAs c_lo..c_hi
    for seg, cs in pieces.items():
        b, g = divmod(seg, G)
        seg_a = G * prefix[b] + g * tiles[b]
        c_lo, c_hi = cta_of_tile(seg_a), cta_of_tile(seg_a + tiles[b] - 1)
        assert sorted(cs) == list(range(c_lo, c_hi + 1)) and c_hi > c_lo
    # split-combine: CTA c merges the segment cut at the start of decode CTA c's
    # range when that is the segment's first cut; every split segment exactly once
    merged = {}
    for c in range(1, P):
        a = c * W // P
        b, g, j, tb = cursor_at(a)
        seg_a = G * prefix[b] + g * tb
        if seg_a == a or cta_of_tile(seg_a) != c - 1:
            continue
        seg = b * G + g
        assert seg not in merged
        merged[seg] = (cta_of_tile(seg_a), cta_of_tile(seg_a + tb - 1))
    assert set(merged) == set(pieces)
    for seg, (c_lo, c_hi) in merged.items():
        assert sorted(pieces[seg]) == list(range(c_lo, c_hi + 1))
    # work balance: ranges differ by at most one tile and none is empty
    sizes = [(c + 1) * W // P - c * W // P for c in range(P)]
    assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1


@pytest.mark.parametrize("seed", range(40))
def test_schedule_random(seed):
    rng = random.Random(seed)
    B = rng.choice([1, 2, 3, 7, 16, 64])
    G = rng.choice([1, 2, 8, 64])
    Lmax = rng.choice([1, 127, 128, 129, 1000, 4096])
    seq = [rng.choice([0, 1, Lmax, rng.randint(0, Lmax)]) for _ in range(B)]
    if sum(seq) == 0:
        seq[0] = 1
    W = G * sum(tiles_of(s) for s in seq)
    for P in {1, 2, 3, 148, max(1, min(1024, W)), min(1024, B * G * tiles_of(Lmax))}:
        schedule(seq, G, P, Lmax)


def test_schedule_workloads():
    from kv_cache_decode_06_b300.inputs import CONFIGS, draw_seq_lens
    for name in ("tiny", "mistral7b", "llama3_70b", "long_ragged"):
        c = CONFIGS[name]
        seq = draw_seq_lens(c).tolist()
        schedule(seq, c.G, 148, c.Lmax)
