"""CPU check of the decode kernels' work split, written from the same rules.

The kernels give CTA c of Pw the static tiles [c*Ws/Pw, (c+1)*Ws/Pw) of the
(b, g, j)-ordered tile list and, for long lists, put the last Wd tiles in a
pool of 4-tile chunks that CTAs claim in any order.  Every range cuts segments
into pieces; a piece that is not a whole segment stores its partial state in a
slot (static: c + (b*G + g); chunk j: MAX_CTAS + B*G + j*4 + piece index).  The
split-combine kernel then merges every segment with two or more pieces,
enumerating their slots from the split alone.

This test replays those rules in Python for many shapes and claim orders and
checks that every tile is processed exactly once, slots are distinct and inside
the workspace, the merge's enumeration is exactly the set of slots written for
each split segment (in tile order), a segment with one piece is whole, and TMA
coordinates stay within the tensor map.
"""
import random

import pytest

MAX_CTAS = 1024
CHUNK = 4
POOL_SEG_CHUNKS = 16
MAX_DYN_TILES = 8192
POOL_MIN_TILES_PER_CTA = 64


def tiles_of(s, tile):
    return (s + tile - 1) // tile


def dyn_cap(B, G, Lmax):
    """Mirror of the host's pool capacity: a quarter of the most 128-position tiles, capped, whole chunks."""
    cap = min((B * G * tiles_of(Lmax, 128) + 3) // 4, MAX_DYN_TILES)
    return cap - cap % CHUNK


def make_split(W, grid, pool_max, cap):
    """Mirror of make_split: returns (Ws, Pw, nchunks)."""
    Wd = 0
    if cap > 0 and W >= POOL_MIN_TILES_PER_CTA * grid:
        Wd = min(W // 4, pool_max, cap)
        Wd -= Wd % CHUNK
    Ws = W - Wd
    return Ws, min(Ws, grid), Wd // CHUNK


def schedule(seq, G, grid, Lmax, tile=128, pool=True, rng=None):
    B = len(seq)
    tiles = [tiles_of(min(max(s, 0), Lmax), tile) for s in seq]
    prefix = [0]
    for t in tiles:
        prefix.append(prefix[-1] + t)
    W = G * prefix[B]
    last_long = max([b for b in range(B) if tiles[b] > POOL_SEG_CHUNKS * CHUNK], default=-1)
    pool_max = G * (prefix[B] - prefix[last_long + 1])
    cap = dyn_cap(B, G, Lmax) if pool else 0
    Ws, Pw, nchunks = make_split(W, grid, pool_max, cap)

    def cta_of_tile(t):
        return ((t + 1) * Pw - 1) // Ws

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

    def seg_start(c):
        return G * prefix[c[0]] + c[1] * c[3]

    def chunk_slot(j, p):
        return MAX_CTAS + B * G + j * CHUNK + p

    def segment_slots(s, a, T):
        """Mirror of segment_slots: the slots of segment s's pieces in tile order."""
        out = []
        e = a + T
        if a < Ws:
            hi = min(e, Ws) - 1
            out += [c + s for c in range(cta_of_tile(a), cta_of_tile(hi) + 1)]
        if e > Ws:
            lo = max(a, Ws)
            j_lo, j_hi = (lo - Ws) // CHUNK, (e - 1 - Ws) // CHUNK
            c0 = cursor_at(Ws + j_lo * CHUNK)
            p_lo = 0
            while c0[0] * G + c0[1] != s and p_lo < CHUNK:
                c0 = cursor_at(seg_start(c0) + c0[3])
                p_lo += 1
            out.append(chunk_slot(j_lo, p_lo))
            out += [chunk_slot(j, 0) for j in range(j_lo + 1, j_hi + 1)]
        return out

    # ranges: every CTA's static range, then the chunks, claimed in any order by any CTA
    ranges = []
    for c in range(min(grid, Pw)):
        u0, u1 = c * Ws // Pw, (c + 1) * Ws // Pw
        if u1 > u0:
            ranges.append((c, -1, u0, u1))
    for j in range(nchunks):
        ranges.append((rng.randrange(grid) if rng else j % grid, j, Ws + j * CHUNK, Ws + (j + 1) * CHUNK))
    if rng is not None:
        rng.shuffle(ranges)

    seen, slots, written, owned_segs = {}, {}, {}, set()
    for (c, j, u0, u1) in ranges:
        assert 0 <= u0 < u1 <= W
        cur = cursor_at(u0)
        piece_u0, range_piece = u0, 0
        for u in range(u0, u1):
            b, g, jj, tb = cur
            assert 0 <= b < B and 0 <= g < G and 0 <= jj < tb
            key = (b, g, jj)
            assert key not in seen
            seen[key] = (c, j)
            # TMA box: tensor-map row jj*128 of the segment, z = b*G+g
            assert 0 <= jj * tile < Lmax and 0 <= b * G + g < B * G
            first = (u == u0) or jj == 0
            last = (u + 1 == u1) or (jj + 1 == tb)
            if first:
                piece_u0 = u
            if last:
                seg = b * G + g
                if piece_u0 == seg_start(cur) and jj + 1 == tb:
                    owned_segs.add(seg)
                else:
                    slot = c + seg if j < 0 else chunk_slot(j, range_piece)
                    assert j < 0 or range_piece < CHUNK
                    assert slot not in slots and slot < MAX_CTAS + B * G + cap
                    slots[slot] = seg
                    written.setdefault(seg, []).append((piece_u0, slot))
                range_piece += 1
            cursor_next(cur)
    # every tile of every segment exactly once
    expect = {(b, g, jj) for b in range(B) for g in range(G) for jj in range(tiles[b])}
    assert set(seen) == expect
    # the combine kernel: each segment with two or more pieces is merged from exactly
    # its slots, in tile order; a segment with one piece was written whole
    for b in range(B):
        for g in range(G):
            T = tiles[b]
            if T == 0:
                continue
            s = b * G + g
            enum = segment_slots(s, G * prefix[b] + g * T, T)
            if len(enum) < 2:
                assert s in owned_segs and s not in written
            else:
                assert s not in owned_segs
                assert enum == [sl for _, sl in sorted(written[s])]
    # static work balance: ranges differ by at most one tile and none is empty
    if Pw:
        sizes = [(c + 1) * Ws // Pw - c * Ws // Pw for c in range(Pw)]
        assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1
    return Ws, nchunks


@pytest.mark.parametrize("seed", range(60))
def test_schedule_random(seed):
    rng = random.Random(seed)
    B = rng.choice([1, 2, 3, 7, 16, 64])
    G = rng.choice([1, 2, 8, 64])
    Lmax = rng.choice([1, 127, 128, 129, 1000, 4096, 20000])
    seq = [rng.choice([0, 0, 1, Lmax, rng.randint(0, Lmax)]) for _ in range(B)]
    if sum(seq) == 0:
        seq[0] = 1
    W = G * sum(tiles_of(s, 128) for s in seq)
    for P in {1, 2, 3, 148, max(1, min(1024, W)), min(1024, B * G * tiles_of(Lmax, 128))}:
        for tile in (128, 256):
            schedule(seq, G, P, Lmax, tile=tile, pool=True, rng=rng)
            schedule(seq, G, P, Lmax, tile=tile, pool=False)


def test_pool_sizes():
    """A quarter of the tiles goes to the pool when segments are short and there are >= 64 tiles per CTA."""
    Ws, nchunks = schedule([4096] * 80, 8, 148, 4096, rng=random.Random(1))   # 32-tile segments, 138 per CTA
    assert nchunks * CHUNK == 80 * 8 * 32 // 4 and Ws == 80 * 8 * 32 - nchunks * CHUNK
    _, nchunks = schedule([4096] * 16, 8, 148, 4096)                           # 27 tiles per CTA: static only
    assert nchunks == 0
    _, nchunks = schedule([100] * 4, 2, 148, 128)                              # too few tiles per CTA
    assert nchunks == 0
    # a long last sequence keeps the pool out of it
    _, nchunks = schedule([8192] * 8 + [64 * 128 + 1], 8, 8, 65 * 128, rng=random.Random(2))
    assert nchunks == 0


def test_failing_claims_reset_the_ticket():
    """Replay of the claim protocol: each CTA ends with one failing claim; the last resets."""
    for grid, nchunks in [(1, 1), (3, 5), (148, 128), (148, 1)]:
        rng = random.Random(grid + nchunks)
        ticket = fails = 0
        claimed, resets = [], 0
        active = list(range(grid))
        while active:
            c = rng.choice(active)
            j = ticket
            ticket += 1
            if j < nchunks:
                claimed.append(j)
            else:
                active.remove(c)
                f = fails
                fails += 1
                if f == grid - 1:
                    ticket = fails = 0
                    resets += 1
        assert sorted(claimed) == list(range(nchunks)) and resets == 1 and ticket == 0 and fails == 0


def test_schedule_workloads():
    from kv_cache_decode_06_b300.inputs import CONFIGS, draw_seq_lens
    pooled = {}
    for name in ("tiny", "mistral7b", "llama3_70b", "long_ragged"):
        c = CONFIGS[name]
        seq = draw_seq_lens(c).tolist()
        for pool in (True, False):
            _, nchunks = schedule(seq, c.G, 148, c.Lmax, pool=pool, rng=random.Random(7))
            if pool:
                pooled[name] = nchunks > 0
    # the short Mistral-7B step splits statically; the long Llama-3-70B one claims a pool
    assert pooled == {"tiny": False, "mistral7b": False, "llama3_70b": True, "long_ragged": True}
    c = CONFIGS["t5xxl_sweep"]
    for G in (1, 8, 64):
        schedule([c.Lmax] * c.B, G, 148, c.Lmax, tile=256, rng=random.Random(G))
