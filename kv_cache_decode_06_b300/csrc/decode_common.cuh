// Work decomposition shared by the decode kernels and the split-combine.
//
// Work unit: a tile of 128 (or, in the paired d = 64 layout, 256) consecutive
// cache positions of one (sequence b, K/V head g) pair, a "segment".  Segment
// s = b*G + g holds the tiles that meet the attended positions [t0_b, T_b) of
// sequence b: T_b = seq_lens[b] (Lmax when seq_lens is null), t0_b = T_b - window
// with a sliding window shorter than T_b, else 0.  Tile j of the segment covers
// positions [(j0_b + j) * tile, ...), j0_b = t0_b / tile.  All tiles of all
// segments form one list in (b, g, j) order, W tiles long.
//
// Static part.  The first Ws tiles are split evenly: CTA c of Pw = min(grid, Ws)
// takes the contiguous range [c*Ws/Pw, (c+1)*Ws/Pw), the same number of tiles
// (+-1) however ragged the lengths are; the grid is one wave.
//
// Dynamic part.  The last Wd = W - Ws tiles form a pool of chunks of `chunk`
// tiles that CTAs claim, once their static range is issued, with an atomic
// ticket: the memory bandwidth an SM gets varies by tens of percent, and the
// CTAs that stream faster take more chunks, so the grid finishes together.
// Every CTA makes exactly one failing claim; the one whose failing claim is the
// grid's last resets the ticket for the next call.  Only trailing sequences
// whose segments hold at most 16 chunks enter the pool, which bounds the pieces
// of a segment, and the pool never exceeds the workspace's capacity.
//
// A range (static or chunk) cuts segments into "pieces".  A piece that covers
// its whole segment is finished in place (out = acc / l).  Otherwise its
// partial softmax state (m, l, acc) goes to a workspace slot, and the
// split-combine kernel, which runs when the decode grid has completed, merges
// the pieces of every split segment, enumerating them from the split alone.
//
// Partial slots.  Static piece of segment s cut by CTA c: slot c + s.  This is
// one-to-one: if c < c' then every segment of c is <= every segment of c', so
// c + s = c' + s' with c < c' would need s > s'; these slots are below
// kMaxCtas + B*G.  Chunk j's p-th piece (a chunk of `chunk` tiles meets at most
// `chunk` segments): slot kMaxCtas + B*G + j*chunk + p.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace gqa {

constexpr int kTile = 128;          // tensor-map rows per tile (128 positions, or 128 position pairs)
constexpr int kBoxCols = 64;        // bf16 elements per 128-byte swizzled row
constexpr int kBoxBytes = kTile * 128;
constexpr int kMaxBatch = 1024;
constexpr int kMaxCtas = 1024;        // GQA_MAX_CTAS
constexpr int kChunk = 4;             // tiles per dynamic-pool chunk
constexpr int kPoolSegChunks = 16;    // longest segment (in chunks) that may enter the pool
constexpr int kPoolMinTilesPerCta = 64;   // tiles per CTA below which the split is static only

struct DecodeParams {
    const __nv_bfloat16 *q;   // [B, H, D]
    const int32_t *seq_lens;  // [B]; null: every sequence holds Lmax positions
    int window;               // > 0: attend to the last `window` positions only
    // paged cache (block_table non-null): the K/V tensor maps view a pool of
    // pages [num_pages, G, page_size, D]; row b of the table lists sequence b's pages
    const int32_t *block_table;   // [B, max_pages]
    int page_shift;               // log2(page_size)
    int max_pages, num_pages;
    // fused append (k_new non-null): the new token's K/V rows [B, G, D] replace
    // position T_b - 1 in the tiles read and are written to the cache (k_dst, v_dst:
    // the contiguous cache or the page pool)
    const __nv_bfloat16 *k_new, *v_new;
    __nv_bfloat16 *k_dst, *v_dst;
    int withhold_k;           // test-hooks build only: CTA 0 skips its K copy number withhold_k (-1: none)
    float *out;               // [B, H, D]
    unsigned int *flags;      // workspace flag word
    unsigned int *ticket;     // dynamic-pool claims (zero between calls)
    unsigned int *fails;      // failing claims (zero between calls)
    int dyn_cap;              // pool tiles the workspace has slots for (0: no pool)
    int tile_shift;           // log2(cache positions per tile): 7, or 8 for the paired d = 64 layout
    float *partials;          // slots of n*(D+2) floats: m[n], l[n], acc[n][D]
    int B, H, G, n, Lmax;
    float scale_log2;         // scale * log2(e): scores are kept in base-2 units
};

__device__ __forceinline__ int tiles_of(int seq, int shift) { return (seq + (1 << shift) - 1) >> shift; }

__device__ __forceinline__ int clamp_seq(int s, int Lmax) { return s < 0 ? 0 : (s > Lmax ? Lmax : s); }

// T_b: valid positions of sequence b, clamped into [0, Lmax].
__device__ __forceinline__ int seq_len_of(const DecodeParams &p, int b) {
    return p.seq_lens ? clamp_seq(__ldg(p.seq_lens + b), p.Lmax) : p.Lmax;
}

// t0_b: first attended position (sliding window), 0 without a window.
__device__ __forceinline__ int window_start(const DecodeParams &p, int T) {
    return (p.window > 0 && T > p.window) ? T - p.window : 0;
}

// Tiles of sequence b's segments: those meeting [t0_b, T_b).
__device__ __forceinline__ int segment_tiles(const DecodeParams &p, int T, int shift) {
    return tiles_of(T, shift) - (window_start(p, T) >> shift);
}

// Tile counts stay below 2^31 (kMaxBatch * heads * tiles per sequence), so the
// split arithmetic below avoids 64-bit divisions, which are long instruction
// sequences on the start-up path of every CTA.

// First tile of CTA c's static range: floor(c * W / P), 0 <= c <= P <= kMaxCtas.
__device__ __forceinline__ long long range_start(int c, long long W, int P) {
    const unsigned w = (unsigned)W, q = w / (unsigned)P, rem = w % (unsigned)P;
    return (long long)c * q + ((unsigned)c * rem) / (unsigned)P;   // c * rem < 2^20
}

// The CTA whose range holds tile t (0 <= t < W): floor(((t + 1) * P - 1) / W),
// from a single-precision estimate corrected with exact products.
__device__ __forceinline__ int cta_of_tile(long long t, long long W, int P) {
    const long long num = (t + 1) * P - 1;
    int c = (int)((float)num / (float)W);
    c = c < 0 ? 0 : (c > P - 1 ? P - 1 : c);
    while ((long long)(c + 1) * W <= num) ++c;
    while ((long long)c * W > num) --c;
    return c;
}

// The split of the W tiles between the static ranges and the dynamic pool.
struct WorkSplit {
    long long W, Ws;   // all tiles; statically split tiles
    int Pw;            // CTAs with a static range
    int nchunks;       // chunks in the pool (0: no dynamic part)
};

// grid = launched CTAs.  The pool takes a quarter of the tiles, at most
// `pool_max` (the short trailing segments) and `cap` (workspace slots), and only
// when there are at least kPoolMinTilesPerCta tiles per CTA: every chunk ends a
// piece (about a microsecond of pipeline drain), which pays only when the
// static ranges are long enough for per-SM bandwidth differences to add up to
// more than that.  cap = 0 disables it.
__device__ __forceinline__ WorkSplit make_split(long long W, int grid, long long pool_max, int cap) {
    WorkSplit w;
    w.W = W;
    long long Wd = 0;
    if (cap > 0 && W >= (long long)kPoolMinTilesPerCta * grid) {
        Wd = W / 4;
        if (Wd > pool_max) Wd = pool_max;
        if (Wd > cap) Wd = cap;
        Wd -= Wd % kChunk;
    }
    w.Ws = W - Wd;
    w.nchunks = (int)(Wd / kChunk);
    w.Pw = (int)(w.Ws < grid ? w.Ws : grid);
    return w;
}

struct Cursor {
    int b, g, j, tiles;
};

// prefix[b] = tiles of sequences 0..b-1, prefix[B] = total.
__device__ __forceinline__ Cursor cursor_at(long long u, const int *prefix, int B, int G) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((long long)G * prefix[mid] <= u) lo = mid; else hi = mid - 1;
    }
    Cursor c;
    c.b = lo;
    c.tiles = prefix[lo + 1] - prefix[lo];
    const int r = (int)(u - (long long)G * prefix[lo]);   // < G * tiles < 2^31
    c.g = r / c.tiles;
    c.j = r - c.g * c.tiles;
    return c;
}

__device__ __forceinline__ void cursor_next(Cursor &c, const int *prefix, int B, int G) {
    if (++c.j < c.tiles) return;
    c.j = 0;
    if (++c.g < G) return;
    c.g = 0;
    do { ++c.b; } while (c.b < B && prefix[c.b + 1] == prefix[c.b]);
    if (c.b < B) c.tiles = prefix[c.b + 1] - prefix[c.b];
}

// First tile of the cursor's segment in the tile list.
__device__ __forceinline__ long long segment_start(const Cursor &c, const int *prefix, int G) {
    return (long long)G * prefix[c.b] + (long long)c.g * c.tiles;
}

// Block-wide: clamps seq_lens into [0, Lmax] and writes the prefix sums of
// the segments' tile counts; with a flag word, CTA 0 records a clamp in it.
// `scratch` needs 33 ints; scratch[32] receives the last sequence whose
// segments are too long for the dynamic pool (-1 if none).  Ends with
// __syncthreads().
__device__ inline void build_prefix(const DecodeParams &p, int shift, int *prefix, int *scratch,
                                    unsigned int *flags) {
    const int tid = threadIdx.x, nth = blockDim.x, B = p.B;
    if (tid == 0) scratch[32] = -1;
    const int per = (B + nth - 1) / nth;
    const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
    int local = 0;
    bool bad = false;
    for (int b = b0; b < b1; ++b) {
        if (p.seq_lens) {
            const int s = __ldg(p.seq_lens + b);
            bad |= (s < 0 || s > p.Lmax);
        }
        local += segment_tiles(p, seq_len_of(p, b), shift);
    }
    // exclusive scan of `local` over the block
    const int lane = tid & 31, warp = tid >> 5, nwarps = (nth + 31) >> 5;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < nwarps; ++w) {
        const int x = scratch[w];
        if (w < warp) before += x;
        total += x;
    }
    int run = before + incl - local, last_long = -1;
    for (int b = b0; b < b1; ++b) {
        prefix[b] = run;
        const int tb = segment_tiles(p, seq_len_of(p, b), shift);
        run += tb;
        if (tb > kPoolSegChunks * kChunk) last_long = b;
    }
    if (last_long >= 0) atomicMax(scratch + 32, last_long);
    if (tid == 0) prefix[B] = total;
    if (bad && flags && blockIdx.x == 0) atomicOr(flags, 0x1u /* GQA_FLAG_SEQ_LEN_CLAMPED */);
    __syncthreads();
}

// Warp-wide version of build_prefix for the calling warp alone (no block
// barrier): lane l takes sequences [l*per, (l+1)*per).  *last_long receives the
// last sequence whose segments are too long for the dynamic pool (-1 if none).
// Ends with __syncwarp().
// tlen (nullable): receives T_b, the clamped sequence lengths.
__device__ inline void build_prefix_warp(const DecodeParams &p, int shift, int *prefix, int *last_long,
                                         unsigned int *flags, int *tlen) {
    const int lane = threadIdx.x & 31, B = p.B;
    const int per = (B + 31) >> 5;
    const int b0 = min(B, lane * per), b1 = min(B, b0 + per);
    int local = 0, ll = -1;
    bool bad = false;
    for (int b = b0; b < b1; ++b) {
        int T = p.Lmax;
        if (p.seq_lens) {
            const int sv = __ldg(p.seq_lens + b);
            bad |= (sv < 0 || sv > p.Lmax);
            T = clamp_seq(sv, p.Lmax);
        }
        const int tb = segment_tiles(p, T, shift);
        if (tlen) tlen[b] = T;
        prefix[b] = local;   // exclusive within this lane; offset below
        local += tb;
        if (tb > kPoolSegChunks * kChunk) ll = b;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const int before = incl - local;
    for (int b = b0; b < b1; ++b) prefix[b] += before;
    if (lane == 31) prefix[B] = incl;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ll = max(ll, __shfl_xor_sync(0xffffffffu, ll, o));
    if (lane == 0) *last_long = ll;
    if (__any_sync(0xffffffffu, bad) && flags && blockIdx.x == 0 && lane == 0)
        atomicOr(flags, 0x1u /* GQA_FLAG_SEQ_LEN_CLAMPED */);
    __syncwarp();
}

// Where a CTA keeps T_b beside the tile prefix: the prefix array's unused tail,
// when the batch leaves room for it (null otherwise).
__device__ __forceinline__ int *seq_len_array(int *prefix, int B) {
    return 2 * B + 1 <= kMaxBatch + 1 ? prefix + B + 1 : nullptr;
}

// Segments with no valid position get out = 0 (the empty sum).  CTA c takes
// sequences b with b % P == c.
template <int D>
__device__ void zero_empty_sequences(const DecodeParams &p, const int *prefix, int P, int tid, int nthreads) {
    for (int b = blockIdx.x; b < p.B; b += P) {
        if (prefix[b + 1] != prefix[b]) continue;
        float4 *o = reinterpret_cast<float4 *>(p.out + (size_t)b * p.H * D);
        for (int x = tid; x < p.H * D / 4; x += nthreads) o[x] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// Partial slot layout (floats): m[n] | l[n] | pad to a multiple of 4 | acc[n][D].
// The acc block starts 16-byte aligned so it can be read as float4.
__host__ __device__ constexpr int slot_acc_offset(int n) { return (2 * n + 3) & ~3; }
__host__ __device__ constexpr long long slot_floats(int n, int D) { return slot_acc_offset(n) + (long long)n * D; }

__device__ __forceinline__ float *slot_ptr(const DecodeParams &p, int slot, int D) {
    return p.partials + (size_t)slot * (size_t)slot_floats(p.n, D);
}

// Tiles after the last sequence too long for the pool (build_prefix's scratch[32]).
__device__ __forceinline__ long long pool_tail_tiles(const int *prefix, int B, int G, int last_long) {
    return (long long)G * (prefix[B] - prefix[last_long + 1]);
}

// Slot of the p-th piece of dynamic chunk j.
__device__ __forceinline__ int chunk_slot(const DecodeParams &p, int j, int piece) {
    return kMaxCtas + p.B * p.G + j * kChunk + piece;
}

// Slots of every piece of one segment, in tile order: `ns` static pieces in
// slots s0, s0 + 1, ..., then `nd` chunk pieces: d0 for the first, then
// d1, d1 + kChunk, d1 + 2 * kChunk, ... (later chunks start inside the segment,
// so their piece index is 0).
struct SegmentSlots {
    int ns, s0, nd, d0, d1;
    __device__ __forceinline__ int count() const { return ns + nd; }
    __device__ __forceinline__ int operator()(int k) const {
        if (k < ns) return s0 + k;
        k -= ns;
        return k == 0 ? d0 : d1 + (k - 1) * kChunk;
    }
};

// The pieces of segment s = b*G + g, which starts at tile a and holds T tiles.
__device__ __forceinline__ SegmentSlots segment_slots(const DecodeParams &p, const WorkSplit &w, const int *prefix,
                                                      int s, long long a, int T) {
    SegmentSlots r{0, 0, 0, 0, 0};
    const long long e = a + T;   // one past the last tile
    if (a < w.Ws) {
        const long long hi = (e < w.Ws ? e : w.Ws) - 1;
        const int c_lo = cta_of_tile(a, w.Ws, w.Pw), c_hi = cta_of_tile(hi, w.Ws, w.Pw);
        r.ns = c_hi - c_lo + 1;
        r.s0 = c_lo + s;
    }
    if (e > w.Ws) {
        const long long lo = a > w.Ws ? a : w.Ws;
        const int j_lo = (int)((lo - w.Ws) / kChunk), j_hi = (int)((e - 1 - w.Ws) / kChunk);
        // the segment's piece index in chunk j_lo = segments met in the chunk before
        // it (segment numbers skip empty sequences, so count them by walking)
        Cursor c0 = cursor_at(w.Ws + (long long)j_lo * kChunk, prefix, p.B, p.G);
        int p_lo = 0;
        while (c0.b * p.G + c0.g != s && p_lo < kChunk) {
            c0 = cursor_at(segment_start(c0, prefix, p.G) + c0.tiles, prefix, p.B, p.G);
            ++p_lo;
        }
        r.nd = j_hi - j_lo + 1;
        r.d0 = chunk_slot(p, j_lo, p_lo);
        r.d1 = chunk_slot(p, j_lo + 1, 0);
    }
    return r;
}

// 2^x with the hardware approximation (relative error ~2^-22); 2^-inf = +0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Synchronisation of the 128 compute threads through an mbarrier with a bounded
// wait, so an aborting CTA can never hang in it.
struct GroupSync {
    uint64_t *bar;
    uint32_t phase;
    __device__ bool operator()(const AbortState &ab) {
        mbar_arrive(bar);
        const bool ok = mbar_wait(bar, phase & 1u, ab);
        ++phase;
        return ok;
    }
};

}  // namespace gqa
