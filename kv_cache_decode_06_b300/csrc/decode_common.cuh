// Work decomposition shared by the decode kernels and the split-combine.
//
// Work unit: a tile of 128 consecutive cache positions of one (sequence b,
// K/V head g) pair, a "segment".  Segment s = b*G + g holds
// tiles_b = ceil(seq_lens[b] / 128) tiles.  All tiles of all segments form one
// list in (b, g, j) order, W tiles long.  CTA c of P processes the contiguous
// range [c*W/P, (c+1)*W/P): every CTA gets the same number of tiles (+-1), however
// ragged the sequence lengths are, and the whole grid is one wave.  When there
// are fewer tiles than CTAs, only the first W CTAs take tiles (P = min(grid, W)),
// so no working range is empty.
//
// A CTA's range cuts segments into "pieces".  A piece that covers its whole
// segment is finished in place (out = acc / l).  Otherwise the piece's partial
// softmax state (m, l, acc) goes to a workspace slot, and the split-combine
// kernel, which runs when the decode grid has completed, merges the pieces of
// every split segment.  The decode kernel has no atomics, counters or fences.
//
// Partial slot of the piece of segment s cut by CTA c: slot = c + s.  This is
// one-to-one: if c < c' then every segment of c is <= every segment of c', so
// c + s = c' + s' with c < c' would need s > s'.  The pieces of segment s lie in
// slots c_lo + s .. c_hi + s, c_lo and c_hi the CTAs of its first and last tile.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace gqa {

constexpr int kTile = 128;          // cache positions per tile
constexpr int kBoxCols = 64;        // bf16 elements per 128-byte swizzled row
constexpr int kBoxBytes = kTile * 128;
constexpr int kMaxBatch = 1024;

struct DecodeParams {
    const __nv_bfloat16 *q;   // [B, H, D]
    const int32_t *seq_lens;  // [B]
    float *out;               // [B, H, D]
    unsigned int *flags;      // workspace flag word
    float *partials;          // slots of n*(D+2) floats: m[n], l[n], acc[n][D]
    int B, H, G, n, Lmax;
    float scale_log2;         // scale * log2(e): scores are kept in base-2 units
};

__device__ __forceinline__ int tiles_of(int seq) { return (seq + kTile - 1) / kTile; }

__device__ __forceinline__ int clamp_seq(int s, int Lmax) { return s < 0 ? 0 : (s > Lmax ? Lmax : s); }

__device__ __forceinline__ long long range_start(int c, long long W, int P) {
    return (long long)c * W / P;
}

// The CTA whose range holds tile t (0 <= t < W).
__device__ __forceinline__ int cta_of_tile(long long t, long long W, int P) {
    return (int)(((t + 1) * P - 1) / W);
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
    const long long r = u - (long long)G * prefix[lo];
    c.g = (int)(r / c.tiles);
    c.j = (int)(r % c.tiles);
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

// Block-wide: clamps seq_lens into [0, Lmax] and writes the tile prefix sums;
// with a flag word, CTA 0 records a clamp in it.  `scratch` needs 32 ints.
// Ends with __syncthreads().
__device__ inline void build_prefix(const int32_t *seq_lens, int B, int Lmax, int *prefix, int *scratch,
                             unsigned int *flags) {
    const int tid = threadIdx.x, nth = blockDim.x;
    const int per = (B + nth - 1) / nth;
    const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
    int local = 0;
    bool bad = false;
    for (int b = b0; b < b1; ++b) {
        const int s = __ldg(seq_lens + b);
        bad |= (s < 0 || s > Lmax);
        local += tiles_of(clamp_seq(s, Lmax));
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
    int run = before + incl - local;
    for (int b = b0; b < b1; ++b) {
        prefix[b] = run;
        run += tiles_of(clamp_seq(__ldg(seq_lens + b), Lmax));
    }
    if (tid == 0) prefix[B] = total;
    if (bad && flags && blockIdx.x == 0) atomicOr(flags, 0x1u /* GQA_FLAG_SEQ_LEN_CLAMPED */);
    __syncthreads();
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

// First tile of the cursor's segment in the tile list.
__device__ __forceinline__ long long segment_start(const Cursor &c, const int *prefix, int G) {
    return (long long)G * prefix[c.b] + (long long)c.g * c.tiles;
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
