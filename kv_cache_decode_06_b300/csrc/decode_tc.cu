// GQA decode on the fifth-generation tensor cores (tcgen05 + TMEM).
//
// The query heads of one group are one operand of two small GEMMs per tile, so
// every K/V tile read from HBM serves all n = H/G heads:
//   S^T [128 pos x N]  = K_tile [128 x d] . Q_g^T [d x N]            (K-major A and B)
//   O^T [M x kOW]      = V_tile^T [M x 128] . [P_hi; P_lo]^T          (MN-major A, K-major B)
// N is n rounded up to 16, 32 or 64 (the extra columns are never read).  The
// value GEMM stacks the probabilities' bf16 hi and lo parts (and, in the paired
// d = 64 layout, the even and odd positions) as column blocks of one GEMM, so
// the probabilities enter it with ~16 significant bits in 8 instructions per
// tile.  At 64 heads per group and d = 64 the heads are the GEMM rows instead
// (S = Q.K^T, O = P.V): one softmax thread then owns one head's scores.
// Operands come from 128-byte-swizzled shared memory written by TMA;
// accumulators live in TMEM.
// ["Grouped-query attention (GQA)" concept page, "Implementation sketch",
//  decode-step pseudocode; arxiv:2305.13245 §2.2]
//
// Warp roles (224 threads): warp 0 = TMA producer (Q, K, V; hands the work
// ranges to the others), warp 1 = score-GEMM issuer and TMEM owner, warp 6 =
// value-GEMM issuer, warps 2-5 = softmax + epilogue (thread <-> TMEM lane).
// Paged-cache instances (256 threads) add warp 7, which loads the block-table
// entries and copies K and V; the producer thread then issues only Q and hands
// out the work ranges.
//
// Producer and MMA issuers are event loops: each issues the next operation
// whose inputs are ready.  K slot s is handed back as soon as the score GEMM of
// its tile has read it, V slot s after the value GEMM.  Per tile the softmax group
//   1. loads its S row, reduces the per-head maximum over the tile's positions
//      (transposed butterfly in the warp, then the 4 warps via shared memory),
//   2. writes P(i) and hands it to the value-GEMM warp,
//   3. folds the O of the tile two steps back into register accumulators with
//      that tile's rescale factor (so TMEM never needs rescaling); O is triple
//      buffered in TMEM, so a value GEMM has two softmax steps to finish.
// Three instance families (kVar): the plain contiguous cache; the contiguous
// cache with a window or a fused append; the paged cache.  Each carries only its
// own producer code.  Work split and pieces are shared with the CUDA-core path
// (decode_common.cuh); pieces that are not a whole segment leave their partial
// state in the workspace for the split-combine kernel (combine.cu).
//
// Build with -DGQA_TRACE for a per-CTA timeline (clock64 stamps of the
// pipeline events, see the slot map at TraceSlot) readable with gqa_trace_copy.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "decode_common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

#ifdef GQA_TRACE
namespace gqa {
constexpr int kTraceSlots = 1024;
__device__ unsigned long long g_trace[1024 * kTraceSlots];
}  // namespace gqa
#define GQA_TRACE_AT(slot, value)                                                                         \
    do {                                                                                                  \
        if ((slot) < gqa::kTraceSlots)                                                                    \
            gqa::g_trace[(size_t)blockIdx.x * gqa::kTraceSlots + (slot)] = (unsigned long long)(value);  \
    } while (0)
extern "C" int gqa_trace_copy(void *dst, size_t bytes) {
    if (bytes > sizeof(gqa::g_trace)) bytes = sizeof(gqa::g_trace);
    return (int)cudaMemcpyFromSymbol(dst, gqa::g_trace, bytes);
}
#else
#define GQA_TRACE_AT(slot, value) \
    do {                          \
    } while (0)
#endif

namespace gqa {

namespace {

// Trace slots per CTA (clock64 unless noted).  Per-tile slots hold tiles 0..127.
enum TraceSlot {
    kTrGlobalStart = 0,   // %globaltimer at entry (ns)
    kTrStart = 1,         // entry
    kTrSetup = 2,         // barriers, TMEM and the tile prefix ready
    kTrEnd = 3,           // exit
    kTrTiles = 4,         // tiles of this CTA (a count)
    kTrGlobalEnd = 5,     // %globaltimer at exit (ns)
    kTrFirstQ = 6,        // first Q copy issued
    kTrFirstK = 7,        // first K copy issued
    kTrProdIn = 8,        // producer thread starts its loop
    kTrRing0 = 9,         // first range handed on
    kTrPreQ = 10,         // first Q copy about to be issued
    kTrDepDone = 11,      // the grids this one depends on have completed
    kTrKIssue = 16,       // + i: K copy of tile i issued
    kTrSIssue = 144,      // + i: score GEMM of tile i issued
    kTrPvIssue = 272,     // + i: value GEMM of tile i issued
    kTrVIssue = 400,      // + i: V(i) copy issued
    kTrProbe = 940,       // + 4i + {0,1,2,3}: K(i) copy call entered, returned; V(i) the same
    kTrKReady = 528,      // + i: the MMA issuer first sees K(i) landed
    kTrPFull = 656,       // + i: P(i) handed over
    kTrVReady = 784,      // + i: the MMA issuer first sees V(i) landed
    kTrPieceEnd = 912     // + 2k / + 2k + 1: start / end of the k-th piece epilogue
};

constexpr int kSmemLimit = 232448;   // 227 KB opt-in per CTA

constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }
constexpr int cmin(int a, int b) { return a < b ? a : b; }

constexpr int pow2_cols(int c) { return c <= 32 ? 32 : c <= 64 ? 64 : c <= 128 ? 128 : c <= 256 ? 256 : 512; }

constexpr int kRing = 4;   // work ranges in flight from the producer to the other roles

// Where a K or V slot's staged row (the appended token) goes: tile row `rel`
// (position T - 1 minus the tile's first position) and, when dst is not null,
// the cache row in global memory.
struct PatchInfo {
    __nv_bfloat16 *dst;
    int rel;
    int on;   // 0: nothing staged for this slot
};
static_assert(sizeof(PatchInfo) == 16, "PatchInfo layout");

// One work range (the static range or a claimed chunk) as the producer hands it on.
struct RangeEntry {
    long long ub;   // first tile
    int len;        // tiles
    int chunk;      // chunk id, -1 for the static range, -2 = no more work
};

// D = head dim, N = MMA N (>= 16), NH = heads held per thread (power of two >= n).
// kPair (D = 64 only): the cache is read as rows of two positions (256 bytes), a
// tile is 128 such rows = 256 positions in two column boxes (even positions,
// odd positions), and scores run as two GEMMs per tile, one per box.  A tile
// then moves as many bytes as a D = 128 tile, so the per-tile work of the
// softmax group is spread over twice the positions.
//
// The value GEMM is one M x kOW x 128 product per tile, whatever the layout.
// Its B operand stacks the probability rows [part][hi, lo][kNPV heads]; its A
// operand is V^T, with M = 128 rows (the two 64-dim boxes at D = 128; at
// kPair, box 0 = dims of the even positions, box 1 = dims of the odd ones) or
// M = 64 (D = 64, one box).  Row m of the result, column block (c, hi/lo),
// is wanted where part c matches the box of row m (always, without kPair);
// the other blocks are never read.  hi and lo land in separate columns and are
// added when O is folded; at kPair, rows m and m + 64 (even and odd positions
// of dim m) are added at the end of a piece.  One tcgen05.mma then covers
// 16 positions of every head, part and hi/lo half: 8 instructions per tile.
// kVar: 0 = plain instance (contiguous cache, every valid position); 1 = the
// contiguous-cache variants (sliding window, fused append); 2 = paged cache (with
// or without window and append).  Each instance carries only its own code and
// staging: the producer's loop must stay short (instruction fetch misses on a
// long loop cost it hundreds of nanoseconds per tile).
template <int D, bool kPair, int N, int NH, int kVar = 0>
struct TcCfg {
    static constexpr bool kExt = kVar != 0;
    static constexpr bool kPaged = kVar == 2;
    static_assert(!kPair || D == 64, "the paired layout is for D = 64");
    static constexpr int kColBoxes = (D == 128 || kPair) ? 2 : 1;   // 64-column boxes per tile row
    static constexpr int kQBoxes = D / kBoxCols;                     // 64-column boxes per q row
    static constexpr int kParts = kPair ? 2 : 1;                     // score GEMMs per tile
    static constexpr int kTileShift = kPair ? 8 : 7;                 // log2(positions per tile)
    static constexpr int kTilePos = 1 << kTileShift;
    static constexpr int kTileBytes = kColBoxes * kBoxBytes;         // one K or V tile
    // K/V tile layout in shared memory: tensor-map row r, column box c at
    // c * kHalfStride + (r / 8) * kGroupStride + (r % 8) * 128, 128-byte swizzled
    // within each 8-row group.  Whole-tile layout: the column boxes one after the
    // other (16 KB apart), the 8-row groups dense.  Paged instances with two
    // column boxes interleave them per 8-row group ([group][box][8 rows][128 B]):
    // a page of the pool is then one TMA box (a five-dimensional tensor map) that
    // lands as whole groups, whatever the page size, and the tensor cores read the
    // same tile through descriptors with these strides.
    static constexpr bool kInter = kPaged && kColBoxes == 2;
    static constexpr int kHalfStride = kInter ? 1024 : kBoxBytes;
    static constexpr int kGroupStride = kInter ? 2048 : 1024;
    static __device__ __forceinline__ int row_off(int r) { return (r >> 3) * kGroupStride + (r & 7) * 128; }
    // heads on M (64 query heads per group at d = 64), see below: Q is stored twice, as
    // the 128 rows of the score GEMM's A operand
    static constexpr bool kHM = (D == 64 && NH == 64 && !kPair);
    static constexpr int kQBytes = kQBoxes * N * 128 * (kHM ? 2 : 1);   // one Q buffer (N rows x d)
    // rows of one (part, hi/lo) block of the value GEMM's B operand: the heads,
    // padded to 8 (the value GEMM's N = kOW stays a multiple of 16)
    static constexpr int kNPV = NH <= 8 ? 8 : N;
    static constexpr int kOW = 2 * kParts * kNPV;                    // value GEMM N: [part][hi, lo][kNPV]
    static constexpr int kPBufBytes = 2 * kOW * 128;                 // one P buffer: [64-position half][kOW rows]
    // small shared state, in floats
    static constexpr int kRedF = 2 * 4 * NH;                     // [2][4 warps][NH] tile maxima
    static constexpr int kLredF = 4 * NH;                        // [4 warps][NH] l sums
    static constexpr int kMF = 3 * NH;                           // [3][NH] running max after tile i
    static constexpr int kAF = 4 * NH;                           // [4][NH] rescale factor of tile i
    static constexpr int kSmallBytes = 4 * (kRedF + kLredF + kMF + kAF) + 33 * 4 + (kMaxBatch + 1) * 4 + kRing * 16;
    static constexpr int bar_bytes(int SK, int SV, int QB) { return (2 * SK + 2 * SV + 2 * QB + 14 + 2 + 2 * kRing + 1) * 8 + 16; }
    static constexpr int fixed_bytes(int QB) {
        return QB * kQBytes + 2 * kPBufBytes + kSmallBytes + bar_bytes(8, 8, QB) + kIdBytes + kIdBars * 8 +
               1024 /* alignment slack */;
    }
    // Per K or V slot, beside the tile: the appended token's row as copied from
    // global memory, and where it goes (fused append; unused otherwise).
    static constexpr int kRowBytes = D * 2;
    static constexpr int kStageRow = kExt ? kRowBytes : 0;
    static constexpr int kStageInfo = kExt ? (int)sizeof(PatchInfo) : 0;
    static constexpr int kSlotCost = kTileBytes + kStageRow + kStageInfo;
    // page-id ring (paged cache): kIdRing entries of kIdStride ints, the page ids of
    // one tile's pages followed by T_b, written by the page-id warp; an entry
    // completes once the warp has issued the tile's K copy, and is free again once
    // the producer thread has taken it
    static constexpr int kIdRing = 8;
    static constexpr int kIdMax = kTilePos / 16;        // pages per tile at the smallest page (16 positions)
    static constexpr int kIdStride = kIdMax + 4;        // ids, T_b, padding to 16 bytes
    static constexpr int kIdBytes = kPaged ? kIdRing * kIdStride * 4 : 0;
    static constexpr int kIdBars = kPaged ? 2 * kIdRing : 0;
    // K and V rings: as deep as shared memory allows (at most 8), V one deeper when
    // a single extra tile still fits (V slots are held until the value GEMM is done)
    static constexpr int avail(int QB) { return kSmemLimit - fixed_bytes(QB); }
    static constexpr int pairs_for(int QB) { return cmin(8, avail(QB) / (2 * kSlotCost)); }
    static constexpr int kQBuf = pairs_for(2) >= 3 || pairs_for(1) == pairs_for(2) ? 2 : 1;
    static constexpr int kSK = pairs_for(kQBuf);
    static constexpr int kSV = (kSK < 8 && avail(kQBuf) - 2 * kSK * kSlotCost >= kSlotCost) ? kSK + 1 : kSK;
    static_assert(kSK >= 2, "shared memory too small for two stages");
    // P buffers: three when they fit beside the rings (the softmax then waits for the
    // value GEMM three tiles back before reusing one), else two
    static constexpr int layout_bytes(int pbuf) {
        return (kSK + kSV) * kSlotCost + kQBuf * kQBytes + pbuf * kPBufBytes + kSmallBytes + 8 +
               (2 * kSK + 2 * kSV + 2 * kQBuf + 12 + pbuf + 2 + 2 * kRing + kIdBars + 1) * 8 + 16 + 1024 + kIdBytes;
    }
    static constexpr int kPBuf = layout_bytes(3) <= kSmemLimit ? 3 : 2;
    // layout (offsets from the 1024-aligned base)
    static constexpr int kOffK = 0;                                       // [SK] K tiles
    static constexpr int kOffV = kSK * kTileBytes;                        // [SV] V tiles
    static constexpr int kOffQ = kOffV + kSV * kTileBytes;                // [QB] Q buffers
    static constexpr int kOffP = kOffQ + kQBuf * kQBytes;                 // [PB buffers][part][hi, lo]
    static constexpr int kOffRed = kOffP + kPBuf * kPBufBytes;
    static constexpr int kOffLred = kOffRed + kRedF * 4;
    static constexpr int kOffM = kOffLred + kLredF * 4;
    static constexpr int kOffA = kOffM + kMF * 4;
    static constexpr int kOffPrefix = kOffA + kAF * 4;                    // i32 [kMaxBatch + 1]
    static constexpr int kOffScratch = kOffPrefix + (kMaxBatch + 1) * 4;  // i32 [33]
    static constexpr int kOffRing = (kOffScratch + 33 * 4 + 15) / 16 * 16;  // RangeEntry [kRing]
    static constexpr int kOffStage = kOffRing + kRing * 16;                 // [SK + SV] appended rows
    static constexpr int kOffPatch = kOffStage + (kSK + kSV) * kStageRow;   // PatchInfo [SK + SV]
    static constexpr int kOffIds = kOffPatch + (kSK + kSV) * kStageInfo;     // int [kIdRing][kIdStride]
    static constexpr int kOffBar = kOffIds + kIdBytes;
    // barriers: kfull[SK] kempty[SK] vfull[SV] vempty[SV] qfull[QB] qempty[QB] sfull[2] sfree[2]
    //           pfull[PB] ofull[3] ofree[3] red[2] grp done rfull[kRing] rempty[kRing]
    //           (paged) idfull[kIdRing] idempty[kIdRing]; pre
    static constexpr int kNumBars = 2 * kSK + 2 * kSV + 2 * kQBuf + 12 + kPBuf + 2 + 2 * kRing + kIdBars + 1;
    static constexpr int kOffFlags = kOffBar + kNumBars * 8;     // abort, tmem base
    static constexpr int kSmemBytes = kOffFlags + 16 + 1024;
    static_assert(kSmemBytes <= kSmemLimit, "shared memory layout too large");
    static_assert(NH < 4 || (kOffRed % 16 == 0 && kOffLred % 16 == 0 && kOffM % 16 == 0 && kOffA % 16 == 0),
                  "float4 alignment");
    // warps: producer, score MMA, 4 softmax, value MMA, and (paged instances) the
    // page-id warp, which copies K and V
    static constexpr int kThreads = kPaged ? 256 : 224;
    // TMEM: S accumulators [2][part][N] then O accumulators [3][kOW] (O is folded two tiles behind)
    // Heads on M (64 query heads per group at d = 64): the score GEMM is S = [Q; Q]·K^T
    // with the 64 heads twice as its 128 rows and the tile's 128 positions as
    // columns; TMEM lane r holds head r % 64, and its thread takes positions
    // 64 * (r / 64) .. + 63, so two threads share a head and every lane works.  The
    // value GEMM is O = P·V (P: [heads][positions], K-major, A operand; V: B
    // operand, MN-major), O [64 heads][d] in TMEM (M = 64: 16 lanes per quadrant).
    // P buffer: hi then lo, each two 64-position halves of 64 rows x 128 bytes (the
    // same 32 KB as otherwise).
    static constexpr int kOCol = kHM ? 2 * kTile : 2 * kParts * N;   // S buffers first
    static constexpr int kOBuf = kHM ? D : kOW;                      // columns of one O buffer
    static constexpr int kTmemCols = pow2_cols(kOCol + 3 * kOBuf);
    static_assert(kOCol + 3 * kOBuf <= 512, "TMEM columns");
    static_assert(!kHM || kPBufBytes == 2 * 2 * 64 * 128, "heads-on-M P buffer");
    static constexpr int kPvM = kHM ? 64 : kPair ? 128 : D;
    static_assert(kOW % 16 == 0 && kOW <= 256, "value GEMM N");
    static_assert(!kPair || NH * 64 * 4 <= kPBufBytes, "piece-end exchange fits a P buffer");
    // butterfly: number of head-halving steps (the rest are plain reductions)
    static constexpr int kHalve = ilog2(NH) < 5 ? ilog2(NH) : 5;
};

// Reduce v[0..NH) over the 32 lanes of the warp, head by head, with ~NH shuffles
// instead of 5*NH: each step hands half of the remaining heads to the partner
// lane.  Afterwards lane l holds, in v[j] (j < NH >> kHalve), the full reduction
// of head (prefix(l) * (NH >> kHalve) + j), prefix(l) = l's top kHalve bits.
template <int NH, bool kMax>
__device__ __forceinline__ void butterfly_reduce(float (&v)[NH], int lane) {
#pragma unroll
    for (int s = 0; s < 5; ++s) {
        const int o = 16 >> s;
        const int k = NH >> s;
        if (k >= 2) {
            const bool upper = (lane & o) != 0;
#pragma unroll
            for (int j = 0; j < k / 2; ++j) {
                const float send = upper ? v[j] : v[j + k / 2];
                const float keep = upper ? v[j + k / 2] : v[j];
                const float recv = __shfl_xor_sync(0xffffffffu, send, o);
                v[j] = kMax ? fmaxf(keep, recv) : keep + recv;
            }
        } else {
            const float recv = __shfl_xor_sync(0xffffffffu, v[0], o);
            v[0] = kMax ? fmaxf(v[0], recv) : v[0] + recv;
        }
    }
}

// After butterfly_reduce: store this warp's per-head results to dst[NH] (one
// writer lane per head).
template <int NH, int kHalve>
__device__ __forceinline__ void butterfly_store(const float (&v)[NH], int lane, float *dst) {
    constexpr int kPer = NH >> kHalve;
    const int low_bits = 5 - kHalve;
    if ((lane & ((1 << low_bits) - 1)) == 0) {
        const int prefix = lane >> low_bits;
#pragma unroll
        for (int j = 0; j < kPer; ++j) dst[prefix * kPer + j] = v[j];
    }
}

// out[h] = op(src[0*NH + h], src[1*NH + h], src[2*NH + h], src[3*NH + h]) for the
// four warps' per-head values, read as float4 where NH allows.
// kStride: distance between the warps' rows (NH, or the full head count when
// reducing a chunk of heads).
template <int NH, bool kMax, int kStride = NH>
__device__ __forceinline__ void reduce4(const float *src, float (&out)[NH]) {
    if constexpr (NH >= 4) {
#pragma unroll
        for (int h = 0; h < NH; h += 4) {
            const float4 a = *reinterpret_cast<const float4 *>(src + h);
            const float4 b = *reinterpret_cast<const float4 *>(src + kStride + h);
            const float4 c = *reinterpret_cast<const float4 *>(src + 2 * kStride + h);
            const float4 d = *reinterpret_cast<const float4 *>(src + 3 * kStride + h);
            if (kMax) {
                out[h] = fmaxf(fmaxf(a.x, b.x), fmaxf(c.x, d.x));
                out[h + 1] = fmaxf(fmaxf(a.y, b.y), fmaxf(c.y, d.y));
                out[h + 2] = fmaxf(fmaxf(a.z, b.z), fmaxf(c.z, d.z));
                out[h + 3] = fmaxf(fmaxf(a.w, b.w), fmaxf(c.w, d.w));
            } else {
                out[h] = (a.x + b.x) + (c.x + d.x);
                out[h + 1] = (a.y + b.y) + (c.y + d.y);
                out[h + 2] = (a.z + b.z) + (c.z + d.z);
                out[h + 3] = (a.w + b.w) + (c.w + d.w);
            }
        }
    } else {
#pragma unroll
        for (int h = 0; h < NH; ++h) {
            const float a = src[h], b = src[kStride + h], c = src[2 * kStride + h], d = src[3 * kStride + h];
            out[h] = kMax ? fmaxf(fmaxf(a, b), fmaxf(c, d)) : (a + b) + (c + d);
        }
    }
}

template <int NH>
__device__ __forceinline__ void load_vec(const float *src, float (&out)[NH]) {
    if constexpr (NH >= 4) {
#pragma unroll
        for (int h = 0; h < NH; h += 4) {
            const float4 a = *reinterpret_cast<const float4 *>(src + h);
            out[h] = a.x;
            out[h + 1] = a.y;
            out[h + 2] = a.z;
            out[h + 3] = a.w;
        }
    } else {
#pragma unroll
        for (int h = 0; h < NH; ++h) out[h] = src[h];
    }
}

template <int NH>
__device__ __forceinline__ void store_vec(float *dst, const float (&v)[NH]) {
    if constexpr (NH >= 4) {
#pragma unroll
        for (int h = 0; h < NH; h += 4)
            *reinterpret_cast<float4 *>(dst + h) = make_float4(v[h], v[h + 1], v[h + 2], v[h + 3]);
    } else {
#pragma unroll
        for (int h = 0; h < NH; ++h) dst[h] = v[h];
    }
}

// A page id read from the block table, or (flagged) one past the pool when it
// is not a page of the pool: the tensor map then fills the rows with zeros.
__device__ __noinline__ void flag_bad_page(const DecodeParams &p) { atomicOr(p.flags, 0x4u /* GQA_FLAG_BAD_PAGE */); }

__device__ __forceinline__ int checked_page(const DecodeParams &p, int page) {
    if (page >= 0 && page < p.num_pages) return page;
    flag_bad_page(p);
    return p.num_pages;
}

// The producer's copy of T_b for the sequence its cursor is in: one load per
// sequence, and none at all for a contiguous cache without window or append.
struct SeqLenCache {
    int b = -1, T = 0;
    __device__ __forceinline__ int get(const DecodeParams &p, int bb) {
        if (bb != b) {
            b = bb;
            T = seq_len_of(p, bb);
        }
        return T;
    }
};

// First cache position of tile j of a segment of sequence length T.
template <class C>
__device__ __forceinline__ int tile_first_pos(const DecodeParams &p, int T, int j) {
    return ((window_start(p, T) >> C::kTileShift) + j) << C::kTileShift;
}

// Producer, variant instances: copies the K or V tile at cursor c (sequence
// length T) into `dst`, completing on `bar`.  Contiguous cache: one box per
// column box at the tile's first row.  Paged cache (ids: the tile's page ids in
// shared memory, from the page-id warp): one box per column box from the page
// holding the tile, or one per page of the tile, skipping pages without an
// attended position (id -1; their rows are masked).  With an appended row
// for the tile (row_new: the tile holds position T - 1), the row is copied
// beside the tile and `info` says where it goes; `info` is written before the
// arrival that publishes it.
template <class C>
__device__ __noinline__ void produce_tile(const DecodeParams &p, const CUtensorMap *tm, uint8_t *dst, uint64_t *bar,
                                             const Cursor &c, int T, uint64_t pol, const __nv_bfloat16 *row_new,
                                             uint8_t *stage_row, PatchInfo *info, __nv_bfloat16 *row_dst,
                                             const int *ids) {
    constexpr int kPairShift = C::kParts - 1;   // tensor-map rows hold 2 positions in the paired layout
    const int seg = c.b * p.G + c.g;
    const int pos0 = tile_first_pos<C>(p, T, c.j);
    const int ps = 1 << p.page_shift;
    const bool app = row_new != nullptr && c.j + 1 == c.tiles;
    uint32_t bytes = 0;
    if (app) {
        __nv_bfloat16 *d = nullptr;
        if (!ids) {
            d = row_dst + ((size_t)seg * p.Lmax + (T - 1)) * (C::kRowBytes / 2);
        } else {
            const int page = ids[ps >= C::kTilePos ? 0 : ((T - 1 - pos0) >> p.page_shift)];   // page of T-1
            if (page >= 0 && page < p.num_pages)
                d = row_dst + (((size_t)page * p.G + c.g) * (size_t)ps + ((T - 1) & (ps - 1))) * (C::kRowBytes / 2);
        }
        info->dst = d;
        info->rel = T - 1 - pos0;
        bytes = C::kRowBytes;
    }
    info->on = app ? 1 : 0;
    if (!ids) {
        mbar_arrive_expect_tx(bar, bytes + C::kTileBytes);
#pragma unroll
        for (int cb = 0; cb < C::kColBoxes; ++cb)
            tma_load_3d(dst + cb * kBoxBytes, tm, cb * kBoxCols, pos0 >> kPairShift, seg, bar, pol);
    } else if (ps >= C::kTilePos) {
        const int z = checked_page(p, ids[0]) * p.G + c.g;
        const int y = (pos0 & (ps - 1)) >> kPairShift;
        mbar_arrive_expect_tx(bar, bytes + C::kTileBytes);
        if constexpr (C::kInter) {
            tma_load_5d(dst, tm, 0, 0, 0, y >> 3, z, bar, pol);
        } else {
#pragma unroll
            for (int cb = 0; cb < C::kColBoxes; ++cb) tma_load_3d(dst + cb * kBoxBytes, tm, cb * kBoxCols, y, z, bar, pol);
        }
    } else {
        const int prow = ps >> kPairShift;   // tensor-map rows per page
        // compact loops: this code runs from the instruction cache beside the
        // other roles' loops, and a long unrolled body costs more in fetch misses
        // than the loop overhead
        const int nb = C::kTilePos / ps;
        int loads = 0;
#pragma unroll 1
        for (int k = 0; k < nb; ++k) loads += ids[k] != -1;
        mbar_arrive_expect_tx(bar, bytes + (uint32_t)(loads * prow * 128 * C::kColBoxes));
#pragma unroll 1
        for (int k = 0; k < nb; ++k) {
            const int id = ids[k];
            if (id != -1) {
                const int z = checked_page(p, id) * p.G + c.g;
                if constexpr (C::kInter) {
                    tma_load_5d(dst + C::row_off(k * prow), tm, 0, 0, 0, 0, z, bar, pol);
                } else {
#pragma unroll
                    for (int cb = 0; cb < C::kColBoxes; ++cb)
                        tma_load_3d(dst + cb * kBoxBytes + k * prow * 128, tm, cb * kBoxCols, 0, z, bar, pol);
                }
            }
        }
    }
    if (app) bulk_load(stage_row, row_new + (size_t)seg * (C::kRowBytes / 2), C::kRowBytes, bar);
}

// Producer, plain instances: contiguous cache, every valid position: tile j of
// segment b*G + g is tensor-map rows j*128 .. (j0: the segment's first tile,
// nonzero only with a window).
template <class C>
__device__ __forceinline__ void produce_plain_tile(const DecodeParams &p, const CUtensorMap *tm, uint8_t *dst,
                                                   uint64_t *bar, const Cursor &c, uint64_t pol, int j0 = 0) {
    mbar_arrive_expect_tx(bar, C::kTileBytes);
#pragma unroll
    for (int cb = 0; cb < C::kColBoxes; ++cb)
        tma_load_3d(dst + cb * kBoxBytes, tm, cb * kBoxCols, (j0 + c.j) * kTile, c.b * p.G + c.g, bar, pol);
}

// The last tile of a segment, `rows` tensor-map rows of it (a multiple of 16 below
// 128): boxes of 64, 32 and 16 rows from the tail maps, each at its place in the
// slot (multiples of 16 rows keep the 128-byte swizzle pattern of a whole tile).
// The slot's rows past `rows` keep older data; the softmax masks those positions
// of K and clears those rows of V, as for any position past the sequence.
template <class C>
__device__ __noinline__ void produce_tail_tile(const DecodeParams &p, const CUtensorMap *tails, uint8_t *dst,
                                               uint64_t *bar, const Cursor &c, uint64_t pol, int rows) {
    mbar_arrive_expect_tx(bar, (uint32_t)(rows * 128 * C::kColBoxes));
    int r0 = 0;
#pragma unroll
    for (int t = 0; t < 3; ++t) {
        const int h = 64 >> t;
        if (rows & h) {
#pragma unroll
            for (int cb = 0; cb < C::kColBoxes; ++cb)
                tma_load_3d(dst + cb * kBoxBytes + r0 * 128, tails + t, cb * kBoxCols, c.j * kTile + r0,
                            c.b * p.G + c.g, bar, pol);
            r0 += h;
        }
    }
}

// Tensor-map rows of tile c.j worth loading: all 128, or for a segment's last tile
// the rows holding attended positions, rounded up to 16 (tlen: T_b per sequence,
// null when the batch leaves no room for it).
template <class C>
__device__ __forceinline__ int plain_tile_rows(const Cursor &c, const int *tlen) {
    if (!tlen || c.j + 1 != c.tiles) return kTile;
    const int rem = tlen[c.b] - (c.j << C::kTileShift);   // attended positions in the tile, >= 1
    const int rows = C::kParts == 2 ? (rem + 1) >> 1 : rem;
    return (rows + 15) & ~15;
}

// Producer, contiguous-cache variant instances: tiles without an appended row stay
// on a short inline path (the plain copy at the window's offset); the tile holding
// an appended row goes to produce_tile, out of line.  Short hot code matters here:
// the long general path costs several hundred nanoseconds per call in instruction
// fetches.
template <class C>
__device__ __forceinline__ void produce_variant_tile(const DecodeParams &p, const CUtensorMap *tm, uint8_t *dst,
                                                     uint64_t *bar, const Cursor &c, int T, uint64_t pol,
                                                     const __nv_bfloat16 *row_new, uint8_t *stage_row,
                                                     PatchInfo *info, __nv_bfloat16 *row_dst) {
    static_assert(!C::kPaged, "the page-id warp copies the tiles of a paged cache");
    if (row_new == nullptr || c.j + 1 != c.tiles) {
        if (row_new) info->on = 0;
        produce_plain_tile<C>(p, tm, dst, bar, c, pol, window_start(p, T) >> C::kTileShift);
        return;
    }
    produce_tile<C>(p, tm, dst, bar, c, T, pol, row_new, stage_row, info, row_dst, nullptr);
}

// Page-id warp, paged cache: copies the K or V tile at cursor c with the whole warp.
// Lane k holds the page id of the tile's page k (`id`; -1 for a page without an
// attended position, whose rows are masked) and `ids` the same ids in shared
// memory.  Each lane issues one box: page lane / kColBoxes, column box lane %
// kColBoxes (at most 16 pages of 16 positions x 2 column boxes per tile), so the
// copy of a tile of small pages costs one issue slot instead of one per box; a
// box's issue cost in a single thread, not the copy engine, bounds small pages.
// Lane 0 sets the byte count before any lane issues.  The tile holding an
// appended row goes to produce_tile on lane 0.
template <class C>
__device__ __forceinline__ void produce_paged_tile(const DecodeParams &p, const CUtensorMap *tm, uint8_t *dst,
                                                   uint64_t *bar, const Cursor &c, int T, uint64_t pol, int id,
                                                   int lane, const __nv_bfloat16 *row_new, uint8_t *stage_row,
                                                   PatchInfo *info, __nv_bfloat16 *row_dst, const int *ids) {
    static_assert(C::kIdMax * C::kColBoxes <= 32, "one box per lane");
    constexpr int kPairShift = C::kParts - 1;
    if (row_new != nullptr && c.j + 1 == c.tiles) {
        if (lane == 0) produce_tile<C>(p, tm, dst, bar, c, T, pol, row_new, stage_row, info, row_dst, ids);
        __syncwarp();
        return;
    }
    const int ps = 1 << p.page_shift;
    const bool whole = ps >= C::kTilePos;                   // one page holds the tile
    const int nb = whole ? 1 : C::kTilePos / ps;            // pages of the tile
    const int rows = whole ? kTile : ps >> kPairShift;      // tensor-map rows per box
    const unsigned loads = __ballot_sync(0xffffffffu, lane < nb && id != -1);
    if (lane == 0) {
        if (row_new) info->on = 0;   // before the arrival that publishes it
        mbar_arrive_expect_tx(bar, (uint32_t)(__popc(loads) * rows * 128 * C::kColBoxes));
    }
    __syncwarp();
    const int y = whole ? (tile_first_pos<C>(p, T, c.j) & (ps - 1)) >> kPairShift : 0;
    if constexpr (C::kInter) {
        // one box per page: lane k copies page k, both column boxes, as whole 8-row groups
        if ((loads >> lane) & 1u)
            tma_load_5d(dst + C::row_off(lane * rows), tm, 0, 0, 0, y >> 3, checked_page(p, id) * p.G + c.g, bar, pol);
    } else {
        const int k = lane / C::kColBoxes, cb = lane % C::kColBoxes;
        const int my_id = __shfl_sync(0xffffffffu, id, k < C::kIdMax ? k : 0);
        if (k < nb && ((loads >> k) & 1u))
            tma_load_3d(dst + cb * kBoxBytes + k * rows * 128, tm, cb * kBoxCols, y,
                        checked_page(p, my_id) * p.G + c.g, bar, pol);
    }
}

// MMA issuer: writes a slot's staged row (the appended token) into its tile,
// row info.rel, in the 128-byte swizzled layout the TMA produced, and to the
// cache in global memory; then makes the tile visible to the tensor cores.
template <class C>
__device__ __noinline__ void patch_tile(uint8_t *tile, const uint8_t *stage_row, const PatchInfo info) {
    constexpr bool kPairL = C::kParts == 2;
    const int rel = info.rel;
    const int r = kPairL ? rel >> 1 : rel;   // tensor-map row of the position
#pragma unroll
    for (int q = 0; q < C::kRowBytes / 16; ++q) {
        const uint4 v = *reinterpret_cast<const uint4 *>(stage_row + q * 16);
        const int cb = kPairL ? (rel & 1) : (q >> 3);   // column box: the position's half, or dims 64q'..
        const int qq = q & 7;                           // 16-byte chunk inside the 128-byte row
        *reinterpret_cast<uint4 *>(tile + cb * C::kHalfStride + C::row_off(r) + ((qq ^ (r & 7)) << 4)) = v;
        if (info.dst) reinterpret_cast<uint4 *>(info.dst)[q] = v;
    }
    fence_proxy_async_smem();
}

template <int D, bool kPair, int N, int NH, int kVar>
__global__ void __launch_bounds__(kVar == 2 ? 256 : 224, 1)
    gqa_decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ TailMaps tails,
                         const DecodeParams p) {
    using C = TcCfg<D, kPair, N, NH, kVar>;
    constexpr bool kExt = C::kExt, kPaged = C::kPaged;
    constexpr int SK = C::kSK, SV = C::kSV, QB = C::kQBuf, NP = C::kParts, PB = C::kPBuf;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *red = reinterpret_cast<float *>(smem + C::kOffRed);
    float *lred = reinterpret_cast<float *>(smem + C::kOffLred);
    float *mrun_s = reinterpret_cast<float *>(smem + C::kOffM);
    float *alpha_s = reinterpret_cast<float *>(smem + C::kOffA);
    int *prefix = reinterpret_cast<int *>(smem + C::kOffPrefix);
    int *scratch = reinterpret_cast<int *>(smem + C::kOffScratch);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    uint64_t *kfull = bars, *kempty = kfull + SK, *vfull = kempty + SK, *vempty = vfull + SV;
    uint64_t *qfull = vempty + SV, *qempty = qfull + QB;
    uint64_t *sfull = qempty + QB, *sfree = sfull + 2, *pfull = sfree + 2, *ofull = pfull + PB, *ofree = ofull + 3;
    uint64_t *redbar = ofree + 3, *grp = redbar + 2, *done = grp + 1, *rfull = done + 1, *rempty = rfull + kRing;
    RangeEntry *ring = reinterpret_cast<RangeEntry *>(smem + C::kOffRing);
    int *ids_ring = reinterpret_cast<int *>(smem + C::kOffIds);
    uint64_t *idfull = rempty + kRing, *idempty = idfull + C::kIdRing;   // paged instances only
    uint64_t *prebar = rempty + kRing + C::kIdBars;
    uint8_t *kstage = smem + C::kOffStage, *vstage = kstage + SK * C::kRowBytes;
    PatchInfo *kinfo = reinterpret_cast<PatchInfo *>(smem + C::kOffPatch), *vinfo = kinfo + SK;
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + C::kOffFlags);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + C::kOffFlags + 8);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = gridDim.x;
    const AbortState ab{s_abort, p.flags};
    if (tid == 64) {
        GQA_TRACE_AT(kTrGlobalStart, globaltimer_ns());
        GQA_TRACE_AT(kTrStart, clock64());
    }

    if (tid == 0) {
        for (int s = 0; s < SK; ++s) {
            mbar_init(&kfull[s], 1);
            mbar_init(&kempty[s], 1);
        }
        for (int s = 0; s < SV; ++s) {
            mbar_init(&vfull[s], 1);
            mbar_init(&vempty[s], 1);
        }
        for (int s = 0; s < QB; ++s) {
            mbar_init(&qfull[s], 1);
            mbar_init(&qempty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sfull[s], 1);
            mbar_init(&sfree[s], 128);
            mbar_init(&redbar[s], 4);
        }
        for (int s = 0; s < PB; ++s) mbar_init(&pfull[s], 128);
        for (int s = 0; s < 3; ++s) {
            mbar_init(&ofull[s], 1);
            mbar_init(&ofree[s], 128);
        }
        mbar_init(grp, 128);
        for (int s = 0; s < kRing; ++s) {
            mbar_init(&rfull[s], 1);
            // both MMA issuers, the 128 softmax threads and (paged cache) the page-id warp
            mbar_init(&rempty[s], 2 + 128 + (kPaged ? 1 : 0));
        }
        mbar_init(done, 2);   // one commit from each MMA issuer
        mbar_init(prebar, 32);   // the producer warp, once the tile prefix is in shared memory
        if constexpr (kPaged) {
            for (int s = 0; s < C::kIdRing; ++s) {
                mbar_init(&idfull[s], 1);     // the page-id warp, once K of the tile is issued
                mbar_init(&idempty[s], 1);    // the producer thread, once it has taken the tile
            }
        }
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_q);
        if constexpr (kVar == 0) {
#pragma unroll
            for (int t = 0; t < 3; ++t) {
                tma_prefetch_desc(&tails.k[t]);
                tma_prefetch_desc(&tails.v[t]);
            }
        }
    }
    if (warp == 1) {
        tmem_alloc(s_tmem, C::kTmemCols);
        tmem_relinquish();
    }
    __syncthreads();   // barriers initialised, TMEM allocated
    tc_fence_after_sync();
    const uint32_t tmem = *s_tmem;
    // The next grid on the stream (the split-combine) may start as SMs have room.
    griddep_launch_dependents();
    // Everything above is on-chip; inputs and outputs are touched only once the
    // grids this one depends on have completed.
    griddep_wait();
    if (tid == 64) GQA_TRACE_AT(kTrDepDone, clock64());
    // The producer warp builds the tile prefix alone and goes straight on to its
    // first copies; the other roles wait for it on an mbarrier.
    bool pre_ok = true;
    if (warp == 0) {
        build_prefix_warp(p, C::kTileShift, prefix, scratch + 32, p.flags, seq_len_array(prefix, p.B));
        mbar_arrive(prebar);
    } else {
        pre_ok = mbar_wait(prebar, 0, ab);   // false only if the CTA aborts: its roles then do nothing
    }
    if (tid == 64) GQA_TRACE_AT(kTrSetup, clock64());

    const int G = p.G, n = p.n;
    const WorkSplit wsplit = make_split((long long)G * prefix[p.B], P, pool_tail_tiles(prefix, p.B, G, scratch[32]),
                                        p.dyn_cap);
    int kissued = 0, vissued = 0, qissued = 0;

    if (!pre_ok) {
        // the producer warp never published the tile prefix: nothing to do
    } else if (warp == 0) {
        // ================================================================ producer
        // Hands every work range to the other roles through the ring: the static
        // range first, then one claimed chunk at a time, then an end marker.
        if (lane == 0) {
            GQA_TRACE_AT(kTrProdIn, clock64());
            const int *tlen = seq_len_array(prefix, p.B);   // plain instances: the last tiles' lengths
            const uint64_t pol_kv = l2_policy_evict_first();
            const uint64_t pol_q = l2_policy_evict_last();
            RangeEntry next{0, 0, -1};
            bool have_next = false;
            if ((int)blockIdx.x < wsplit.Pw) {
                next.ub = range_start(blockIdx.x, wsplit.Ws, wsplit.Pw);
                next.len = (int)(range_start(blockIdx.x + 1, wsplit.Ws, wsplit.Pw) - next.ub);
                have_next = next.len > 0;
            }
            int pushed = 0, piece = 0, v_r = 0;
            bool k_done = false, v_done = false;
            long long k_u = 0, k_end = 0, k_ub = 0, v_u = 0, v_end = 0;
            Cursor kc{0, 0, 0, 1}, vc{0, 0, 0, 1};
            SeqLenCache k_lens, v_lens;
            IdlePoll poll;
            // paged instances: the page-id warp copies the V tiles, so this thread stops
            // once the K side has issued everything
            while (kPaged ? !k_done : !v_done) {
                bool progress = false;
                // ---- the next range, once the K side has issued the current one
                if (!k_done && k_u == k_end) {
                    if (!have_next) {
                        next.chunk = -2;
                        next.len = 0;
                        if (wsplit.nchunks > 0) {
                            const unsigned j = atomicAdd(p.ticket, 1u);
                            if (j < (unsigned)wsplit.nchunks) {
                                next.ub = wsplit.Ws + (long long)j * kChunk;
                                next.len = kChunk;
                                next.chunk = (int)j;
                            } else if (atomicAdd(p.fails, 1u) == (unsigned)P - 1) {
                                // every CTA has failed once: nobody claims again in this launch
                                atomicExch(p.ticket, 0u);
                                atomicExch(p.fails, 0u);
                            }
                        }
                        have_next = true;
                    }
                    const int slot = pushed % kRing;
                    if (pushed < kRing ||
                        ((kPaged || v_r > pushed - kRing) && mbar_test_wait(&rempty[slot], ((pushed / kRing) - 1) & 1))) {
                        ring[slot] = next;
                        mbar_arrive(&rfull[slot]);   // release: the entry is visible to the waiters
                        if (pushed == 0) GQA_TRACE_AT(kTrRing0, clock64());
                        ++pushed;
                        have_next = false;
                        if (next.chunk == -2) {
                            k_done = true;
                        } else {
                            k_ub = k_u = next.ub;
                            k_end = next.ub + next.len;
                            kc = cursor_at(k_u, prefix, p.B, G);
                        }
                        progress = true;
                    }
                }
                // ---- K of the next tile (and Q when it starts a piece)
                if (k_u < k_end) {
                    const int i = kissued;
                    const bool first = (k_u == k_ub) || (kc.j == 0);
                    const bool last = (k_u + 1 == k_end) || (kc.j + 1 == kc.tiles);
                    const int st = i % SK, qb = piece % QB;
                    // K runs at most one tile ahead of V: a tile's V then lands about when its
                    // probabilities are ready, and a piece's last value GEMM does not wait long
                    // (paged instances: the page-id warp has copied K of the tile once idfull
                    // completes; this thread then only issues Q and paces the range claims)
                    if ((kPaged || vissued >= i) &&
                        (!first || piece < QB || mbar_test_wait(&qempty[qb], ((piece / QB) - 1) & 1)) &&
                        (kPaged || i < SK || mbar_test_wait(&kempty[st], ((i / SK) - 1) & 1)) &&
                        (!kPaged || mbar_test_wait(&idfull[i % C::kIdRing], (i / C::kIdRing) & 1))) {
                        if (first) {
                            if (i == 0) GQA_TRACE_AT(kTrPreQ, clock64());
                            mbar_arrive_expect_tx(&qfull[qb], C::kQBytes);
                            uint8_t *qdst = smem + C::kOffQ + qb * C::kQBytes;
                            const int y = kc.b * p.H + kc.g * n;
#pragma unroll
                            for (int c = 0; c < C::kQBoxes; ++c)
                                tma_load_2d(qdst + c * N * 128, &tm_q, c * kBoxCols, y, &qfull[qb], pol_q);
                            if constexpr (C::kHM)   // the second copy: rows 64..127 of the A operand
                                tma_load_2d(qdst + N * 128, &tm_q, 0, y, &qfull[qb], pol_q);
                            ++qissued;
                            if (i == 0) GQA_TRACE_AT(kTrFirstQ, clock64());
                        }
                        uint8_t *kdst = smem + C::kOffK + st * C::kTileBytes;
                        if (!kPaged && i < 20) GQA_TRACE_AT(kTrProbe + 4 * i, clock64());
                        if constexpr (kPaged) {
                            mbar_arrive(&idempty[i % C::kIdRing]);   // the ring entry may be reused
                        } else
#ifdef GQA_TEST_HOOKS
                        if (i == p.withhold_k && blockIdx.x == 0) {
                            // test hook: this copy is never made, so the score GEMM's bounded
                            // wait for it runs out and the CTA takes its abort path
                        } else
#endif
                        if constexpr (kExt) {
                            produce_variant_tile<C>(p, &tm_k, kdst, &kfull[st], kc, k_lens.get(p, kc.b), pol_kv,
                                                    p.k_new, kstage + st * C::kRowBytes, &kinfo[st], p.k_dst);
                        } else {
                            const int rows = plain_tile_rows<C>(kc, tlen);
                            if (rows == kTile)
                                produce_plain_tile<C>(p, &tm_k, kdst, &kfull[st], kc, pol_kv);
                            else
                                produce_tail_tile<C>(p, tails.k, kdst, &kfull[st], kc, pol_kv, rows);
                        }
                        if (!kPaged && i < 20) GQA_TRACE_AT(kTrProbe + 4 * i + 1, clock64());
                        if (i == 0) GQA_TRACE_AT(kTrFirstK, clock64());
                        if (!kPaged && i < 128) GQA_TRACE_AT(kTrKIssue + i, clock64());
                        ++kissued;
                        ++k_u;
                        if (last) ++piece;
                        cursor_next(kc, prefix, p.B, G);
                        progress = true;
                    }
                }
                // ---- V of the next tile (walks the same ranges, never ahead of K)
                if (!kPaged && v_u == v_end && v_r < pushed) {
                    const RangeEntry e = ring[v_r % kRing];   // written by this thread
                    ++v_r;
                    if (e.chunk == -2) {
                        v_done = true;
                    } else {
                        v_u = e.ub;
                        v_end = e.ub + e.len;
                        vc = cursor_at(v_u, prefix, p.B, G);
                    }
                    progress = true;
                }
                if (!kPaged && v_u < v_end && vissued < kissued) {
                    const int i = vissued, st = i % SV;
                    if (i < SV || mbar_test_wait(&vempty[st], ((i / SV) - 1) & 1)) {
                        uint8_t *vdst = smem + C::kOffV + st * C::kTileBytes;
                        if (i < 20) GQA_TRACE_AT(kTrProbe + 4 * i + 2, clock64());
                        if constexpr (kPaged) {
                            // never reached: the page-id warp copies V
                        } else if constexpr (kExt) {
                            produce_variant_tile<C>(p, &tm_v, vdst, &vfull[st], vc, v_lens.get(p, vc.b), pol_kv,
                                                    p.v_new, vstage + st * C::kRowBytes, &vinfo[st], p.v_dst);
                        } else {
                            const int rows = plain_tile_rows<C>(vc, tlen);
                            if (rows == kTile)
                                produce_plain_tile<C>(p, &tm_v, vdst, &vfull[st], vc, pol_kv);
                            else
                                produce_tail_tile<C>(p, tails.v, vdst, &vfull[st], vc, pol_kv, rows);
                        }
                        if (i < 20) GQA_TRACE_AT(kTrProbe + 4 * i + 3, clock64());
                        if (i < 128) GQA_TRACE_AT(kTrVIssue + i, clock64());
                        ++vissued;
                        ++v_u;
                        cursor_next(vc, prefix, p.B, G);
                        progress = true;
                    }
                }
                if (progress) {
                    poll.progressed();
                } else if (!poll.step(ab)) {
                    break;
                }
            }
        }
    } else if (warp == 1 || warp == 6) {
        // ================================================================ MMA issuers
        // Warp 1 issues the score GEMMs, warp 6 the value GEMMs: a tcgen05.mma takes
        // tens of nanoseconds to issue, and two issuing threads halve the serial time
        // per tile.  Each writes its own accumulators and commits its own barriers.
        const bool do_s = warp == 1, do_pv = warp == 6;
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(128, N, false, false);
            constexpr uint32_t idPV = idesc_bf16_f32(C::kPvM, C::kOW, true, false);
            const uint32_t sbase = smem_addr(smem);
            Cursor cur{0, 0, 0, 1};
            long long s_u = 0, s_end = 0, s_ub = 0;
            int s_i = 0, pv_i = 0, piece = 0, r_read = 0, pv_avail = 0;
            bool ranges_done = false;   // the end marker has been read
#ifdef GQA_TRACE
            int k_seen = -1, v_seen = -1;
#endif
            IdlePoll poll;
            while (!(ranges_done && (do_s ? s_u == s_end : pv_i == pv_avail))) {
                bool progress = false;
                // ---- the next range, once this role has used up the current one
                if (!ranges_done && (do_s ? s_u == s_end : pv_i == pv_avail)) {
                    const int slot = r_read % kRing;
                    if (mbar_test_wait(&rfull[slot], (r_read / kRing) & 1)) {
                        const RangeEntry e = ring[slot];
                        mbar_arrive(&rempty[slot]);
                        ++r_read;
                        if (e.chunk == -2) {
                            ranges_done = true;
                        } else if (do_s) {
                            s_ub = s_u = e.ub;
                            s_end = e.ub + e.len;
                            cur = cursor_at(s_u, prefix, p.B, G);
                        } else {
                            pv_avail += e.len;
                        }
                        progress = true;
                    }
                }
                // ---- scores of tile s_i: needs its K, its piece's Q and a free S buffer
                if (do_s && s_u < s_end) {
                    const bool first = (s_u == s_ub) || (cur.j == 0);
                    const bool last = (s_u + 1 == s_end) || (cur.j + 1 == cur.tiles);
                    const int st = s_i % SK, bi = s_i & 1, qb = piece % QB;
                    const bool kready = mbar_test_wait(&kfull[st], (s_i / SK) & 1);
#ifdef GQA_TRACE
                    if (kready && s_i > k_seen) {
                        if (s_i < 128) GQA_TRACE_AT(kTrKReady + s_i, clock64());
                        k_seen = s_i;
                    }
#endif
                    if ((!first || mbar_test_wait(&qfull[qb], (piece / QB) & 1)) && kready &&
                        (s_i < 2 || mbar_test_wait(&sfree[bi], ((s_i >> 1) - 1) & 1))) {
                        tc_fence_after_sync();
                        if (kExt && p.k_new && kinfo[st].on)   // the appended key replaces its row first
                            patch_tile<C>(smem + C::kOffK + st * C::kTileBytes, kstage + st * C::kRowBytes, kinfo[st]);
                        const uint32_t kb = sbase + C::kOffK + st * C::kTileBytes;
                        const uint32_t qbase = sbase + C::kOffQ + qb * C::kQBytes;
                        // part c (paired layout: the box of even / odd positions) -> S columns [bi][c];
                        // base descriptors once, then constant offsets (K step = 32 bytes in a box)
                        const uint64_t kd0 = sdesc_sw128(kb, 16, C::kGroupStride), qd0 = sdesc_sw128(qbase, 16, 1024);
                        if constexpr (C::kHM) {
                            // S [2 x 64 heads x 128 positions] = [Q; Q]·K^T: Q is the A operand (d = 64: one K atom)
                            constexpr uint32_t idS_hm = idesc_bf16_f32(128, kTile, false, false);
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk)
                                umma_bf16(tmem + bi * kTile, sdesc_add(qd0, kk * 32), sdesc_add(kd0, kk * 32), idS_hm,
                                          kk != 0);
                        } else {
#pragma unroll
                            for (int c = 0; c < NP; ++c)
#pragma unroll
                                for (int kk = 0; kk < D / 16; ++kk)
                                    umma_bf16(tmem + (bi * NP + c) * N,
                                              sdesc_add(kd0, (kPair ? c : (kk >> 2)) * C::kHalfStride + (kk & 3) * 32),
                                              sdesc_add(qd0, (kk >> 2) * (N * 128) + (kk & 3) * 32), idS, kk != 0);
                        }
                        umma_commit(&sfull[bi]);
                        umma_commit(&kempty[st]);
                        if (last) {
                            umma_commit(&qempty[qb]);
                            ++piece;
                        }
                        if (s_i < 128) GQA_TRACE_AT(kTrSIssue + s_i, clock64());
                        cursor_next(cur, prefix, p.B, G);
                        ++s_u;
                        ++s_i;
                        progress = true;
                    }
                }
                // ---- values of tile pv_i: needs its V, its P (so its scores are done) and a free O buffer
                if (do_pv && pv_i < pv_avail) {
                    const int st = pv_i % SV, pbi = pv_i % PB, ob = pv_i % 3;
                    const bool vready = mbar_test_wait(&vfull[st], (pv_i / SV) & 1);
#ifdef GQA_TRACE
                    if (vready && pv_i > v_seen) {
                        if (pv_i < 128) GQA_TRACE_AT(kTrVReady + pv_i, clock64());
                        v_seen = pv_i;
                    }
#endif
                    if (vready && mbar_test_wait(&pfull[pbi], (pv_i / PB) & 1) &&
                        (pv_i < 3 || mbar_test_wait(&ofree[ob], ((pv_i / 3) - 1) & 1))) {
                        tc_fence_after_sync();
                        if (kExt && p.v_new && vinfo[st].on)   // the appended value replaces its row first
                            patch_tile<C>(smem + C::kOffV + st * C::kTileBytes, vstage + st * C::kRowBytes, vinfo[st]);
                        const uint32_t vb = sbase + C::kOffV + st * C::kTileBytes;
                        const uint32_t d_o = tmem + C::kOCol + ob * C::kOBuf;
                        // A = V^T, MN-major: the column boxes are the M atoms (LBO), the 8-row groups
                        // the K steps (SBO); 16 positions = two groups
                        const uint64_t vd0 = sdesc_sw128(vb, C::kHalfStride, C::kGroupStride);
                        const uint64_t pd0 = sdesc_sw128(sbase + C::kOffP + pbi * C::kPBufBytes, 16, 1024);
                        if constexpr (C::kHM) {
                            // O [64 heads x d] = P_hi·V + P_lo·V: P is the A operand (K-major, two
                            // 64-position halves of 8 KB), V the B operand (MN-major, 16 positions = 2 KB)
                            constexpr uint32_t idPV_hm = idesc_bf16_f32(64, D, false, true);
#pragma unroll
                            for (int half = 0; half < 2; ++half)
#pragma unroll
                                for (int kk = 0; kk < kTile / 16; ++kk)
                                    umma_bf16(d_o, sdesc_add(pd0, half * 16384 + (kk >> 2) * 8192 + (kk & 3) * 32),
                                              sdesc_add(vd0, kk * 2048), idPV_hm, (half | kk) != 0);
                        } else {
#pragma unroll
                            for (int kk = 0; kk < kTile / 16; ++kk)
                                umma_bf16(d_o, sdesc_add(vd0, kk * 2 * C::kGroupStride),
                                          sdesc_add(pd0, (kk >> 2) * (C::kOW * 128) + (kk & 3) * 32), idPV, kk != 0);
                        }
                        umma_commit(&ofull[ob]);
                        umma_commit(&vempty[st]);
                        if (pv_i < 128) GQA_TRACE_AT(kTrPvIssue + pv_i, clock64());
                        ++pv_i;
                        progress = true;
                    }
                }
                if (progress) {
                    poll.progressed();
                } else if (!poll.step(ab)) {
                    break;
                }
            }
            umma_commit(done);
            mbar_wait_teardown(done, 0);
        }
    } else if (warp < 6) {
        if constexpr (C::kHM) {
        // ================================================================ softmax, heads on M
        // S side: TMEM lane r = q4*32 + lane holds head hs = r % 64; its thread takes the
        // positions of half hf = r / 64 of the tile.  The two threads of a head agree on the
        // tile maximum through shared memory (one barrier per tile).  O side: the O
        // accumulator of head ho = q4*16 + lane lives in TMEM lane q4*32 + lane (lanes < 16),
        // folded by that thread with the rescale factors the S side publishes.
        const int q4 = warp & 3;
        const int tg = tid - 64;                 // 0..127 within the group (V row cleared by this thread)
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const int r = q4 * 32 + lane;
        const int hs = r & 63, hf = r >> 6;      // S side: head and position half
        const int ho = q4 * 16 + lane;           // O side: head (lanes < 16)
        const bool has_out = lane < 16 && ho < n;
        zero_empty_sequences<D>(p, prefix, P, tg, 128);
        GroupSync gsync{grp, 0};
        float accv[D];
        float l_half = 0.f, m_run = 0.f;
        int seq_b = 0, win_b = 0, piece_i0 = 0, npe = 0, i = 0, rr = 0;
        long long piece_u0 = 0;
        bool ok = true;
#pragma unroll
        for (int j = 0; j < D; ++j) accv[j] = 0.f;

        // fold O of tile t into accv with that tile's rescale factor (published by the S side)
        auto fold_hm = [&](int t) -> bool {
            const int ob = t % 3;
            if (!mbar_wait(&ofull[ob], (t / 3) & 1, ab)) return false;
            tc_fence_after_sync();
            const float al = alpha_s[(t % 4) * NH + (ho & 63)];
            const uint32_t oc = tmem + lane_off + C::kOCol + ob * C::kOBuf;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                tmem_ld_32x32b<32>(oc + c0, o);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) accv[c0 + j] = fmaf(accv[c0 + j], al, __uint_as_float(o[j]));
            }
            tc_fence_before_sync();
            mbar_arrive(&ofree[ob]);
            return true;
        };

        while (ok) {
          const int rslot = rr % kRing;
          if (!mbar_wait(&rfull[rslot], (rr / kRing) & 1, ab)) { ok = false; break; }
          const RangeEntry range = ring[rslot];
          mbar_arrive(&rempty[rslot]);
          ++rr;
          if (range.chunk == -2) break;
          Cursor cur = cursor_at(range.ub, prefix, p.B, G);
          int range_piece = 0;
          for (int k = 0; k < range.len && ok; ++k, ++i) {
            const long long u = range.ub + k;
            const bool first = (k == 0) || (cur.j == 0);
            const bool last = (k + 1 == range.len) || (cur.j + 1 == cur.tiles);
            const int bi = i & 1;
            if (first) {
                piece_u0 = u;
                piece_i0 = i;
                seq_b = seq_len_of(p, cur.b);
                win_b = kExt ? window_start(p, seq_b) : 0;
                l_half = 0.f;
#pragma unroll
                for (int j = 0; j < D; ++j) accv[j] = 0.f;
            }
            if (!mbar_wait(&sfull[bi], (i >> 1) & 1, ab)) { ok = false; break; }
            if (tg == 0 && i < 128) GQA_TRACE_AT(kTrPFull + i, clock64());
            tc_fence_after_sync();
            const int tile_pos0 = ((win_b >> C::kTileShift) + cur.j) << C::kTileShift;
            const int hi_pos = seq_b - tile_pos0;              // >= 1
            const int lo_pos = kExt ? win_b - tile_pos0 : 0;   // > 0 only in a window's first tile
            const uint32_t sc = tmem + lane_off + bi * kTile + hf * 64;
            // pass 1: this half's maximum, then the head's from both halves
            float mt = -INFINITY;
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 32) {
                uint32_t sv[32];
                tmem_ld_32x32b<32>(sc + c0, sv);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int pos = hf * 64 + c0 + j;
                    if (pos < hi_pos && pos >= lo_pos) mt = fmaxf(mt, __uint_as_float(sv[j]) * p.scale_log2);
                }
            }
            red[bi * 128 + r] = mt;
            __syncwarp();
            if (lane == 0) mbar_arrive(&redbar[bi]);
            if (!mbar_wait(&redbar[bi], (i >> 1) & 1, ab)) { ok = false; break; }
            const float mh = fmaxf(red[bi * 128 + hs], red[bi * 128 + hs + 64]);   // finite: a tile has a position
            const float m_new = (i == piece_i0) ? mh : fmaxf(m_run, mh);
            const float alpha = (i == piece_i0) ? 0.f : ex2(m_run - m_new);
            m_run = m_new;
            if (hf == 0) {
                alpha_s[(i % 4) * NH + hs] = alpha;
                mrun_s[(i % 3) * NH + hs] = m_new;
            }
            // P buffer i % PB last held P(i - PB): its value GEMM must be done with it
            const int pbi = i % PB;
            if (i >= PB && !mbar_wait(&ofull[(i - PB) % 3], ((i - PB) / 3) & 1, ab)) { ok = false; break; }
            // pass 2: probabilities of this half, the half's sum, and P row hs, half hf, as bf16
            // hi (first 16 KB) + lo (next 16 KB), K-major, 128-byte swizzle: 16-byte chunk
            // (pos % 64) / 8 stored at chunk ((pos % 64) / 8) ^ (hs % 8)
            uint8_t *prow = smem + C::kOffP + pbi * C::kPBufBytes + hf * 8192 + hs * 128;
            float sum = 0.f;
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 32) {
                uint32_t sv[32];
                tmem_ld_32x32b<32>(sc + c0, sv);
                tmem_wait_ld();
#pragma unroll
                for (int g8 = 0; g8 < 4; ++g8) {
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int j2 = 0; j2 < 4; ++j2) {
                        float pv[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int j = g8 * 8 + j2 * 2 + e, pos = hf * 64 + c0 + j;
                            pv[e] = (pos < hi_pos && pos >= lo_pos)
                                        ? ex2(__uint_as_float(sv[j]) * p.scale_log2 - m_new) : 0.f;
                            sum += pv[e];
                        }
                        const __nv_bfloat162 h2 = __floats2bfloat162_rn(pv[0], pv[1]);
                        const float2 hf2 = __bfloat1622float2(h2);
                        const __nv_bfloat162 l2 = __floats2bfloat162_rn(pv[0] - hf2.x, pv[1] - hf2.y);
                        hw[j2] = *reinterpret_cast<const uint32_t *>(&h2);
                        lw[j2] = *reinterpret_cast<const uint32_t *>(&l2);
                    }
                    const int ch = (c0 + g8 * 8) >> 3;   // 16-byte chunk of the half row
                    uint8_t *dst = prow + ((ch ^ (hs & 7)) << 4);
                    *reinterpret_cast<uint4 *>(dst) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *reinterpret_cast<uint4 *>(dst + 16384) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                }
            }
            l_half = fmaf(l_half, alpha, sum);
            tc_fence_before_sync();
            mbar_arrive(&sfree[bi]);
            // ---- clear V rows outside [lo, hi) (they may hold anything, NaN included): row tg
            if (hi_pos < C::kTilePos || lo_pos > 0) {
                const int sv = i % SV;
                if (!mbar_wait(&vfull[sv], (i / SV) & 1, ab)) { ok = false; break; }
                if (!(tg < hi_pos && tg >= lo_pos)) {
                    uint4 *w = reinterpret_cast<uint4 *>(smem + C::kOffV + sv * C::kTileBytes + C::row_off(tg));
#pragma unroll
                    for (int q = 0; q < 8; ++q) w[q] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(&pfull[pbi]);
            // ---- fold O of the tile before the previous one (its alpha was published two
            // barriers ago)
            if (i - 2 >= piece_i0 && !fold_hm(i - 2)) { ok = false; break; }

            if (last) {
                if (tg == 0) GQA_TRACE_AT(kTrPieceEnd + 2 * npe, clock64());
                lred[r] = l_half;
                if (!gsync(ab)) { ok = false; break; }        // also publishes tile i's alpha and m
                if (i - 1 >= piece_i0 && !fold_hm(i - 1)) { ok = false; break; }
                if (!fold_hm(i)) { ok = false; break; }
                const int seg = cur.b * G + cur.g;
                const long long seg_a = (long long)G * prefix[cur.b] + (long long)cur.g * cur.tiles;
                const bool owned = (piece_u0 == seg_a) && (cur.j + 1 == cur.tiles);
                if (has_out) {
                    const float L = lred[ho] + lred[ho + 64];
                    if (owned) {
                        float4 *o4 = reinterpret_cast<float4 *>(p.out + ((size_t)cur.b * p.H + (size_t)cur.g * n + ho) * D);
#pragma unroll
                        for (int c = 0; c < D / 4; ++c)
                            o4[c] = make_float4(accv[4 * c] / L, accv[4 * c + 1] / L, accv[4 * c + 2] / L,
                                                accv[4 * c + 3] / L);
                    } else {
                        const int slot = range.chunk < 0 ? (int)blockIdx.x + seg : chunk_slot(p, range.chunk, range_piece);
                        float *sp = slot_ptr(p, slot, D);
                        sp[ho] = mrun_s[(i % 3) * NH + ho];
                        sp[n + ho] = L;
                        float4 *a4 = reinterpret_cast<float4 *>(sp + slot_acc_offset(n) + ho * D);
#pragma unroll
                        for (int c = 0; c < D / 4; ++c)
                            a4[c] = make_float4(accv[4 * c], accv[4 * c + 1], accv[4 * c + 2], accv[4 * c + 3]);
                    }
                }
                // lred is next written at the next piece's end, after that piece's barriers
                if (tg == 0) GQA_TRACE_AT(kTrPieceEnd + 2 * npe + 1, clock64());
                ++npe;
                ++range_piece;
            }
            cursor_next(cur, prefix, p.B, G);
          }
        }
        if (tg == 0) GQA_TRACE_AT(kTrTiles, i);
        } else {
        // ================================================================ softmax + epilogue
        const int q4 = warp & 3;                 // TMEM lane quadrant of this warp
        const int r = q4 * 32 + lane;            // tile position (S) / head dim (O, d = 128)
        const int tg = tid - 64;                 // 0..127 within the group
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        // dim held in the O accumulator by this thread (M = 64 puts 16 rows in each
        // quadrant; at kPair rows r and r + 64 hold the even and odd positions' share
        // of dim r, and the threads r < 64 hold the sum after a piece ends)
        const int odim = kPair ? (r & 63) : (D == 128) ? r : q4 * 16 + lane;
        const bool has_dim = kPair ? (r < 64) : (D == 128) || lane < 16;
        const uint32_t o_part = (kPair && r >= 64) ? 2 * C::kNPV : 0;   // this row's (part) column block
        // heads are handled in chunks of CH: at 64 heads per group the per-head
        // arrays of a whole tile would not fit in registers (up to 32 they do, and a
        // single pass over the scores is cheaper)
        constexpr int CH = NH <= 32 ? NH : 16;
        constexpr int NCH = NH / CH;
        constexpr int kHalveCH = ilog2(CH) < 5 ? ilog2(CH) : 5;
        zero_empty_sequences<D>(p, prefix, P, tg, 128);
        GroupSync gsync{grp, 0};
        float l_part[NH], acc[NH];
        int seq_b = 0, win_b = 0, piece_i0 = 0, npe = 0, i = 0, rr = 0;
        long long piece_u0 = 0;
        bool ok = true;

        // fold O of tile t into acc with that tile's rescale factor
        auto fold_o = [&](int t) -> bool {
            const int ob = t % 3;
            if (!mbar_wait(&ofull[ob], (t / 3) & 1, ab)) return false;
            tc_fence_after_sync();
            // hi and lo columns and the rescale factors, at most 16 heads at a time
            // (bounds the registers at NH = 64)
            const uint32_t oc = tmem + lane_off + C::kOCol + ob * C::kOBuf + o_part;
#pragma unroll
            for (int h0 = 0; h0 < NH; h0 += CH) {
                uint32_t ohi[CH], olo[CH];
                float al[CH];
                load_vec<CH>(alpha_s + (t % 4) * NH + h0, al);
                tmem_ld_32x32b<CH>(oc + h0, ohi);
                tmem_ld_32x32b<CH>(oc + C::kNPV + h0, olo);
                tmem_wait_ld();
#pragma unroll
                for (int h = 0; h < CH; ++h)
                    acc[h0 + h] = fmaf(acc[h0 + h], al[h], __uint_as_float(ohi[h]) + __uint_as_float(olo[h]));
            }
            tc_fence_before_sync();
            mbar_arrive(&ofree[ob]);
            return true;
        };

        while (ok) {
          // ---- the next work range from the producer
          const int rslot = rr % kRing;
          if (!mbar_wait(&rfull[rslot], (rr / kRing) & 1, ab)) { ok = false; break; }
          const RangeEntry range = ring[rslot];
          mbar_arrive(&rempty[rslot]);
          ++rr;
          if (range.chunk == -2) break;
          Cursor cur = cursor_at(range.ub, prefix, p.B, G);
          int range_piece = 0;   // pieces of this range finished so far (a chunk's slot index)
          for (int k = 0; k < range.len && ok; ++k, ++i) {
            const long long u = range.ub + k;
            const bool first = (k == 0) || (cur.j == 0);
            const bool last = (k + 1 == range.len) || (cur.j + 1 == cur.tiles);
            const int bi = i & 1;
            if (first) {
                piece_u0 = u;
                piece_i0 = i;
                seq_b = seq_len_of(p, cur.b);
                win_b = kExt ? window_start(p, seq_b) : 0;
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                    l_part[h] = 0.f;
                    acc[h] = 0.f;
                }
            }
            const int pbi = i % PB;   // this tile's P buffer
            if constexpr (NCH == 1) {
            // ---- scores of this tile: S^T row r of every part (heads 0..NH-1); part c of row r
            // is position r, or 2r + c in the paired layout
            if (!mbar_wait(&sfull[bi], (i >> 1) & 1, ab)) { ok = false; break; }
            tc_fence_after_sync();
            uint32_t sraw[NP][NH];
#pragma unroll
            for (int c = 0; c < NP; ++c) tmem_ld_32x32b<NH>(tmem + lane_off + (bi * NP + c) * N, sraw[c]);
            tmem_wait_ld();
            tc_fence_before_sync();
            mbar_arrive(&sfree[bi]);
            // attended positions of this tile: [lo, hi) relative to its first position
            const int tile_pos0 = ((win_b >> C::kTileShift) + cur.j) << C::kTileShift;
            const int valid_cnt = seq_b - tile_pos0;   // hi, >= 1
            const int lo = kExt ? win_b - tile_pos0 : 0;   // > 0 only in a window's first tile
            bool valid[NP];
            float x[NP][NH], red_v[NH];
#pragma unroll
            for (int h = 0; h < NH; ++h) red_v[h] = -INFINITY;
#pragma unroll
            for (int c = 0; c < NP; ++c) {
                const int pos = kPair ? 2 * r + c : r;
                valid[c] = pos < valid_cnt && pos >= lo;
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                    x[c][h] = valid[c] ? __uint_as_float(sraw[c][h]) * p.scale_log2 : -INFINITY;
                    red_v[h] = fmaxf(red_v[h], x[c][h]);
                }
            }
            butterfly_reduce<NH, true>(red_v, lane);
            butterfly_store<NH, C::kHalve>(red_v, lane, red + (bi * 4 + q4) * NH);
            __syncwarp();
            if (lane == 0) mbar_arrive(&redbar[bi]);
            if (!mbar_wait(&redbar[bi], (i >> 1) & 1, ab)) { ok = false; break; }
            float m_new[NH], alpha[NH];
            reduce4<NH, true>(red + bi * 4 * NH, m_new);        // tile maximum per head
            if (i == piece_i0) {
#pragma unroll
                for (int h = 0; h < NH; ++h) alpha[h] = 0.f;      // nothing to rescale yet
            } else {
                float m_old[NH];
                load_vec<NH>(mrun_s + ((i + 2) % 3) * NH, m_old);   // state after tile i-1
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                    m_new[h] = fmaxf(m_old[h], m_new[h]);        // finite: every tile has a valid position
                    alpha[h] = ex2(m_old[h] - m_new[h]);
                }
            }
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                float sx = 0.f;
#pragma unroll
                for (int c = 0; c < NP; ++c) {
                    x[c][h] = ex2(x[c][h] - m_new[h]);           // 0 at invalid positions
                    sx += x[c][h];
                }
                l_part[h] = fmaf(l_part[h], alpha[h], sx);
            }
            if (tg == 0) {
                store_vec<NH>(mrun_s + (i % 3) * NH, m_new);
                store_vec<NH>(alpha_s + (i % 4) * NH, alpha);
            }
            // ---- clear V rows outside [lo, hi): past the end of a sequence, before a window's
            // start, or in pages not copied; they may hold anything, NaN included
            if (valid_cnt < C::kTilePos || lo > 0) {
                const int sv = i % SV;
                if (!mbar_wait(&vfull[sv], (i / SV) & 1, ab)) { ok = false; break; }
                uint8_t *vrow = smem + C::kOffV + sv * C::kTileBytes + C::row_off(r);
#pragma unroll
                for (int c = 0; c < C::kColBoxes; ++c) {
                    // paired layout: box c holds the positions of part c; otherwise a row's
                    // boxes hold the dims of one position (part 0)
                    if (!valid[kPair ? c : 0]) {
                        uint4 *w = reinterpret_cast<uint4 *>(vrow + c * C::kHalfStride);
#pragma unroll
                        for (int k = 0; k < 8; ++k) w[k] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
            // ---- probabilities to shared memory as bf16 hi + lo (K-major, 128-byte swizzle):
            // row (c * 2 + hi/lo) * kNPV + h of the value GEMM's B operand, position r;
            // P buffer i % PB last held P(i - PB): its value GEMM must be done with it
            if (i >= PB && !mbar_wait(&ofull[(i - PB) % 3], ((i - PB) / 3) & 1, ab)) { ok = false; break; }
#pragma unroll
            for (int c = 0; c < NP; ++c) {
                uint8_t *phi = smem + C::kOffP + pbi * C::kPBufBytes + (r >> 6) * (C::kOW * 128) +
                               (c * 2) * (C::kNPV * 128);
                uint8_t *plo = phi + C::kNPV * 128;
                const int col = r & 63;
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                    if (h < n) {
                        const int off = h * 128 + ((((col >> 3) ^ (h & 7))) << 4) + (col & 7) * 2;
                        const __nv_bfloat16 hi = __float2bfloat16_rn(x[c][h]);
                        const __nv_bfloat16 lo = __float2bfloat16_rn(x[c][h] - __bfloat162float(hi));
                        *reinterpret_cast<__nv_bfloat16 *>(phi + off) = hi;
                        *reinterpret_cast<__nv_bfloat16 *>(plo + off) = lo;
                    }
                }
            }
            } else {
            // ---- scores of this tile, CH heads at a time: pass 1 takes the tile maxima
            // (one barrier for all heads), pass 2 reloads the scores from TMEM and turns
            // them into probabilities; the S buffer is released after pass 2
            if (!mbar_wait(&sfull[bi], (i >> 1) & 1, ab)) { ok = false; break; }
            tc_fence_after_sync();
            const int tile_pos0 = ((win_b >> C::kTileShift) + cur.j) << C::kTileShift;
            const int valid_cnt = seq_b - tile_pos0;   // hi, >= 1
            const int lo = kExt ? win_b - tile_pos0 : 0;   // > 0 only in a window's first tile
            bool valid[NP];
#pragma unroll
            for (int c = 0; c < NP; ++c) {
                const int pos = kPair ? 2 * r + c : r;
                valid[c] = pos < valid_cnt && pos >= lo;
            }
#pragma unroll
            for (int h0 = 0; h0 < NH; h0 += CH) {
                uint32_t sr[NP][CH];
#pragma unroll
                for (int c = 0; c < NP; ++c) tmem_ld_32x32b<CH>(tmem + lane_off + (bi * NP + c) * N + h0, sr[c]);
                tmem_wait_ld();
                float rv[CH];
#pragma unroll
                for (int h = 0; h < CH; ++h) {
                    rv[h] = -INFINITY;
#pragma unroll
                    for (int c = 0; c < NP; ++c)
                        rv[h] = fmaxf(rv[h], valid[c] ? __uint_as_float(sr[c][h]) * p.scale_log2 : -INFINITY);
                }
                butterfly_reduce<CH, true>(rv, lane);
                butterfly_store<CH, kHalveCH>(rv, lane, red + (bi * 4 + q4) * NH + h0);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&redbar[bi]);
            if (!mbar_wait(&redbar[bi], (i >> 1) & 1, ab)) { ok = false; break; }
            // P buffer i % PB last held P(i - PB): its value GEMM must be done with it
            if (i >= PB && !mbar_wait(&ofull[(i - PB) % 3], ((i - PB) / 3) & 1, ab)) { ok = false; break; }
#pragma unroll
            for (int h0 = 0; h0 < NH; h0 += CH) {
                float m_new[CH], alpha[CH];
                reduce4<CH, true, NH>(red + bi * 4 * NH + h0, m_new);   // tile maximum per head
                if (i == piece_i0) {
#pragma unroll
                    for (int h = 0; h < CH; ++h) alpha[h] = 0.f;      // nothing to rescale yet
                } else {
                    float m_old[CH];
                    load_vec<CH>(mrun_s + ((i + 2) % 3) * NH + h0, m_old);   // state after tile i-1
#pragma unroll
                    for (int h = 0; h < CH; ++h) {
                        m_new[h] = fmaxf(m_old[h], m_new[h]);
                        alpha[h] = ex2(m_old[h] - m_new[h]);
                    }
                }
                uint32_t sr[NP][CH];
#pragma unroll
                for (int c = 0; c < NP; ++c) tmem_ld_32x32b<CH>(tmem + lane_off + (bi * NP + c) * N + h0, sr[c]);
                tmem_wait_ld();
#pragma unroll
                for (int h = 0; h < CH; ++h) {
                    float sx = 0.f;
#pragma unroll
                    for (int c = 0; c < NP; ++c) {
                        const float xv = valid[c] ? ex2(__uint_as_float(sr[c][h]) * p.scale_log2 - m_new[h]) : 0.f;
                        sx += xv;
                        if (h0 + h < n) {
                            uint8_t *phi = smem + C::kOffP + pbi * C::kPBufBytes + (r >> 6) * (C::kOW * 128) +
                                           (c * 2) * (C::kNPV * 128);
                            const int col = r & 63, hh = h0 + h;
                            const int off = hh * 128 + ((((col >> 3) ^ (hh & 7))) << 4) + (col & 7) * 2;
                            const __nv_bfloat16 hi = __float2bfloat16_rn(xv);
                            const __nv_bfloat16 lo2 = __float2bfloat16_rn(xv - __bfloat162float(hi));
                            *reinterpret_cast<__nv_bfloat16 *>(phi + off) = hi;
                            *reinterpret_cast<__nv_bfloat16 *>(phi + C::kNPV * 128 + off) = lo2;
                        }
                    }
                    l_part[h0 + h] = fmaf(l_part[h0 + h], alpha[h], sx);
                }
                if (tg == 0) {
                    store_vec<CH>(mrun_s + (i % 3) * NH + h0, m_new);
                    store_vec<CH>(alpha_s + (i % 4) * NH + h0, alpha);
                }
            }
            tc_fence_before_sync();
            mbar_arrive(&sfree[bi]);
            // ---- clear V rows outside [lo, hi): past the end of a sequence, before a window's
            // start, or in pages not copied; they may hold anything, NaN included
            if (valid_cnt < C::kTilePos || lo > 0) {
                const int sv = i % SV;
                if (!mbar_wait(&vfull[sv], (i / SV) & 1, ab)) { ok = false; break; }
                uint8_t *vrow = smem + C::kOffV + sv * C::kTileBytes + C::row_off(r);
#pragma unroll
                for (int c = 0; c < C::kColBoxes; ++c) {
                    // paired layout: box c holds the positions of part c; otherwise a row's
                    // boxes hold the dims of one position (part 0)
                    if (!valid[kPair ? c : 0]) {
                        uint4 *w = reinterpret_cast<uint4 *>(vrow + c * C::kHalfStride);
#pragma unroll
                        for (int k = 0; k < 8; ++k) w[k] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
            }
            fence_proxy_async_smem();
            mbar_arrive(&pfull[pbi]);
            if (tg == 0 && i < 128) GQA_TRACE_AT(kTrPFull + i, clock64());
            // ---- fold O of the tile before the previous one (its GEMM ran during two softmax steps)
            if (i - 2 >= piece_i0 && !fold_o(i - 2)) { ok = false; break; }

            if (last) {
                if (tg == 0) GQA_TRACE_AT(kTrPieceEnd + 2 * npe, clock64());
                // ---- l = sum over the 128 position slots, per head
                butterfly_reduce<NH, false>(l_part, lane);
                butterfly_store<NH, C::kHalve>(l_part, lane, lred + q4 * NH);
                if (!gsync(ab)) { ok = false; break; }        // also publishes tile i's alpha
                if (i - 1 >= piece_i0 && !fold_o(i - 1)) { ok = false; break; }
                if (!fold_o(i)) { ok = false; break; }
                if constexpr (kPair) {
                    // odd positions' share (rows 64..127) to the even rows, through the P
                    // buffer of tile i + 1: its last value GEMM is done (ofull of tile i was
                    // waited for) and the next P write follows the next tile's max barrier
                    float *xch = reinterpret_cast<float *>(smem + C::kOffP + ((i + 1) % PB) * C::kPBufBytes);
                    if (r >= 64) {
#pragma unroll
                        for (int h = 0; h < NH; ++h) xch[h * 64 + (r - 64)] = acc[h];
                    }
                    if (!gsync(ab)) { ok = false; break; }
                    if (r < 64) {
#pragma unroll
                        for (int h = 0; h < NH; ++h) acc[h] += xch[h * 64 + r];
                    }
                }
                const int seg = cur.b * G + cur.g;
                const long long seg_a = (long long)G * prefix[cur.b] + (long long)cur.g * cur.tiles;
                const bool owned = (piece_u0 == seg_a) && (cur.j + 1 == cur.tiles);
                float *orow = p.out + ((size_t)cur.b * p.H + (size_t)cur.g * n) * D;
                const int slot = range.chunk < 0 ? (int)blockIdx.x + seg : chunk_slot(p, range.chunk, range_piece);
                float *sp = owned ? nullptr : slot_ptr(p, slot, D);
                const int aoff = slot_acc_offset(n);
#pragma unroll
                for (int h0 = 0; h0 < NH; h0 += CH) {   // CH heads at a time (registers)
                    float L[CH];
                    reduce4<CH, false, NH>(lred + h0, L);
                    if (owned) {
#pragma unroll
                        for (int h = 0; h < CH; ++h)
                            if (h0 + h < n && has_dim) orow[(h0 + h) * D + odim] = acc[h0 + h] / L[h];
                    } else {
#pragma unroll
                        for (int h = 0; h < CH; ++h)
                            if (h0 + h < n && has_dim) sp[aoff + (h0 + h) * D + odim] = acc[h0 + h];
                        if (tg == 0) {
                            float mcur[CH];
                            load_vec<CH>(mrun_s + (i % 3) * NH + h0, mcur);
#pragma unroll
                            for (int h = 0; h < CH; ++h) {
                                if (h0 + h < n) {
                                    sp[h0 + h] = mcur[h];
                                    sp[n + h0 + h] = L[h];
                                }
                            }
                        }
                    }
                }
                // lred is next written after the next tile's max barrier, which every
                // thread reaches only after its reads here.
                if (tg == 0) GQA_TRACE_AT(kTrPieceEnd + 2 * npe + 1, clock64());
                ++npe;
                ++range_piece;
            }
            cursor_next(cur, prefix, p.B, G);
          }
        }
        if (tg == 0) GQA_TRACE_AT(kTrTiles, i);
        }
    } else if (kPaged) {
        // ================================================================ page-id warp (paged cache)
        // Walks the same tiles as the producer: lane k loads the block-table entry of
        // the tile's page k, then the warp copies the tile's K and then its V
        // (produce_paged_tile: one box per page, one page per lane).  Its id-ring
        // entry completes once K is issued; the producer thread paces its range
        // claims and Q copies on it and frees it (the ids and T_b are written into
        // it only for the appended-row path, which reads them).  One warp issues
        // both copies in order, K(i) V(i) K(i+1): K never runs ahead of V, which
        // measured faster than a second warp copying V beside this one.
        int rr = 0, ti = 0, k_copies = 0, v_copies = 0;
        bool ok = true;
        const uint64_t pol_kv = l2_policy_evict_first();
        const int *tlen = seq_len_array(prefix, p.B);   // T_b per sequence, when the batch leaves room
        const int ps = 1 << p.page_shift;
        while (ok) {
            const int rslot = rr % kRing;
            if (!mbar_wait(&rfull[rslot], (rr / kRing) & 1, ab)) break;
            const RangeEntry range = ring[rslot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&rempty[rslot]);
            ++rr;
            if (range.chunk == -2) break;
            Cursor cur = cursor_at(range.ub, prefix, p.B, G);
            int cached_b = -1, T = 0;
            for (int k = 0; k < range.len; ++k, ++ti) {
                const int slot = ti % C::kIdRing, sk = ti % SK, sv = ti % SV;
                if (cur.b != cached_b) {
                    cached_b = cur.b;
                    T = tlen ? tlen[cur.b] : seq_len_of(p, cur.b);
                }
                // the block-table entries first: their latency overlaps the waits below
                const int t0 = window_start(p, T), pos0 = tile_first_pos<C>(p, T, cur.j);
                const int32_t *trow = p.block_table + (size_t)cur.b * p.max_pages;
                int id = -1;
                if (lane < C::kIdMax) {
                    if (ps >= C::kTilePos) {
                        if (lane == 0) id = __ldg(trow + (pos0 >> p.page_shift));
                    } else {
                        const int pos = pos0 + lane * ps;
                        if (pos < pos0 + C::kTilePos && pos < T && pos + ps > t0) id = __ldg(trow + (pos >> p.page_shift));
                    }
                }
                bool go = true;
                if (lane == 0 && ti < 20) GQA_TRACE_AT(kTrProbe + 4 * ti, clock64());
                if (lane == 0)
                    go = (ti < C::kIdRing || mbar_wait(&idempty[slot], ((ti / C::kIdRing) - 1) & 1, ab)) &&
                         (ti < SK || mbar_wait(&kempty[sk], ((ti / SK) - 1) & 1, ab));
                if (lane == 0 && ti < 20) GQA_TRACE_AT(kTrProbe + 4 * ti + 1, clock64());
                if (!__shfl_sync(0xffffffffu, go, 0)) {
                    ok = false;
                    break;
                }
                int *e = ids_ring + slot * C::kIdStride;
                if (p.k_new) {   // the ids in shared memory, for the appended-row path
                    if (lane < C::kIdMax) e[lane] = id;
                    if (lane == 0) e[C::kIdMax] = T;
                    __syncwarp();
                }
                produce_paged_tile<C>(p, &tm_k, smem + C::kOffK + sk * C::kTileBytes, &kfull[sk], cur, T, pol_kv, id,
                                      lane, p.k_new, kstage + sk * C::kRowBytes, &kinfo[sk], p.k_dst, e);
                ++k_copies;
                if (lane == 0 && ti < 128) GQA_TRACE_AT(kTrKIssue + ti, clock64());
                if (lane == 0) mbar_arrive(&idfull[slot]);   // K of the tile is issued
                // ---- V of the tile
                if (lane == 0) go = ti < SV || mbar_wait(&vempty[sv], ((ti / SV) - 1) & 1, ab);
                if (lane == 0 && ti < 20) GQA_TRACE_AT(kTrProbe + 4 * ti + 2, clock64());
                if (!__shfl_sync(0xffffffffu, go, 0)) {
                    ok = false;
                    break;
                }
                produce_paged_tile<C>(p, &tm_v, smem + C::kOffV + sv * C::kTileBytes, &vfull[sv], cur, T, pol_kv, id,
                                      lane, p.v_new, vstage + sv * C::kRowBytes, &vinfo[sv], p.v_dst, e);
                ++v_copies;
                if (lane == 0 && ti < 128) GQA_TRACE_AT(kTrVIssue + ti, clock64());
                cursor_next(cur, prefix, p.B, G);
            }
        }
        if (lane == 0 && *s_abort) {
            // let this warp's copies in flight land before the CTA's shared memory is released
            for (int k = k_copies > SK ? k_copies - SK : 0; k < k_copies; ++k)
                mbar_wait_teardown(&kfull[k % SK], (k / SK) & 1);
            for (int k = v_copies > SV ? v_copies - SV : 0; k < v_copies; ++k)
                mbar_wait_teardown(&vfull[k % SV], (k / SV) & 1);
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (tid == 64) {
        GQA_TRACE_AT(kTrEnd, clock64());
        GQA_TRACE_AT(kTrGlobalEnd, globaltimer_ns());
    }
    if (warp == 0 && lane == 0 && *s_abort) {
        // let copies in flight land before the CTA's shared memory is released
        const int kown = kPaged ? 0 : kissued;   // paged: the page-id warp copies K and V
        for (int k = kown > SK ? kown - SK : 0; k < kown; ++k)
            mbar_wait_teardown(&kfull[k % SK], (k / SK) & 1);
        for (int k = vissued > SV ? vissued - SV : 0; k < vissued; ++k)
            mbar_wait_teardown(&vfull[k % SV], (k / SV) & 1);
        for (int k = qissued > QB ? qissued - QB : 0; k < qissued; ++k)
            mbar_wait_teardown(&qfull[k % QB], (k / QB) & 1);
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, bool kPair, int N, int NH, int kVar>
cudaError_t launch_tc_t(const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tq, const TailMaps &tails,
                        const DecodeParams &p, int ctas, cudaStream_t stream) {
    using C = TcCfg<D, kPair, N, NH, kVar>;
    auto kern = gqa_decode_tc_kernel<D, kPair, N, NH, kVar>;
    static unsigned long long attr_set = 0;   // one bit per device; setting twice is harmless
    int dev = 0;
    cudaGetDevice(&dev);
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(attr_set & bit)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set |= bit;
    }
    return launch_pdl(kern, ctas, C::kThreads, C::kSmemBytes, stream, tk, tv, tq, tails, p);
}

template <int D, bool kPair, int kVar>
cudaError_t launch_tc_d(const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tq, const TailMaps &tails,
                        const DecodeParams &p, int ctas, cudaStream_t stream) {
    const int n = p.n;
    if (n <= 1) return launch_tc_t<D, kPair, 16, 1, kVar>(tk, tv, tq, tails, p, ctas, stream);
    if (n <= 2) return launch_tc_t<D, kPair, 16, 2, kVar>(tk, tv, tq, tails, p, ctas, stream);
    if (n <= 4) return launch_tc_t<D, kPair, 16, 4, kVar>(tk, tv, tq, tails, p, ctas, stream);
    if (n <= 8) return launch_tc_t<D, kPair, 16, 8, kVar>(tk, tv, tq, tails, p, ctas, stream);
    if (n <= 16) return launch_tc_t<D, kPair, 16, 16, kVar>(tk, tv, tq, tails, p, ctas, stream);
    if constexpr (!kPair) {
        if (n <= 32) return launch_tc_t<D, kPair, 32, 32, kVar>(tk, tv, tq, tails, p, ctas, stream);
        return launch_tc_t<D, kPair, 64, 64, kVar>(tk, tv, tq, tails, p, ctas, stream);
    }
    return cudaErrorNotSupported;
}

template <int kVar>
cudaError_t launch_tc_layout(const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tq,
                             const TailMaps &tails, const DecodeParams &p, int D, bool paired, int ctas,
                             cudaStream_t stream) {
    if (D == 128) return launch_tc_d<128, false, kVar>(tk, tv, tq, tails, p, ctas, stream);
    if (paired) return launch_tc_d<64, true, kVar>(tk, tv, tq, tails, p, ctas, stream);
    return launch_tc_d<64, false, kVar>(tk, tv, tq, tails, p, ctas, stream);
}

}  // namespace

int tc_max_heads() { return 64; }

int tc_rows_for(int n) { return n <= 16 ? 16 : (n <= 32 ? 32 : 64); }

bool tc_paired(int D, int Lmax, int n) { return D == 64 && Lmax % 2 == 0 && n <= 16; }

cudaError_t launch_decode_tc(const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tq,
                             const TailMaps &tails, const DecodeParams &p, int D, bool paired, int ctas,
                             cudaStream_t stream) {
    // the variants run the instances built for them
    if (p.block_table) return launch_tc_layout<2>(tk, tv, tq, tails, p, D, paired, ctas, stream);
    if (p.window > 0 || p.k_new) return launch_tc_layout<1>(tk, tv, tq, tails, p, D, paired, ctas, stream);
    return launch_tc_layout<0>(tk, tv, tq, tails, p, D, paired, ctas, stream);
}

}  // namespace gqa
