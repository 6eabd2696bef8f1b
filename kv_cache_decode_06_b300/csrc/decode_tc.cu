// GQA decode on the fifth-generation tensor cores (tcgen05 + TMEM).
//
// The query heads of one group form the N side of two small GEMMs per
// 128-position tile, with the positions (scores) or the head dims (values) on
// the M side, so every K/V tile read from HBM serves all n = H/G heads:
//   S^T [128 pos x N]  = K_tile [128 x d] . Q_g^T [d x N]       (K-major A and B)
//   O^T [d x N]        = V_tile^T [d x 128] . P^T [128 x N]     (MN-major A, K-major B)
// N is n rounded up to at least 16 (the extra columns are never read).
// Operands come from 128-byte-swizzled shared memory written by TMA;
// accumulators live in TMEM.  P is split into bf16 hi + lo parts (two MMAs), so
// the probabilities enter the value GEMM with ~16 significant bits, not 8.
// ["Grouped-query attention (GQA)" concept page, "Implementation sketch",
//  decode-step pseudocode; arxiv:2305.13245 §2.2]
//
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = MMA issuer and TMEM
// owner, warps 2-5 = softmax + epilogue (thread <-> TMEM lane: a position of
// the tile for S, a head dim for O).  Per tile the softmax group
//   1. loads its S row, reduces the per-head maximum over the 128 positions
//      (transposed butterfly in the warp, then the 4 warps via shared memory),
//   2. writes P(i) and hands it to the MMA warp,
//   3. folds the previous tile's O into register accumulators with that tile's
//      rescale factor (so TMEM never needs rescaling).
// The MMA warp issues each GEMM as soon as its own inputs are ready, so the value
// GEMM of tile i never waits for tile i+1's data.  Work split, pieces and the
// last-arriver combine are shared with the CUDA-core path.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "decode_common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

namespace gqa {

namespace {

constexpr int kSmemLimit = 232448;   // 227 KB opt-in per CTA

constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

// D = head dim, N = MMA N (>= 16), NH = heads held per thread (power of two >= n).
template <int D, int N, int NH>
struct TcCfg {
    static constexpr int kBoxes = D / kBoxCols;
    static constexpr int kTileBytes = kBoxes * kBoxBytes;        // one K or V tile (128 positions)
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kQBytes = kBoxes * N * 128;             // one Q buffer (N rows x d)
    static constexpr int kPBytes = 2 * N * 128;                  // one P part: N rows x 128 positions
    static constexpr int kMisc = 8192 + (kMaxBatch + 1) * 4 + 1024;
    static constexpr int kQBuf = (2 * kQBytes + 4 * kPBytes + 2 * kStageBytes + kMisc <= kSmemLimit) ? 2 : 1;
    static constexpr int kFixed = kQBuf * kQBytes + 4 * kPBytes;
    static constexpr int kStagesFit = (kSmemLimit - kMisc - kFixed) / kStageBytes;
    static constexpr int kStages = kStagesFit > 6 ? 6 : kStagesFit;
    static_assert(kStages >= 2, "shared memory too small for two stages");
    static constexpr int kOffQ = kStages * kStageBytes;
    static constexpr int kOffP = kOffQ + kQBuf * kQBytes;        // [2 buffers][hi, lo]
    static constexpr int kOffRed = kOffP + 4 * kPBytes;          // f32 [2][4][NH] per-warp tile maxima
    static constexpr int kOffLred = kOffRed + 2 * 4 * NH * 4;    // f32 [4][NH] per-warp l sums
    static constexpr int kOffM = kOffLred + 4 * NH * 4;          // f32 [3][NH] running max after tile i
    static constexpr int kOffA = kOffM + 3 * NH * 4;             // f32 [3][NH] rescale factor of tile i
    static constexpr int kOffPrefix = kOffA + 3 * NH * 4;        // i32 [kMaxBatch + 1]
    static constexpr int kOffScratch = kOffPrefix + (kMaxBatch + 1) * 4;
    static constexpr int kOffBar = (kOffScratch + 32 * 4 + 7) / 8 * 8;
    // barriers: kfull[S] vfull[S] kvempty[S] qfull[QB] qempty[QB] sfull[2] sfree[2] pfull[2]
    //           ofull[2] ofree[2] red[2] grp done
    static constexpr int kNumBars = 3 * kStages + 2 * kQBuf + 12 + 2;
    static constexpr int kOffFlags = kOffBar + kNumBars * 8;     // abort, last, tmem base
    static constexpr int kSmemBytes = kOffFlags + 16 + 1024;
    static_assert(kSmemBytes <= kSmemLimit, "shared memory layout too large");
    static constexpr int kThreads = 192;
    static constexpr int kTmemCols = (4 * N <= 32) ? 32 : (4 * N <= 64) ? 64 : (4 * N <= 128) ? 128 : 256;
    static constexpr int kPvM = (D == 128) ? 128 : 64;
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

struct GroupSync128 {
    uint64_t *bar;
    uint32_t phase;
    __device__ bool operator()(const AbortState &ab) {
        mbar_arrive(bar);
        const bool ok = mbar_wait(bar, phase & 1u, ab);
        ++phase;
        return ok;
    }
};

template <int D, int N, int NH>
__global__ void __launch_bounds__(192, 1)
    gqa_decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_q, const DecodeParams p) {
    using C = TcCfg<D, N, NH>;
    constexpr int S = C::kStages, QB = C::kQBuf;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *red = reinterpret_cast<float *>(smem + C::kOffRed);
    float *lred = reinterpret_cast<float *>(smem + C::kOffLred);
    float *mrun_s = reinterpret_cast<float *>(smem + C::kOffM);
    float *alpha_s = reinterpret_cast<float *>(smem + C::kOffA);
    int *prefix = reinterpret_cast<int *>(smem + C::kOffPrefix);
    int *scratch = reinterpret_cast<int *>(smem + C::kOffScratch);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    uint64_t *kfull = bars, *vfull = kfull + S, *kvempty = vfull + S;
    uint64_t *qfull = kvempty + S, *qempty = qfull + QB;
    uint64_t *sfull = qempty + QB, *sfree = sfull + 2, *pfull = sfree + 2, *ofull = pfull + 2, *ofree = ofull + 2;
    uint64_t *redbar = ofree + 2, *grp = redbar + 2, *done = grp + 1;
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + C::kOffFlags);
    volatile int *s_last = s_abort + 1;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + C::kOffFlags + 8);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = gridDim.x;
    const AbortState ab{s_abort, p.flags};

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&kfull[s], 1);
            mbar_init(&vfull[s], 1);
            mbar_init(&kvempty[s], 1);
        }
        for (int s = 0; s < QB; ++s) {
            mbar_init(&qfull[s], 1);
            mbar_init(&qempty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sfull[s], 1);
            mbar_init(&sfree[s], 128);
            mbar_init(&pfull[s], 128);
            mbar_init(&ofull[s], 1);
            mbar_init(&ofree[s], 128);
            mbar_init(&redbar[s], 4);
        }
        mbar_init(grp, 128);
        mbar_init(done, 1);
        *s_abort = 0;
        *s_last = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_q);
    }
    if (warp == 1) {
        tmem_alloc(s_tmem, C::kTmemCols);
        tmem_relinquish();
    }
    build_prefix(p.seq_lens, p.B, p.Lmax, prefix, scratch, p.flags);   // ends with __syncthreads
    tc_fence_after_sync();
    const uint32_t tmem = *s_tmem;

    const int G = p.G, n = p.n;
    const long long W = (long long)G * prefix[p.B];
    const int Pw = (int)(W < P ? W : P);
    long long u0 = 0, u1 = 0;
    if ((int)blockIdx.x < Pw) {
        u0 = range_start(blockIdx.x, W, Pw);
        u1 = range_start(blockIdx.x + 1, W, Pw);
    }
    const int ntiles = (int)(u1 - u0);
    int issued = 0, qissued = 0;

    if (warp == 0) {
        // ================================================================ producer
        if (lane == 0 && ntiles > 0) {
            const uint64_t pol_kv = l2_policy_evict_first();
            const uint64_t pol_q = l2_policy_evict_last();
            Cursor cur = cursor_at(u0, prefix, p.B, G);
            int piece = 0;
            for (int i = 0; i < ntiles; ++i) {
                const bool first = (i == 0) || (cur.j == 0);
                const bool last = (i + 1 == ntiles) || (cur.j + 1 == cur.tiles);
                if (first) {
                    const int qb = piece % QB;
                    if (piece >= QB && !mbar_wait(&qempty[qb], ((piece / QB) - 1) & 1, ab)) break;
                    mbar_arrive_expect_tx(&qfull[qb], C::kQBytes);
                    uint8_t *qdst = smem + C::kOffQ + qb * C::kQBytes;
                    const int y = cur.b * p.H + cur.g * n;
#pragma unroll
                    for (int c = 0; c < C::kBoxes; ++c)
                        tma_load_2d(qdst + c * N * 128, &tm_q, c * kBoxCols, y, &qfull[qb], pol_q);
                    ++qissued;
                }
                const int st = i % S;
                if (i >= S && !mbar_wait(&kvempty[st], ((i / S) - 1) & 1, ab)) break;
                uint8_t *kdst = smem + st * C::kStageBytes;
                uint8_t *vdst = kdst + C::kTileBytes;
                const int z = cur.b * G + cur.g, y = cur.j * kTile;
                mbar_arrive_expect_tx(&kfull[st], C::kTileBytes);
#pragma unroll
                for (int c = 0; c < C::kBoxes; ++c)
                    tma_load_3d(kdst + c * kBoxBytes, &tm_k, c * kBoxCols, y, z, &kfull[st], pol_kv);
                mbar_arrive_expect_tx(&vfull[st], C::kTileBytes);
#pragma unroll
                for (int c = 0; c < C::kBoxes; ++c)
                    tma_load_3d(vdst + c * kBoxBytes, &tm_v, c * kBoxCols, y, z, &vfull[st], pol_kv);
                ++issued;
                if (last) ++piece;
                cursor_next(cur, prefix, p.B, G);
            }
        }
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        if (lane == 0 && ntiles > 0) {
            constexpr uint32_t idS = idesc_bf16_f32(128, N, false, false);
            constexpr uint32_t idPV = idesc_bf16_f32(C::kPvM, N, true, false);
            const uint32_t sbase = smem_addr(smem);
            Cursor cur = cursor_at(u0, prefix, p.B, G);
            int s_i = 0, pv_i = 0, piece = 0;
            uint32_t idle = 0;
            uint64_t idle_t0 = 0;
            while (pv_i < ntiles) {
                bool progress = false;
                // ---- scores of tile s_i: needs its K, its piece's Q and a free S buffer
                if (s_i < ntiles) {
                    const bool first = (s_i == 0) || (cur.j == 0);
                    const bool last = (s_i + 1 == ntiles) || (cur.j + 1 == cur.tiles);
                    const int st = s_i % S, bi = s_i & 1, qb = piece % QB;
                    if ((!first || mbar_test_wait(&qfull[qb], (piece / QB) & 1)) &&
                        mbar_test_wait(&kfull[st], (s_i / S) & 1) &&
                        (s_i < 2 || mbar_test_wait(&sfree[bi], ((s_i >> 1) - 1) & 1))) {
                        tc_fence_after_sync();
                        const uint32_t kb = sbase + st * C::kStageBytes;
                        const uint32_t qbase = sbase + C::kOffQ + qb * C::kQBytes;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk)
                            umma_bf16(tmem + bi * N,
                                      sdesc_sw128(kb + (kk >> 2) * kBoxBytes + (kk & 3) * 32, 16, 1024),
                                      sdesc_sw128(qbase + (kk >> 2) * (N * 128) + (kk & 3) * 32, 16, 1024), idS,
                                      kk != 0);
                        umma_commit(&sfull[bi]);
                        if (last) {
                            umma_commit(&qempty[qb]);
                            ++piece;
                        }
                        cursor_next(cur, prefix, p.B, G);
                        ++s_i;
                        progress = true;
                    }
                }
                // ---- values of tile pv_i: needs its V, its P and a free O buffer
                if (pv_i < s_i) {
                    const int st = pv_i % S, bi = pv_i & 1;
                    if (mbar_test_wait(&vfull[st], (pv_i / S) & 1) && mbar_test_wait(&pfull[bi], (pv_i >> 1) & 1) &&
                        (pv_i < 2 || mbar_test_wait(&ofree[bi], ((pv_i >> 1) - 1) & 1))) {
                        tc_fence_after_sync();
                        const uint32_t vb = sbase + st * C::kStageBytes + C::kTileBytes;
                        const uint32_t d_o = tmem + 2 * N + bi * N;
#pragma unroll
                        for (int part = 0; part < 2; ++part) {
                            const uint32_t pb = sbase + C::kOffP + (bi * 2 + part) * C::kPBytes;
#pragma unroll
                            for (int kk = 0; kk < kTile / 16; ++kk)
                                umma_bf16(d_o, sdesc_sw128(vb + kk * 2048, kBoxBytes, 1024),
                                          sdesc_sw128(pb + (kk >> 2) * (N * 128) + (kk & 3) * 32, 16, 1024), idPV,
                                          (part | kk) != 0);
                        }
                        umma_commit(&ofull[bi]);
                        umma_commit(&kvempty[st]);
                        ++pv_i;
                        progress = true;
                    }
                }
                if (progress) {
                    idle = 0;
                } else {
                    if (idle == 0) idle_t0 = globaltimer_ns();
                    if ((++idle & 63u) == 0) {
                        if (*s_abort) break;
                        if (globaltimer_ns() - idle_t0 > kWaitLimitNs) {
                            *s_abort = 1;
                            atomicOr(p.flags, 0x2u /* GQA_FLAG_WAIT_TIMEOUT */);
                            break;
                        }
                    }
                }
            }
            umma_commit(done);
            mbar_wait_teardown(done, 0);
        }
    } else {
        // ================================================================ softmax + epilogue
        const int q4 = warp & 3;                 // TMEM lane quadrant of this warp
        const int r = q4 * 32 + lane;            // tile position (S) / head dim (O, d = 128)
        const int tg = tid - 64;                 // 0..127 within the group
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        // dim held in the O accumulator by this thread (M = 64 puts 16 rows in each quadrant)
        const int odim = (D == 128) ? r : q4 * 16 + lane;
        const bool has_dim = (D == 128) || lane < 16;
        zero_empty_sequences<D>(p, prefix, P, tg, 128);
        GroupSync128 gsync{grp, 0};
        float l_part[NH], acc[NH];
        Cursor cur = (ntiles > 0) ? cursor_at(u0, prefix, p.B, G) : Cursor{0, 0, 0, 1};
        int seq_b = 0;
        long long piece_u0 = u0;
        int piece_i0 = 0;
        bool ok = true;

        // fold O of tile i into acc with that tile's rescale factor
        auto fold_o = [&](int i) -> bool {
            const int bi = i & 1;
            if (!mbar_wait(&ofull[bi], (i >> 1) & 1, ab)) return false;
            tc_fence_after_sync();
            uint32_t o[NH];
            tmem_ld_32x32b<NH>(tmem + lane_off + 2 * N + bi * N, o);
            tmem_wait_ld();
            tc_fence_before_sync();
            mbar_arrive(&ofree[bi]);
            const float *al = alpha_s + (i % 3) * NH;
#pragma unroll
            for (int h = 0; h < NH; ++h) acc[h] = fmaf(acc[h], al[h], __uint_as_float(o[h]));
            return true;
        };

        for (int i = 0; i < ntiles && ok; ++i) {
            const long long u = u0 + i;
            const bool first = (i == 0) || (cur.j == 0);
            const bool last = (i + 1 == ntiles) || (cur.j + 1 == cur.tiles);
            const int st = i % S, bi = i & 1;
            if (first) {
                piece_u0 = u;
                piece_i0 = i;
                seq_b = clamp_seq(__ldg(p.seq_lens + cur.b), p.Lmax);
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                    l_part[h] = 0.f;
                    acc[h] = 0.f;
                }
            }
            // ---- scores of this tile: S^T row r (heads 0..NH-1)
            if (!mbar_wait(&sfull[bi], (i >> 1) & 1, ab)) { ok = false; break; }
            tc_fence_after_sync();
            uint32_t sraw[NH];
            tmem_ld_32x32b<NH>(tmem + lane_off + bi * N, sraw);
            tmem_wait_ld();
            tc_fence_before_sync();
            mbar_arrive(&sfree[bi]);
            const int valid_cnt = seq_b - cur.j * kTile;          // >= 1
            const bool valid = r < valid_cnt;
            float x[NH], red_v[NH];
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                x[h] = valid ? __uint_as_float(sraw[h]) * p.scale_log2 : -INFINITY;
                red_v[h] = x[h];
            }
            butterfly_reduce<NH, true>(red_v, lane);
            butterfly_store<NH, C::kHalve>(red_v, lane, red + (bi * 4 + q4) * NH);
            __syncwarp();
            if (lane == 0) mbar_arrive(&redbar[bi]);
            if (!mbar_wait(&redbar[bi], (i >> 1) & 1, ab)) { ok = false; break; }
            const float *mprev = mrun_s + ((i + 2) % 3) * NH;    // state after tile i-1
            float *mcur = mrun_s + (i % 3) * NH;
            float *acur = alpha_s + (i % 3) * NH;
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                const float *rr = red + bi * 4 * NH + h;
                const float tmax = fmaxf(fmaxf(rr[0], rr[NH]), fmaxf(rr[2 * NH], rr[3 * NH]));
                const float m_old = (i == piece_i0) ? -INFINITY : mprev[h];
                const float m_new = fmaxf(m_old, tmax);           // finite: every tile has a valid position
                const float alpha = exp2f(m_old - m_new);         // 0 on the first tile of a piece
                x[h] = exp2f(x[h] - m_new);                       // 0 at invalid positions
                l_part[h] = fmaf(l_part[h], alpha, x[h]);
                if (tg == 0) {
                    mcur[h] = m_new;
                    acur[h] = alpha;
                }
            }
            // ---- the last tile of a sequence: clear V rows past the end (they may hold NaN)
            if (valid_cnt < kTile) {
                if (!mbar_wait(&vfull[st], (i / S) & 1, ab)) { ok = false; break; }
                if (!valid) {
                    uint8_t *vrow = smem + st * C::kStageBytes + C::kTileBytes + r * 128;
#pragma unroll
                    for (int c = 0; c < C::kBoxes; ++c) {
                        uint4 *w = reinterpret_cast<uint4 *>(vrow + c * kBoxBytes);
#pragma unroll
                        for (int k = 0; k < 8; ++k) w[k] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
            // ---- probabilities to shared memory as bf16 hi + lo (K-major, 128-byte swizzle)
            {
                uint8_t *phi = smem + C::kOffP + (bi * 2 + 0) * C::kPBytes + (r >> 6) * (N * 128);
                uint8_t *plo = phi + C::kPBytes;
                const int c = r & 63;
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                    if (h < n) {
                        const int off = h * 128 + ((((c >> 3) ^ (h & 7))) << 4) + (c & 7) * 2;
                        const __nv_bfloat16 hi = __float2bfloat16_rn(x[h]);
                        const __nv_bfloat16 lo = __float2bfloat16_rn(x[h] - __bfloat162float(hi));
                        *reinterpret_cast<__nv_bfloat16 *>(phi + off) = hi;
                        *reinterpret_cast<__nv_bfloat16 *>(plo + off) = lo;
                    }
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(&pfull[bi]);
            // ---- fold the previous tile's O (its GEMM ran while this tile's softmax did)
            if (i > piece_i0 && !fold_o(i - 1)) { ok = false; break; }

            if (last) {
                // ---- l = sum over the 128 position slots, per head
                butterfly_reduce<NH, false>(l_part, lane);
                butterfly_store<NH, C::kHalve>(l_part, lane, lred + q4 * NH);
                if (!gsync(ab)) { ok = false; break; }        // also publishes tile i's alpha
                if (!fold_o(i)) { ok = false; break; }
                const int seg = cur.b * G + cur.g;
                const long long seg_a = (long long)G * prefix[cur.b] + (long long)cur.g * cur.tiles;
                const bool owned = (piece_u0 == seg_a) && (cur.j + 1 == cur.tiles);
                float *orow = p.out + ((size_t)cur.b * p.H + (size_t)cur.g * n) * D;
                float *sp = slot_ptr(p, blockIdx.x + seg, D);
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                    if (h < n) {
                        const float L = lred[h] + lred[NH + h] + lred[2 * NH + h] + lred[3 * NH + h];
                        if (owned) {
                            if (has_dim) orow[h * D + odim] = acc[h] / L;
                        } else {
                            if (has_dim) sp[2 * n + h * D + odim] = acc[h];
                            if (tg == 0) {
                                sp[h] = mcur[h];
                                sp[n + h] = L;
                            }
                        }
                    }
                }
                if (!owned) {
                    __threadfence();
                    if (!gsync(ab)) { ok = false; break; }
                    const int c_lo = cta_of_tile(seg_a, W, Pw);
                    const int c_hi = cta_of_tile(seg_a + cur.tiles - 1, W, Pw);
                    if (tg == 0) {
                        const int prev = atomicAdd(p.counters + seg, 1);
                        *s_last = (prev == c_hi - c_lo) ? 1 : 0;
                    }
                    if (!gsync(ab)) { ok = false; break; }
                    if (*s_last) {
                        __threadfence();
                        combine_segment<D>(p, c_lo + seg, c_hi - c_lo + 1, cur.b, cur.g, tg, 128);
                        if (tg == 0) atomicExch(p.counters + seg, 0);
                    }
                }
                if (!gsync(ab)) { ok = false; break; }   // lred and s_last are reused by the next piece
            }
            cursor_next(cur, prefix, p.B, G);
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0 && lane == 0 && *s_abort) {
        // let copies in flight land before the CTA's shared memory is released
        for (int k = issued > S ? issued - S : 0; k < issued; ++k) {
            mbar_wait_teardown(&kfull[k % S], (k / S) & 1);
            mbar_wait_teardown(&vfull[k % S], (k / S) & 1);
        }
        for (int k = qissued > QB ? qissued - QB : 0; k < qissued; ++k)
            mbar_wait_teardown(&qfull[k % QB], (k / QB) & 1);
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, int N, int NH>
cudaError_t launch_tc_t(const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tq, const DecodeParams &p,
                        int ctas, cudaStream_t stream) {
    using C = TcCfg<D, N, NH>;
    auto kern = gqa_decode_tc_kernel<D, N, NH>;
    static unsigned long long attr_set = 0;   // one bit per device; setting twice is harmless
    int dev = 0;
    cudaGetDevice(&dev);
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(attr_set & bit)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set |= bit;
    }
    kern<<<ctas, C::kThreads, C::kSmemBytes, stream>>>(tk, tv, tq, p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_tc_d(const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tq, const DecodeParams &p,
                        int ctas, cudaStream_t stream) {
    const int n = p.n;
    if (n <= 1) return launch_tc_t<D, 16, 1>(tk, tv, tq, p, ctas, stream);
    if (n <= 2) return launch_tc_t<D, 16, 2>(tk, tv, tq, p, ctas, stream);
    if (n <= 4) return launch_tc_t<D, 16, 4>(tk, tv, tq, p, ctas, stream);
    if (n <= 8) return launch_tc_t<D, 16, 8>(tk, tv, tq, p, ctas, stream);
    if (n <= 16) return launch_tc_t<D, 16, 16>(tk, tv, tq, p, ctas, stream);
    if (n <= 32) return launch_tc_t<D, 32, 32>(tk, tv, tq, p, ctas, stream);
    return launch_tc_t<D, 64, 64>(tk, tv, tq, p, ctas, stream);
}

}  // namespace

int tc_max_heads() { return 64; }

int tc_rows_for(int n) { return n <= 16 ? 16 : (n <= 32 ? 32 : 64); }

cudaError_t launch_decode_tc(const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tq,
                             const DecodeParams &p, int D, int ctas, cudaStream_t stream) {
    if (D == 128) return launch_tc_d<128>(tk, tv, tq, p, ctas, stream);
    return launch_tc_d<64>(tk, tv, tq, p, ctas, stream);
}

}  // namespace gqa
