// GQA decode on CUDA cores (fp32 FMA), for groups of up to 8 query heads.
//
// One CTA = 4 compute warps + 1 producer warp.  The producer streams each
// 128-position K and V tile of the CTA's range into a ring of shared-memory
// stages with TMA (128-byte swizzled boxes, read once from HBM with an
// evict-first L2 policy).  Every K/V tile serves all n = H/G query heads of its
// group.  Compute warp w owns positions 32w..32w+31 of every tile:
//   scores:  lane = position, s[h] = q[h] . k[t] with q broadcast from shared
//            memory (the swizzle makes the 32 row reads conflict-free);
//   softmax: running max m[h] per warp (base-2 units), lane-private running sum
//            l[h], probabilities p[h][t] to a warp-private buffer;
//   values:  lane = output dims, acc[h][dims] += p[h][t] * v[t][dims].
// At the end of a piece the four warps' (m, l, acc) are merged in shared memory
// and written out, or left as a partial for the split-combine kernel.
// ["Grouped-query attention (GQA)" concept page, "Implementation sketch",
//  decode-step pseudocode; arxiv:2305.13245 §2.2]
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "decode_common.cuh"
#include "launch.h"

namespace gqa {

namespace {

template <int D, int NMAX>
struct SimtCfg {
    static constexpr int kBoxes = D / kBoxCols;
    static constexpr int kTileBytes = kBoxes * kBoxBytes;     // one K or V tile
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kStages = (D == 128) ? 3 : 6;
    static constexpr int kWarps = 4;                          // compute warps
    static constexpr int kThreads = (kWarps + 1) * 32;
    static constexpr int kDpl = D / 32;                       // output dims per lane
    static constexpr int kOffQ = kStages * kStageBytes;                    // f32 [2][NMAX][D]
    static constexpr int kOffP = kOffQ + 2 * NMAX * D * 4;                 // f32 [W][NMAX][32]
    static constexpr int kOffAcc = kOffP + kWarps * NMAX * 32 * 4;         // f32 [W][NMAX][D]
    static constexpr int kOffM = kOffAcc + kWarps * NMAX * D * 4;          // f32 [W][NMAX]
    static constexpr int kOffL = kOffM + kWarps * NMAX * 4;                // f32 [W][NMAX]
    static constexpr int kOffPrefix = kOffL + kWarps * NMAX * 4;           // i32 [kMaxBatch + 1]
    static constexpr int kOffScratch = kOffPrefix + (kMaxBatch + 1) * 4;   // i32 [33]
    static constexpr int kOffBar = (kOffScratch + 33 * 4 + 7) / 8 * 8;    // u64 full[S], empty[S], grp
    static constexpr int kOffFlags = kOffBar + (2 * kStages + 1) * 8;      // abort, last
    static constexpr int kSmemBytes = kOffFlags + 16 + 1024;               // + alignment slack
};

template <int D, int NMAX>
__global__ void __launch_bounds__(SimtCfg<D, NMAX>::kThreads, 1)
    gqa_decode_simt_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                           const DecodeParams p) {
    using C = SimtCfg<D, NMAX>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *q_s = reinterpret_cast<float *>(smem + C::kOffQ);
    float *p_s = reinterpret_cast<float *>(smem + C::kOffP);
    float *acc_s = reinterpret_cast<float *>(smem + C::kOffAcc);
    float *m_s = reinterpret_cast<float *>(smem + C::kOffM);
    float *l_s = reinterpret_cast<float *>(smem + C::kOffL);
    int *prefix = reinterpret_cast<int *>(smem + C::kOffPrefix);
    int *scratch = reinterpret_cast<int *>(smem + C::kOffScratch);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    uint64_t *empty = full + C::kStages;
    uint64_t *grp = empty + C::kStages;
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + C::kOffFlags);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = gridDim.x;
    const AbortState ab{s_abort, p.flags};

    if (tid == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], C::kWarps);
        }
        mbar_init(grp, C::kWarps * 32);
        *s_abort = 0;
        fence_mbar_init();
    }
    if (tid == C::kWarps * 32) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    // Inputs and outputs are touched only once the grids this one depends on
    // have completed.
    griddep_wait();
    griddep_launch_dependents();
    build_prefix(p, 7, prefix, scratch, p.flags);  // ends with __syncthreads

    const int G = p.G, n = p.n;
    const long long W = (long long)G * prefix[p.B];
    // Never more working CTAs than tiles, so every working range is non-empty
    // and every CTA between a segment's first and last owner holds a piece.
    const int Pw = (int)(W < P ? W : P);
    long long u0 = 0, u1 = 0;
    if ((int)blockIdx.x < Pw) {
        u0 = range_start(blockIdx.x, W, Pw);
        u1 = range_start(blockIdx.x + 1, W, Pw);
    }
    int issued = 0;

    if (warp == C::kWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && u0 < u1) {
            const uint64_t pol = l2_policy_evict_first();
            Cursor cur = cursor_at(u0, prefix, p.B, G);
            for (long long u = u0; u < u1; ++u, ++issued) {
                const int st = issued % C::kStages;
                if (issued >= C::kStages && !mbar_wait(&empty[st], ((issued / C::kStages) - 1) & 1, ab)) break;
                mbar_arrive_expect_tx(&full[st], C::kStageBytes);
                uint8_t *kdst = smem + st * C::kStageBytes;
                uint8_t *vdst = kdst + C::kTileBytes;
                const int z = cur.b * G + cur.g, y = cur.j * kTile;
#pragma unroll
                for (int c = 0; c < C::kBoxes; ++c)
                    tma_load_3d(kdst + c * kBoxBytes, &tm_k, c * kBoxCols, y, z, &full[st], pol);
#pragma unroll
                for (int c = 0; c < C::kBoxes; ++c)
                    tma_load_3d(vdst + c * kBoxBytes, &tm_v, c * kBoxCols, y, z, &full[st], pol);
                cursor_next(cur, prefix, p.B, G);
            }
        }
    } else {
        // ------------------------------------------------------------ compute
        zero_empty_sequences<D>(p, prefix, P, tid, C::kWarps * 32);
        GroupSync gsync{grp, 0};
        const uint32_t kbase = smem_addr(smem);
        float m_run[NMAX], l_lane[NMAX], acc[NMAX][C::kDpl];
        int piece = 0, seq_b = 0;
        long long piece_u0 = u0;
        Cursor cur = (u0 < u1) ? cursor_at(u0, prefix, p.B, G) : Cursor{0, 0, 0, 1};
        int it = 0;
        for (long long u = u0; u < u1; ++u, ++it) {
            const bool first = (u == u0) || (cur.j == 0);
            const bool last = (u + 1 == u1) || (cur.j + 1 == cur.tiles);
            const float *qp = q_s + (piece & 1) * NMAX * D;
            if (first) {
                piece_u0 = u;
                seq_b = seq_len_of(p, cur.b);
                const __nv_bfloat16 *qg = p.q + ((size_t)cur.b * p.H + (size_t)cur.g * n) * D;
                float *qw = q_s + (piece & 1) * NMAX * D;
                for (int x = tid; x < n * D; x += C::kWarps * 32) qw[x] = __bfloat162float(qg[x]);
#pragma unroll
                for (int h = 0; h < NMAX; ++h) {
                    m_run[h] = -INFINITY;
                    l_lane[h] = 0.f;
#pragma unroll
                    for (int k = 0; k < C::kDpl; ++k) acc[h][k] = 0.f;
                }
                if (!gsync(ab)) break;
            }
            const int st = it % C::kStages;
            if (!mbar_wait(&full[st], (it / C::kStages) & 1, ab)) break;

            // ---- scores: lane = position
            const int row = warp * 32 + lane;
            const int t0w = cur.j * kTile + warp * 32;
            const bool valid = (t0w + lane) < seq_b;
            const uint32_t kt = kbase + st * C::kStageBytes;
            float s[NMAX];
#pragma unroll
            for (int h = 0; h < NMAX; ++h) s[h] = 0.f;
#pragma unroll
            for (int c = 0; c < D / 8; ++c) {
                const uint32_t a = kt + (c >> 3) * kBoxBytes + row * 128 + ((((c & 7) ^ (row & 7))) << 4);
                const uint4 kk = lds128(a);
                const float k0 = bf16lo(kk.x), k1 = bf16hi(kk.x), k2 = bf16lo(kk.y), k3 = bf16hi(kk.y);
                const float k4 = bf16lo(kk.z), k5 = bf16hi(kk.z), k6 = bf16lo(kk.w), k7 = bf16hi(kk.w);
#pragma unroll
                for (int h = 0; h < NMAX; ++h) {
                    if (h < n) {
                        const float4 qa = *reinterpret_cast<const float4 *>(qp + h * D + c * 8);
                        const float4 qb = *reinterpret_cast<const float4 *>(qp + h * D + c * 8 + 4);
                        float x = s[h];
                        x = fmaf(qa.x, k0, x); x = fmaf(qa.y, k1, x); x = fmaf(qa.z, k2, x); x = fmaf(qa.w, k3, x);
                        x = fmaf(qb.x, k4, x); x = fmaf(qb.y, k5, x); x = fmaf(qb.z, k6, x); x = fmaf(qb.w, k7, x);
                        s[h] = x;
                    }
                }
            }
            // ---- online softmax (base 2), per warp
            float *pw = p_s + warp * NMAX * 32;
#pragma unroll
            for (int h = 0; h < NMAX; ++h) {
                if (h < n) {
                    const float x = valid ? s[h] * p.scale_log2 : -INFINITY;
                    float mt = x;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
                    const float m_new = fmaxf(m_run[h], mt);
                    const bool none = (m_new == -INFINITY);     // no valid position seen yet
                    const float alpha = none ? 1.f : ex2(m_run[h] - m_new);
                    const float pr = none ? 0.f : ex2(x - m_new);
                    m_run[h] = m_new;
                    l_lane[h] = fmaf(l_lane[h], alpha, pr);
#pragma unroll
                    for (int k = 0; k < C::kDpl; ++k) acc[h][k] *= alpha;
                    pw[h * 32 + lane] = pr;
                }
            }
            __syncwarp();
            // ---- values: lane = output dims
            const int nv = max(0, min(32, seq_b - t0w));
            const uint32_t vt = kt + C::kTileBytes;
            for (int tt = 0; tt < nv; ++tt) {
                const int vr = warp * 32 + tt;
                float vv[C::kDpl];
                if constexpr (D == 128) {
                    // dims 4*lane .. 4*lane+3: box lane/16, 16-byte chunk (lane%16)/2, half lane%2
                    const int chunk = (lane & 15) >> 1;
                    const uint32_t a = vt + (lane >> 4) * kBoxBytes + vr * 128 + ((chunk ^ (vr & 7)) << 4) + ((lane & 1) << 3);
                    const uint2 w2 = lds64(a);
                    vv[0] = bf16lo(w2.x); vv[1] = bf16hi(w2.x); vv[2] = bf16lo(w2.y); vv[3] = bf16hi(w2.y);
                } else {
                    // dims 2*lane, 2*lane+1: chunk lane/4, word lane%4
                    const int chunk = lane >> 2;
                    const uint32_t a = vt + vr * 128 + ((chunk ^ (vr & 7)) << 4) + ((lane & 3) << 2);
                    const uint32_t w1 = lds32(a);
                    vv[0] = bf16lo(w1); vv[1] = bf16hi(w1);
                }
#pragma unroll
                for (int h = 0; h < NMAX; ++h) {
                    if (h < n) {
                        const float pr = pw[h * 32 + tt];
#pragma unroll
                        for (int k = 0; k < C::kDpl; ++k) acc[h][k] = fmaf(pr, vv[k], acc[h][k]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);

            if (last) {
                // ---- merge the 4 warps' states for this piece
#pragma unroll
                for (int h = 0; h < NMAX; ++h) {
                    if (h < n) {
                        float ls = l_lane[h];
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
                        if (lane == 0) {
                            m_s[warp * NMAX + h] = m_run[h];
                            l_s[warp * NMAX + h] = ls;
                        }
#pragma unroll
                        for (int k = 0; k < C::kDpl; ++k) acc_s[(warp * NMAX + h) * D + lane * C::kDpl + k] = acc[h][k];
                    }
                }
                if (!gsync(ab)) break;
                const int seg = cur.b * G + cur.g;
                const long long seg_a = (long long)G * prefix[cur.b] + (long long)cur.g * cur.tiles;
                const bool owned = (piece_u0 == seg_a) && (cur.j + 1 == cur.tiles);
                const int slot = blockIdx.x + seg;
                float *sp = slot_ptr(p, slot, D);
                float *orow = p.out + ((size_t)cur.b * p.H + (size_t)cur.g * n) * D;
                for (int idx = tid; idx < n * D; idx += C::kWarps * 32) {
                    const int h = idx / D, dim = idx - h * D;
                    float M = -INFINITY;
#pragma unroll
                    for (int w = 0; w < C::kWarps; ++w) M = fmaxf(M, m_s[w * NMAX + h]);
                    float L = 0.f, A = 0.f;
#pragma unroll
                    for (int w = 0; w < C::kWarps; ++w) {
                        const float sc = ex2(m_s[w * NMAX + h] - M);   // 0 for a warp with no position
                        L = fmaf(l_s[w * NMAX + h], sc, L);
                        A = fmaf(acc_s[(w * NMAX + h) * D + dim], sc, A);
                    }
                    if (owned) {
                        orow[idx] = A / L;
                    } else {
                        if (dim == 0) {
                            sp[h] = M;
                            sp[n + h] = L;
                        }
                        sp[slot_acc_offset(n) + idx] = A;
                    }
                }
                if (!gsync(ab)) break;   // the merge buffers are reused by the next piece
                ++piece;
            }
            cursor_next(cur, prefix, p.B, G);
        }
    }

    __syncthreads();
    // If the CTA is aborting, let the copies it issued land before exiting.
    if (warp == C::kWarps && lane == 0 && *s_abort) {
        for (int k = max(0, issued - C::kStages); k < issued; ++k)
            mbar_wait_teardown(&full[k % C::kStages], (k / C::kStages) & 1);
    }
}

template <int D, int NMAX>
cudaError_t launch_simt_t(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p, int ctas,
                          cudaStream_t stream) {
    using C = SimtCfg<D, NMAX>;
    auto kern = gqa_decode_simt_kernel<D, NMAX>;
    static unsigned long long attr_set = 0;   // one bit per device; setting twice is harmless
    int dev = 0;
    cudaGetDevice(&dev);
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(attr_set & bit)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set |= bit;
    }
    return launch_pdl(kern, ctas, C::kThreads, C::kSmemBytes, stream, tk, tv, p);
}

}  // namespace

int simt_max_heads() { return 8; }

cudaError_t launch_decode_simt(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p, int D,
                               int ctas, cudaStream_t stream) {
    const int n = p.n;
    if (D == 128) {
        if (n <= 1) return launch_simt_t<128, 1>(tk, tv, p, ctas, stream);
        if (n <= 2) return launch_simt_t<128, 2>(tk, tv, p, ctas, stream);
        if (n <= 4) return launch_simt_t<128, 4>(tk, tv, p, ctas, stream);
        return launch_simt_t<128, 8>(tk, tv, p, ctas, stream);
    }
    if (n <= 1) return launch_simt_t<64, 1>(tk, tv, p, ctas, stream);
    if (n <= 2) return launch_simt_t<64, 2>(tk, tv, p, ctas, stream);
    if (n <= 4) return launch_simt_t<64, 4>(tk, tv, p, ctas, stream);
    return launch_simt_t<64, 8>(tk, tv, p, ctas, stream);
}

}  // namespace gqa
