// Split-combine: merges the partial softmax states of the segments that the
// decode kernel's work split cut across CTAs, and writes their output rows.
//
// For segment (b, g), cut into pieces k = 0 .. K-1 with states (m_k, l_k, acc_k)
// per query head h (m in base-2 units):
//   M_h = max_k m_kh,   L_h = sum_k l_kh 2^(m_kh - M_h),
//   out[b, g*n + h, :] = (sum_k acc_kh 2^(m_kh - M_h)) / L_h.
// This is the exact rescaling that joins softmax sums over disjoint sets of
// positions; the pages' decode step has no split (every query head attends
// over its whole cache), so the merge only reassembles that sum.
// ["Grouped-query attention (GQA)" concept page, "Implementation sketch",
//  decode-step pseudocode; arxiv:2305.13245 §2.2]
//
// Launched right after the decode kernel with programmatic stream
// serialisation: its CTAs build the tile prefix and the work split (from
// seq_lens, which the decode kernel does not write) while the decode grid
// drains, then wait for it to complete.  Their shared memory is sized to the
// batch (the prefix of B sequences), so that a split-combine block fits on an
// SM beside a decode block: beside the decode kernel it serves, and beside the
// next decode kernel, which it lets start its on-chip set-up at once.  The CTAs take (segment, 256-float4
// part of its n x D outputs) work items in a grid-stride loop, so large head
// groups spread over several CTAs; a segment whose single piece covered it whole
// was written by the decode kernel, the others are merged here from the slots
// the work split assigns to their pieces.  A thread owns four consecutive dims
// of one head and loads the pieces in batches of eight, each batch one round
// trip to L2, merging online.
#include <cuda_runtime.h>

#include "decode_common.cuh"
#include "launch.h"

namespace gqa {

namespace {

constexpr int kCombThreads = 256;
constexpr int kBatch = 8;   // pieces per round trip

// Dynamic shared memory: prefix[B + 1], scratch[33].
__host__ __device__ constexpr size_t combine_smem_bytes(int B) { return (size_t)(B + 1 + 33) * sizeof(int); }

template <int D>
__global__ void __launch_bounds__(kCombThreads) gqa_split_combine_kernel(const DecodeParams p, int grid_main) {
    extern __shared__ int cmb_smem[];
    int *prefix = cmb_smem, *scratch = cmb_smem + p.B + 1;
    // The next grid on the stream (normally the next decode step) may start its
    // on-chip set-up as SMs have room; it touches memory only once this one is done.
    griddep_launch_dependents();
    build_prefix(p, p.tile_shift, prefix, scratch, nullptr);   // ends with __syncthreads
    const int G = p.G, n = p.n;
    const WorkSplit split = make_split((long long)G * prefix[p.B], grid_main,
                                       pool_tail_tiles(prefix, p.B, G, scratch[32]), p.dyn_cap);
    griddep_wait();   // the decode grid has completed: its partials are visible

    const size_t stride = (size_t)slot_floats(n, D);
    const int aoff = slot_acc_offset(n);
    const int nd4 = n * D / 4;
    const int parts = (nd4 + kCombThreads - 1) / kCombThreads;   // CTAs per segment (one float4 per thread each)
    for (int wi = blockIdx.x; wi < p.B * G * parts; wi += gridDim.x) {
        const int s = wi / parts, e = (wi - s * parts) * kCombThreads + threadIdx.x;
        const int b = s / G, g = s - b * G;
        const int T = prefix[b + 1] - prefix[b];
        if (T == 0) continue;
        const long long a = (long long)G * prefix[b] + (long long)g * T;
        const SegmentSlots sl = segment_slots(p, split, prefix, s, a, T);
        const int count = sl.count();
        if (count < 2) continue;   // one piece covered the segment: the decode kernel wrote it
        float4 *orow = reinterpret_cast<float4 *>(p.out + ((size_t)b * p.H + (size_t)g * n) * D);
        if (e < nd4) {
            const int h = (e * 4) / D;
            float M = -INFINITY, L = 0.f;
            float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int k0 = 0; k0 < count; k0 += kBatch) {
                float mk[kBatch], lk[kBatch];
                float4 vk[kBatch];
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    if (k0 + j < count) {
                        const float *sk = p.partials + (size_t)sl(k0 + j) * stride;
                        mk[j] = __ldcg(sk + h);
                        lk[j] = __ldcg(sk + n + h);
                        vk[j] = __ldcg(reinterpret_cast<const float4 *>(sk + aoff) + e);
                    } else {
                        mk[j] = -INFINITY;
                        lk[j] = 0.f;
                        vk[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                float Mb = M;
#pragma unroll
                for (int j = 0; j < kBatch; ++j) Mb = fmaxf(Mb, mk[j]);   // finite: every piece has a position
                const float sc = ex2(M - Mb);                              // 0 on the first batch
                L *= sc;
                A.x *= sc;
                A.y *= sc;
                A.z *= sc;
                A.w *= sc;
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    const float w = ex2(mk[j] - Mb);                       // 0 for the padding entries
                    L = fmaf(lk[j], w, L);
                    A.x = fmaf(vk[j].x, w, A.x);
                    A.y = fmaf(vk[j].y, w, A.y);
                    A.z = fmaf(vk[j].z, w, A.z);
                    A.w = fmaf(vk[j].w, w, A.w);
                }
                M = Mb;
            }
            orow[e] = make_float4(A.x / L, A.y / L, A.z / L, A.w / L);
        }
    }
}

}  // namespace

cudaError_t launch_split_combine(const DecodeParams &p, int D, int grid_main, cudaStream_t stream) {
    // one CTA per segment and 256 float4 of its n x D outputs, at most 4096 (the others
    // loop over the rest): large head groups spread over several CTAs
    const int nd4 = p.n * D / 4;
    const long long work = (long long)p.B * p.G * ((nd4 + kCombThreads - 1) / kCombThreads);
    const int grid = work < 4 * kMaxCtas ? (int)work : 4 * kMaxCtas;
    const size_t smem = combine_smem_bytes(p.B);
    if (D == 128) return launch_pdl(gqa_split_combine_kernel<128>, grid, kCombThreads, smem, stream, p, grid_main);
    return launch_pdl(gqa_split_combine_kernel<64>, grid, kCombThreads, smem, stream, p, grid_main);
}

}  // namespace gqa
