// Mean-pool conversion of K/V projection heads into G groups.
// ["Grouped-query attention (GQA)" concept page, "Converted and uptrained
//  checkpoints" and the conversion pseudocode; arxiv:2305.13245 §2.1]
//
// w_out[o, g, x] = ((w_in[o, g*n, x] + w_in[o, g*n+1, x]) + ... ) / n, every
// addition and the division rounded in fp32 in that order, so the result is
// bit-identical to that sequence.  One pass over HBM: each input element is
// read once, each output element written once, 16-byte accesses when the
// layout allows; each thread keeps up to 8 loads in flight.
#include <cuda_runtime.h>

#include "launch.h"

namespace gqa {

namespace {

// Loads in flight per thread: the n terms of one output are fetched in batches
// of kBatch independent loads, then added in head order.
constexpr int kBatch = 8;

__device__ __forceinline__ float4 add4_rn(float4 a, float4 b) {
    return make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z), __fadd_rn(a.w, b.w));
}

// T is float4 (16-byte accesses) or float.  The first term is assigned, not
// added to zero, so a -0.0 input keeps its sign as in the plain sequence.
template <typename T>
__device__ __forceinline__ T fold_heads(const T *__restrict__ src, long long stride, int n) {
    T acc{};
    for (int j0 = 0; j0 < n; j0 += kBatch) {
        T y[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
            if (j0 + u < n) y[u] = __ldg(src + (long long)(j0 + u) * stride);
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            if (j0 + u >= n) break;
            if constexpr (sizeof(T) == 16)
                acc = (j0 + u == 0) ? y[u] : add4_rn(acc, y[u]);
            else
                acc = (j0 + u == 0) ? y[u] : __fadd_rn(acc, y[u]);
        }
    }
    return acc;
}

// Each block converts one contiguous span of the outputs, blockDim.x at a time;
// a thread's place (o, g, x) advances by additions only (no division in the loop).
template <typename T>
__global__ void __launch_bounds__(256, 4) meanpool_kernel(const T *__restrict__ w, T *__restrict__ out,
                                                       long long outer, int H, int G, long long inner) {
    const int n = H / G;
    const float fn = (float)n;
    const long long total = outer * G * inner;
    const long long per = (total + gridDim.x - 1) / gridDim.x;
    const long long begin = blockIdx.x * per;
    const long long end = begin + per < total ? begin + per : total;
    long long e = begin + threadIdx.x;
    if (e >= end) return;
    long long og = e / inner, x = e - og * inner;
    int g = (int)(og % G);
    long long o = og / G;
    const int step = blockDim.x;
    for (; e < end; e += step) {
        T acc = fold_heads(w + ((o * H + (long long)g * n) * inner + x), inner, n);
        if constexpr (sizeof(T) == 16)
            acc = make_float4(__fdiv_rn(acc.x, fn), __fdiv_rn(acc.y, fn), __fdiv_rn(acc.z, fn),
                              __fdiv_rn(acc.w, fn));
        else
            acc = __fdiv_rn(acc, fn);
        out[e] = acc;
        x += step;
        while (x >= inner) {
            x -= inner;
            if (++g == G) {
                g = 0;
                ++o;
            }
        }
    }
}

template <typename T>
cudaError_t launch_typed(const T *w_in, T *w_out, long long outer, int H, int G, long long inner,
                         cudaStream_t stream) {
    const long long total = outer * G * inner;
    if (total == 0) return cudaSuccess;
    constexpr int threads = 256;
    int dev = 0, sms = 148, per_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, meanpool_kernel<T>, threads, 0) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    // one resident wave: every SM holds the same number of blocks
    long long blocks = (total + threads - 1) / threads;
    const long long cap = (long long)sms * per_sm;
    if (blocks > cap) blocks = cap;
    meanpool_kernel<T><<<(int)blocks, threads, 0, stream>>>(w_in, w_out, outer, H, G, inner);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_meanpool(const float *w_in, float *w_out, long long outer, int H, int G, long long inner,
                            cudaStream_t stream) {
    const bool vec = (inner % 4 == 0) && ((reinterpret_cast<uintptr_t>(w_in) | reinterpret_cast<uintptr_t>(w_out)) % 16 == 0);
    if (vec)
        return launch_typed(reinterpret_cast<const float4 *>(w_in), reinterpret_cast<float4 *>(w_out), outer, H, G,
                            inner / 4, stream);
    return launch_typed(w_in, w_out, outer, H, G, inner, stream);
}

}  // namespace gqa
