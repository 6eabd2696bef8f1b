// Mean-pool conversion of K/V projection heads into G groups.
// ["Grouped-query attention (GQA)" concept page, "Converted and uptrained
//  checkpoints" and the conversion pseudocode; arxiv:2305.13245 §2.1]
//
// w_out[o, g, x] = ((w_in[o, g*n, x] + w_in[o, g*n+1, x]) + ... ) / n, every
// addition and the division rounded in fp32 in that order, so the result is
// bit-identical to that sequence.  One pass over HBM: each input element is
// read once, each output element written once, 16-byte accesses when the
// layout allows.
#include <cuda_runtime.h>

#include "launch.h"

namespace gqa {

namespace {

__global__ void meanpool_vec4_kernel(const float4 *__restrict__ w, float4 *__restrict__ out, long long outer,
                                     int H, int G, long long inner4) {
    const int n = H / G;
    const float fn = (float)n;
    const long long total = outer * G * inner4;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const long long x = e % inner4;
        const long long og = e / inner4;
        const int g = (int)(og % G);
        const long long o = og / G;
        const float4 *src = w + ((o * H + (long long)g * n) * inner4 + x);
        float4 acc = __ldg(src);
        for (int j = 1; j < n; ++j) {
            const float4 y = __ldg(src + (long long)j * inner4);
            acc.x = __fadd_rn(acc.x, y.x);
            acc.y = __fadd_rn(acc.y, y.y);
            acc.z = __fadd_rn(acc.z, y.z);
            acc.w = __fadd_rn(acc.w, y.w);
        }
        acc.x = __fdiv_rn(acc.x, fn);
        acc.y = __fdiv_rn(acc.y, fn);
        acc.z = __fdiv_rn(acc.z, fn);
        acc.w = __fdiv_rn(acc.w, fn);
        out[e] = acc;
    }
}

__global__ void meanpool_scalar_kernel(const float *__restrict__ w, float *__restrict__ out, long long outer,
                                       int H, int G, long long inner) {
    const int n = H / G;
    const float fn = (float)n;
    const long long total = outer * G * inner;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const long long x = e % inner;
        const long long og = e / inner;
        const int g = (int)(og % G);
        const long long o = og / G;
        const float *src = w + ((o * H + (long long)g * n) * inner + x);
        float acc = __ldg(src);
        for (int j = 1; j < n; ++j) acc = __fadd_rn(acc, __ldg(src + (long long)j * inner));
        out[e] = __fdiv_rn(acc, fn);
    }
}

}  // namespace

cudaError_t launch_meanpool(const float *w_in, float *w_out, long long outer, int H, int G, long long inner,
                            cudaStream_t stream) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const bool vec = (inner % 4 == 0) && ((reinterpret_cast<uintptr_t>(w_in) | reinterpret_cast<uintptr_t>(w_out)) % 16 == 0);
    const long long total = outer * G * (vec ? inner / 4 : inner);
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    long long blocks = (total + threads - 1) / threads;
    const long long cap = (long long)sms * 8;
    if (blocks > cap) blocks = cap;
    if (vec)
        meanpool_vec4_kernel<<<(int)blocks, threads, 0, stream>>>(reinterpret_cast<const float4 *>(w_in),
                                                                  reinterpret_cast<float4 *>(w_out), outer, H, G,
                                                                  inner / 4);
    else
        meanpool_scalar_kernel<<<(int)blocks, threads, 0, stream>>>(w_in, w_out, outer, H, G, inner);
    return cudaGetLastError();
}

}  // namespace gqa
