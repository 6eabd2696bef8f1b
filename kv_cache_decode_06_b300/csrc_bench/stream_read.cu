// Read-only stream with the decode kernel's TMA access pattern (see gqa_bench.h):
// the read-bandwidth ceiling the decode kernel is measured against.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gqa_bench.h"
#include "ptx.cuh"

namespace {

constexpr int kBoxCols = 64;                        // bf16 per 128-byte swizzled row
constexpr int kBoxRows = 128;
constexpr int kBoxBytes = kBoxCols * 2 * kBoxRows;  // 16 KiB
constexpr int kTileBytes = 2 * kBoxBytes;           // a K or V tile of the decode at d = 128
constexpr int kStages = 6;
constexpr int kSmemBytes = kStages * kTileBytes + 2 * kStages * 8 + 1024;

// One thread issues the tile copies of this block's range into the ring, one
// thread releases each stage once it has landed.
__global__ void __launch_bounds__(64, 1)
    stream_read_kernel(const __grid_constant__ CUtensorMap tm, long long tiles_per_z, long long ntiles,
                       unsigned int *flags) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * kTileBytes), *empty = full + kStages;
    __shared__ volatile int s_abort;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            gqa::mbar_init(&full[s], 1);
            gqa::mbar_init(&empty[s], 1);
        }
        s_abort = 0;
        gqa::fence_mbar_init();
        gqa::tma_prefetch_desc(&tm);
    }
    __syncthreads();
    const gqa::AbortState ab{&s_abort, flags};
    const long long P = gridDim.x, c = blockIdx.x;
    const long long t0 = c * ntiles / P, t1 = (c + 1) * ntiles / P;
    const int n = (int)(t1 - t0);
    int issued = 0;
    if (threadIdx.x == 0) {
        const uint64_t pol = gqa::l2_policy_evict_first();
        for (int i = 0; i < n; ++i) {
            const int s = i % kStages;
            if (i >= kStages && !gqa::mbar_wait(&empty[s], ((i / kStages) - 1) & 1, ab)) break;
            const long long t = t0 + i;
            const int z = (int)(t / tiles_per_z), j = (int)(t - (long long)z * tiles_per_z);
            gqa::mbar_arrive_expect_tx(&full[s], kTileBytes);
#pragma unroll
            for (int cb = 0; cb < 2; ++cb)
                gqa::tma_load_3d(smem + s * kTileBytes + cb * kBoxBytes, &tm, cb * kBoxCols, j * kBoxRows, z, &full[s],
                                 pol);
            ++issued;
        }
    } else if (threadIdx.x == 32) {
        for (int i = 0; i < n; ++i) {
            const int s = i % kStages;
            if (!gqa::mbar_wait(&full[s], (i / kStages) & 1, ab)) break;
            gqa::mbar_arrive(&empty[s]);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && s_abort) {
        // let copies in flight land before the block's shared memory is released
        for (int k = issued > kStages ? issued - kStages : 0; k < issued; ++k)
            gqa::mbar_wait_teardown(&full[k % kStages], (k / kStages) & 1);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

}  // namespace

extern "C" int gqa_bench_stream_read(const void *buf, long long z, long long rows, int ctas, unsigned int *flags,
                                     void *stream) {
    if (!buf || !flags || z <= 0 || rows <= 0 || rows % kBoxRows != 0 || ctas < 0 ||
        reinterpret_cast<uintptr_t>(buf) % 16 != 0 || z > (1ll << 31) || rows > (1ll << 31))
        return 1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 5;
    }
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
        cudaGetLastError();
        return 5;
    }
    CUtensorMap tm;
    const cuuint64_t dims[3] = {128, (cuuint64_t)rows, (cuuint64_t)z};
    const cuuint64_t strides[2] = {256, (cuuint64_t)rows * 256};
    const cuuint32_t box[3] = {(cuuint32_t)kBoxCols, (cuuint32_t)kBoxRows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (reinterpret_cast<EncodeTiledFn>(fn)(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(buf), dims,
                                            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return 4;
    if (cudaFuncSetAttribute(stream_read_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
        cudaSuccess) {
        cudaGetLastError();
        return 4;
    }
    const long long tiles_per_z = rows / kBoxRows, ntiles = tiles_per_z * z;
    const int grid = (int)(ntiles < (ctas ? ctas : sms) ? ntiles : (ctas ? ctas : sms));
    stream_read_kernel<<<grid, 64, kSmemBytes, static_cast<cudaStream_t>(stream)>>>(tm, tiles_per_z, ntiles, flags);
    if (cudaGetLastError() != cudaSuccess) return 4;
    return 0;
}
