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

// The same stream with every 32 KiB tile fetched as pages: 128/R pages of R rows.
// Page q of the stream (q = tile * 128/R + k) sits at page slot (q * A) mod
// npages with A odd when `scatter` is set (a permutation of the buffer's pages,
// npages a power of two), else at slot q.  one_box = 0: two boxes per page (64
// columns x R rows each, the layout of a whole tile); one_box = 1: one box per
// page through a five-dimensional map (64 columns, 8 rows, 2 column halves, R/8
// row groups, pages), which lands the page as [row group][half][8 rows][128 B].
// Tile i is issued by warp i % warps; lanes 0..L-1 of that warp issue its
// boxes, lane l taking boxes l, l+L, ...; lane 0 waits for the stage and sets the
// byte count first.  The last warp releases the stages.
__global__ void __launch_bounds__(96, 1)
    stream_boxes_kernel(const __grid_constant__ CUtensorMap tm, long long rows_per_z, long long ntiles, int box_rows,
                        int lanes, int scatter, long long npages, int one_box, int warps, unsigned int *flags) {
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
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nb = kBoxRows / box_rows, boxes = one_box ? nb : 2 * nb;
    int issued = 0;
    if (warp < warps) {
        const uint64_t pol = gqa::l2_policy_evict_first();
        for (int i = warp; i < n; i += warps) {
            const int s = i % kStages;
            bool ok = true;
            if (lane == 0) {
                ok = i < kStages || gqa::mbar_wait(&empty[s], ((i / kStages) - 1) & 1, ab);
                if (ok) gqa::mbar_arrive_expect_tx(&full[s], kTileBytes);
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            if (lane < lanes) {
                for (int b = lane; b < boxes; b += lanes) {
                    const int k = one_box ? b : b >> 1, cb = one_box ? 0 : b & 1;
                    const long long q = (t0 + i) * nb + k;
                    const long long slot = scatter ? (long long)(((unsigned long long)q * 0x9E3779B1ull) &
                                                                 (unsigned long long)(npages - 1))
                                                   : q;
                    if (one_box) {
                        gqa::tma_load_5d(smem + s * kTileBytes + k * box_rows * 256, &tm, 0, 0, 0, 0, (int)slot,
                                         &full[s], pol);
                    } else {
                        const long long row = slot * box_rows;
                        const int z = (int)(row / rows_per_z), y = (int)(row - (long long)z * rows_per_z);
                        gqa::tma_load_3d(smem + s * kTileBytes + cb * kBoxBytes + k * box_rows * 128, &tm,
                                         cb * kBoxCols, y, z, &full[s], pol);
                    }
                }
            }
            __syncwarp();
            ++issued;
        }
    } else if (warp == warps && lane == 0) {
        for (int i = 0; i < n; ++i) {
            const int s = i % kStages;
            if (!gqa::mbar_wait(&full[s], (i / kStages) & 1, ab)) break;
            gqa::mbar_arrive(&empty[s]);
        }
    }
    __syncthreads();
    if (warp < warps && lane == 0 && s_abort) {
        for (int k = issued > kStages / warps ? issued - kStages / warps : 0; k < issued; ++k) {
            const int i = warp + k * warps;
            gqa::mbar_wait_teardown(&full[i % kStages], (i / kStages) & 1);
        }
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

}  // namespace

// Prepares a tensor map over bf16 [z, rows, 128] with boxes of 64 columns x box_rows;
// returns 0 or the entry point's error code.
static int encode_map(CUtensorMap *tm, const void *buf, long long z, long long rows, int box_rows, int *sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
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
    const cuuint64_t dims[3] = {128, (cuuint64_t)rows, (cuuint64_t)z};
    const cuuint64_t strides[2] = {256, (cuuint64_t)rows * 256};
    const cuuint32_t box[3] = {(cuuint32_t)kBoxCols, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (reinterpret_cast<EncodeTiledFn>(fn)(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(buf), dims,
                                            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return 4;
    return 0;
}

extern "C" int gqa_bench_stream_read(const void *buf, long long z, long long rows, int ctas, unsigned int *flags,
                                     void *stream) {
    if (!buf || !flags || z <= 0 || rows <= 0 || rows % kBoxRows != 0 || ctas < 0 ||
        reinterpret_cast<uintptr_t>(buf) % 16 != 0 || z > (1ll << 31) || rows > (1ll << 31))
        return 1;
    CUtensorMap tm;
    int sms = 0;
    if (const int e = encode_map(&tm, buf, z, rows, kBoxRows, &sms)) return e;
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

// Prepares the five-dimensional page map over bf16 [npages, page_rows, 128]: (64
// columns, 8 rows, 2 column halves, page_rows / 8 row groups, pages), one box a page.
static int encode_page_map(CUtensorMap *tm, const void *buf, long long npages, int page_rows) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
        cudaGetLastError();
        return 5;
    }
    const cuuint64_t dims[5] = {64, 8, 2, (cuuint64_t)(page_rows / 8), (cuuint64_t)npages};
    const cuuint64_t strides[4] = {256, 128, 2048, (cuuint64_t)page_rows * 256};
    const cuuint32_t box[5] = {64, 8, 2, (cuuint32_t)(page_rows / 8), 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    if (reinterpret_cast<EncodeTiledFn>(fn)(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(buf), dims,
                                            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return 6;
    return 0;
}

extern "C" int gqa_bench_stream_read_pages(const void *buf, long long z, long long rows, int page_rows, int lanes,
                                           int scatter, int one_box, int warps, int ctas, unsigned int *flags,
                                           void *stream) {
    const long long total = z * rows;
    const long long npages = page_rows > 0 ? total / page_rows : 0;
    if (!buf || !flags || z <= 0 || rows <= 0 || rows % kBoxRows != 0 || ctas < 0 ||
        reinterpret_cast<uintptr_t>(buf) % 16 != 0 || z > (1ll << 31) || rows > (1ll << 31) ||
        (page_rows != 16 && page_rows != 32 && page_rows != 64 && page_rows != 128) || lanes < 1 || lanes > 32 ||
        (scatter && (npages & (npages - 1)) != 0) || warps < 1 || warps > 2 || npages > (1ll << 31))
        return 1;
    CUtensorMap tm;
    int sms = 0;
    if (const int e = encode_map(&tm, buf, z, rows, page_rows, &sms)) return e;
    if (one_box)
        if (const int e = encode_page_map(&tm, buf, npages, page_rows)) return e;
    if (cudaFuncSetAttribute(stream_boxes_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
        cudaSuccess) {
        cudaGetLastError();
        return 4;
    }
    const long long ntiles = total / kBoxRows;
    const int grid = (int)(ntiles < (ctas ? ctas : sms) ? ntiles : (ctas ? ctas : sms));
    stream_boxes_kernel<<<grid, 32 * warps + 32, kSmemBytes, static_cast<cudaStream_t>(stream)>>>(
        tm, rows, ntiles, page_rows, lanes, scatter ? 1 : 0, npages, one_box ? 1 : 0, warps, flags);
    if (cudaGetLastError() != cudaSuccess) return 4;
    return 0;
}
