// Internal interface between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <utility>

#include "decode_common.cuh"
#include "gqa.h"

namespace gqa {

// Launch with programmatic stream serialisation: the kernel may start while the
// previous kernel on the stream drains; it waits for it (griddepcontrol.wait)
// before touching global memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), int grid, int block, size_t smem, cudaStream_t stream,
                              Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

int simt_max_heads();
cudaError_t launch_decode_simt(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p, int D,
                               int ctas, cudaStream_t stream);

// The contiguous cache's tensor maps again, with boxes of 64, 32 and 16 rows:
// the last tile of a segment is loaded only as far as its attended rows reach
// (rounded up to 16 rows).  Unused (zero) for a paged cache.
struct TailMaps {
    CUtensorMap k[3];
    CUtensorMap v[3];
};

int tc_max_heads();
int tc_rows_for(int n);   // rows of the q tensor-map box (n rounded up to 16, 32 or 64)
// Whether the tensor-core kernel reads this shape's cache in the paired layout
// (D = 64: rows of two positions, 256-position tiles, tile_shift 8).
bool tc_paired(int D, int Lmax, int n);
cudaError_t launch_decode_tc(const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tq,
                             const TailMaps &tails, const DecodeParams &p, int D, bool paired, int ctas,
                             cudaStream_t stream);

// Leading bytes of a decode workspace that must be zero before its first call:
// GQA_WORKSPACE_HEADER_BYTES (flag word, dynamic-pool ticket, failed-claim
// count), the same for every shape.
size_t decode_workspace_zero_prefix(int B, int G);

// Every host-side check gqa_decode makes (arguments, workspace, path, device),
// without enqueueing anything: the status gqa_decode would return before its
// first launch.  workspace null: the checks of the workspace are skipped (a
// scratch the library owns, whose size and alignment its owner checks).
gqa_status decode_check(const void *q, const void *k_cache, const void *v_cache, const int32_t *seq_lens,
                        float *out, void *workspace, size_t workspace_bytes, int B, int H, int G, int d, int Lmax,
                        float scale);

// The split-combine kernel (combine.cu), launched after a decode kernel of
// grid_main CTAs.
cudaError_t launch_split_combine(const DecodeParams &p, int D, int grid_main, cudaStream_t stream);

cudaError_t launch_meanpool(const float *w_in, float *w_out, long long outer, int H, int G, long long inner,
                            cudaStream_t stream);

}  // namespace gqa
