// Internal interface between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "decode_common.cuh"

namespace gqa {

int simt_max_heads();
cudaError_t launch_decode_simt(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p, int D,
                               int ctas, cudaStream_t stream);

int tc_max_heads();
int tc_rows_for(int n);   // rows of the q tensor-map box (n rounded up to 16, 32 or 64)
cudaError_t launch_decode_tc(const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tq,
                             const DecodeParams &p, int D, int ctas, cudaStream_t stream);

// Leading bytes of a decode workspace that must be zero before a call on a
// fresh (or differently shaped) workspace: the flag word and the counters.
size_t decode_workspace_zero_prefix(int B, int G);

cudaError_t launch_meanpool(const float *w_in, float *w_out, long long outer, int H, int G, long long inner,
                            cudaStream_t stream);

}  // namespace gqa
