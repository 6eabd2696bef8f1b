// GQA decode on the fifth-generation tensor cores (tcgen05 + TMEM).
#include <cuda.h>
#include <cuda_runtime.h>

#include "launch.h"

namespace gqa {

int tc_max_heads() { return 0; }

cudaError_t launch_decode_tc(const CUtensorMap &, const CUtensorMap &, const CUtensorMap &, const DecodeParams &,
                             int, int, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace gqa
