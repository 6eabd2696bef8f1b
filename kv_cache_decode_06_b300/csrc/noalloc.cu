// gqa_decode_noalloc: the decode step for callers that cannot allocate device
// memory.
//
// gqa_decode needs a caller-provided workspace (split-combine partials, the
// dynamic work pool's counters, a flag word).  Some callers have no way to provide one: a plugin
// that only receives the tensors it works on from a host framework that owns
// all device memory, a runtime that reserves its memory once at start-up and
// forbids allocation afterwards, or a latency-critical loop that cannot afford
// cudaMalloc's implicit device synchronisation.  This entry point uses a
// fixed-size scratch array that lives in the library itself instead.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds GQA_NOALLOC_WORKSPACE_BYTES of it until the process exits.  In
// host code its name is only a host-side stand-in, so the device address is
// looked up with cudaGetSymbolAddress, once per device, with that device
// current, and passed to the kernel like any workspace.  The address is kept
// for the life of the process: after a cudaDeviceReset it would be stale, so
// the library must not be used across one.  Nothing here calls cudaMalloc,
// cudaFree or an allocating library routine.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "gqa.h"
#include "launch.h"

namespace {

constexpr size_t kScratchBytes = GQA_NOALLOC_WORKSPACE_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

// Device address of g_noalloc_scratch on the current device (set up on the
// first call per device).
gqa_status scratch_address(void **out) {
    static std::mutex mu;
    static void *addr[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GQA_ERR_DEVICE;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return GQA_ERR_DEVICE;
        }
        addr[dev] = p;
    }
    *out = addr[dev];
    return GQA_OK;
}

}  // namespace

extern "C" gqa_status gqa_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                         const int32_t *seq_lens, float *out, int B, int H, int G, int d, int Lmax,
                                         float scale, void *stream) {
    if (!q || !k_cache || !v_cache || !out) return GQA_ERR_INVALID_ARG;
    size_t need = 0;
    const gqa_status s = gqa_decode_workspace_size(B, H, G, d, Lmax, &need);
    if (s != GQA_OK) return s;
    if (need > kScratchBytes) return GQA_ERR_WORKSPACE;   // this shape needs more scratch than the library holds
    // Every host-side check of gqa_decode (pointer alignment, scale, path and
    // head limits, device) runs before anything is enqueued: a rejected call
    // leaves the stream, and the scratch that a call on another stream may be
    // using, untouched.  The scratch itself (256-byte aligned, kScratchBytes
    // long, checked against `need` above) is not a caller's workspace to check.
    const gqa_status c = gqa::decode_check(q, k_cache, v_cache, seq_lens, out, nullptr, kScratchBytes, B, H, G, d,
                                           Lmax, scale);
    if (c != GQA_OK) return c;
    void *ws = nullptr;
    const gqa_status a = scratch_address(&ws);
    if (a != GQA_OK) return a;
    // Clear the scratch's whole header every time, on the caller's stream: the
    // flag word, so that a flag left by an earlier call does not stay set, and
    // the dynamic-pool ticket and failed-claim count.  A call that ran into a
    // wait limit (GQA_FLAG_WAIT_TIMEOUT) leaves those two counters wherever its
    // aborted thread blocks stopped, and clearing them here is what lets the next
    // call run exactly without any reset by the caller.
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, gqa::decode_workspace_zero_prefix(B, G), st) != cudaSuccess) {
        cudaGetLastError();
        return GQA_ERR_LAUNCH;
    }
    return gqa_decode(q, k_cache, v_cache, seq_lens, out, ws, kScratchBytes, B, H, G, d, Lmax, scale, stream);
}
