// The C ABI: argument checks, tensor maps, path choice and launches.
// Declarations and the contract of every entry point are in include/gqa.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>

#include "gqa.h"
#include "launch.h"

namespace {

using gqa::DecodeParams;
static_assert(gqa::kMaxCtas == GQA_MAX_CTAS, "CTA limit mismatch");

constexpr int kMaxHeadsPerGroup = 64;
constexpr int kMaxHeads = 4096;
constexpr long long kMaxLmax = 1ll << 24;
constexpr long long kMaxTiles = 1ll << 30;   // B * G * ceil(Lmax / 128), far above any cache that fits

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

struct DeviceInfo {
    int sms = 0;
    bool ok = false;
};

// Per-device facts, looked up once per device.
gqa_status device_info(DeviceInfo *out) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    static bool seen[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return GQA_ERR_DEVICE;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!seen[dev]) {
        DeviceInfo d;
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
            d.ok = (major == 10 && minor == 3);
        cudaGetLastError();
        cache[dev] = d;
        seen[dev] = true;
    }
    *out = cache[dev];
    return out->ok ? GQA_OK : GQA_ERR_DEVICE;
}


constexpr size_t kHeaderBytes = 256;

constexpr long long kMaxDynTiles = 8192;   // dynamic-pool tiles the workspace holds slots for, at most

// Dynamic-pool capacity (tiles) for a shape: a quarter of the most 128-position
// tiles it can have, at most kMaxDynTiles, a whole number of chunks.
int dyn_cap_for(int B, int G, int Lmax) {
    const long long w_max = (long long)B * G * ((Lmax + gqa::kTile - 1) / gqa::kTile);
    long long cap = (w_max + 3) / 4;
    if (cap > kMaxDynTiles) cap = kMaxDynTiles;
    return (int)(cap - cap % gqa::kChunk);
}

static_assert(GQA_WORKSPACE_HEADER_BYTES == kHeaderBytes, "header size mismatch");

// Bytes that must be zero before a call: the header (flag word, dynamic-pool
// ticket, failed-claim count), the same for every shape.
size_t zero_prefix_bytes(int B, int G) {
    (void)B;
    (void)G;
    return kHeaderBytes;
}

// Workspace: the zeroed prefix, then the partial slots: one per static piece
// (slot c + s < GQA_MAX_CTAS + B*G), then one per dynamic-pool tile.
size_t workspace_bytes_for(int B, int H, int G, int d, int Lmax) {
    const int n = H / G;
    const size_t slots = (size_t)GQA_MAX_CTAS + (size_t)B * G + (size_t)dyn_cap_for(B, G, Lmax);
    return zero_prefix_bytes(B, G) + slots * (size_t)gqa::slot_floats(n, d) * sizeof(float);
}

gqa_status check_shape(int B, int H, int G, int d, int Lmax) {
    if (B <= 0 || H <= 0 || G <= 0 || d <= 0 || Lmax <= 0) return GQA_ERR_INVALID_ARG;
    if (G > H || H % G != 0) return GQA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return GQA_ERR_UNSUPPORTED;
    if (B > GQA_MAX_BATCH || H > kMaxHeads || H / G > kMaxHeadsPerGroup || Lmax > kMaxLmax)
        return GQA_ERR_UNSUPPORTED;
    // the kernels index 128-position tiles of all K/V heads with 32-bit arithmetic
    if ((long long)B * G * ((Lmax + gqa::kTile - 1) / gqa::kTile) > kMaxTiles) return GQA_ERR_UNSUPPORTED;
    return GQA_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Cache viewed as a 3-D tensor [B*G][Lmax][d] of bf16, loaded in boxes of
// 64 columns (128 bytes, 128-byte swizzle) x 128 positions x 1.  Positions past
// Lmax read as zero.  Paired (d = 64, Lmax even): viewed as [B*G][Lmax/2][128],
// rows of two consecutive positions, so a box of 128 rows and 64 columns holds
// the even (column 0) or the odd (column 64) positions of 256.
// box_rows: 128 (a whole tile), or 64, 32, 16 for the tail maps (the last tile
// of a segment, loaded only as far as its attended rows reach).
bool make_cache_map(CUtensorMap *map, const void *base, int B, int G, int d, int Lmax, bool paired,
                    int box_rows = gqa::kTile) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const int cols = paired ? 2 * d : d, rows = paired ? Lmax / 2 : Lmax;
    const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)B * G};
    const cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)Lmax * d * 2};
    const cuuint32_t box[3] = {(cuuint32_t)gqa::kBoxCols, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q viewed as [B*H][d] bf16, boxes of 64 columns x `rows` rows (128-byte swizzle).
bool make_q_map(CUtensorMap *map, const void *base, int B, int H, int d, int rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)B * H};
    const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
    const cuuint32_t box[2] = {(cuuint32_t)gqa::kBoxCols, (cuuint32_t)rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tensor-core path is faster at every group size measured (H/G = 1 .. 64):
// the CUDA-core path is issue-latency bound even at H/G = 1.  It stays as the
// fallback for shapes the tensor-core path does not take.
int auto_path(int H, int G, int d) {
    (void)d;
    const int n = H / G;
    if (n <= gqa::tc_max_heads()) return GQA_PATH_TCGEN05;
    return GQA_PATH_SIMT;
}

// Paged-cache limits: a page holds at least one 8-row swizzle atom of
// position pairs, and the pool's K/V rows fit the tensor map's 32-bit extent.
constexpr int kMinPage = 16;
constexpr int kMaxPage = 1 << 20;
constexpr long long kMaxPoolRows = 1ll << 31;

// Page pool viewed as [num_pages*G][rows][cols] with rows = page_size, cols = d
// (paired: rows = page_size/2, cols = 2d), 128-byte swizzle, one box = one page
// (or the 128 rows of a tile, for pages longer than a tile).
// cols = 128 (d = 128, or the paired layout): a five-dimensional view (64
// columns, 8 rows, 2 column halves, rows/8 row groups, pages) whose box lands
// the page in shared memory as [row group][half][8 rows][128 B], the layout the
// paged kernel instances read.  Its strides are not increasing (the halves are
// 128 bytes apart, the rows 256): the view only reorders the page's bytes.
// cols = 64: [pages][rows][64] with boxes of 64 columns x min(rows, 128) rows.
bool make_page_map(CUtensorMap *map, const void *base, int num_pages, int G, int d, int page_size, bool paired) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const int cols = paired ? 2 * d : d, rows = paired ? page_size / 2 : page_size;
    const int box_rows = rows < gqa::kTile ? rows : gqa::kTile;
    if (cols == 2 * gqa::kBoxCols) {
        const cuuint64_t dims[5] = {(cuuint64_t)gqa::kBoxCols, 8, 2, (cuuint64_t)rows / 8, (cuuint64_t)num_pages * G};
        const cuuint64_t strides[4] = {(cuuint64_t)cols * 2, (cuuint64_t)gqa::kBoxCols * 2, (cuuint64_t)cols * 2 * 8,
                                       (cuuint64_t)page_size * d * 2};
        const cuuint32_t box[5] = {(cuuint32_t)gqa::kBoxCols, 8, 2, (cuuint32_t)box_rows / 8, 1};
        const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
        return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)num_pages * G};
    const cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)page_size * d * 2};
    const cuuint32_t box[3] = {(cuuint32_t)gqa::kBoxCols, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

#ifdef GQA_TEST_HOOKS
// Test hook (gqa_debug_withhold_copy, test-hooks build only): applies to the
// next decode call only.
std::atomic<int> g_withhold_k{-1};
#endif

// Every decode variant: contiguous or paged cache, with or without the fused
// append, a window, or all positions valid (seq_lens null).
struct DecodeRequest {
    const void *q = nullptr, *k = nullptr, *v = nullptr;   // k, v: cache or page pool
    const void *k_new = nullptr, *v_new = nullptr;         // fused append rows [B, G, d]
    const int32_t *block_table = nullptr;
    int page_size = 0, max_pages = 0, num_pages = 0;
    const int32_t *seq_lens = nullptr;
    float *out = nullptr;
    void *ws = nullptr;
    size_t ws_bytes = 0;
    int B = 0, H = 0, G = 0, d = 0, Lmax = 0;
    float scale = 0.f;
    void *stream = nullptr;
    const gqa_decode_options *opts = nullptr;
    bool own_ws = false;   // the workspace is the library's own scratch, checked by its owner
};

// The score scale a call uses: the caller's value, or 1/sqrt(d) for
// GQA_SCALE_DEFAULT (0), rounded once from the double-precision value.
float resolve_scale(float scale, int d) {
    return scale == 0.f ? (float)(1.0 / std::sqrt((double)d)) : scale;
}

// Every check that needs no device work, in the order the header documents:
// arguments, workspace, path, device.  On GQA_OK, *path_out and *dev_out hold
// the path the call takes and the device's facts.
gqa_status validate(const DecodeRequest &r, int *path_out, DeviceInfo *dev_out) {
    if (!r.q || !r.k || !r.v || !r.out) return GQA_ERR_INVALID_ARG;
    const int B = r.B, H = r.H, G = r.G, d = r.d, Lmax = r.Lmax;
    gqa_status s = check_shape(B, H, G, d, Lmax);
    if (s != GQA_OK) return s;
    if (!std::isfinite(r.scale)) return GQA_ERR_INVALID_ARG;
    if (!aligned(r.k, 16) || !aligned(r.v, 16) || !aligned(r.q, 16) || !aligned(r.out, 16) ||
        !aligned(r.seq_lens, 4) || !aligned(r.k_new, 16) || !aligned(r.v_new, 16) || !aligned(r.block_table, 4))
        return GQA_ERR_INVALID_ARG;
    gqa_decode_options o{};
    if (r.opts) o = *r.opts;
    for (int x : o.reserved)
        if (x != 0) return GQA_ERR_INVALID_ARG;
    if (o.num_ctas < 0 || o.num_ctas > GQA_MAX_CTAS) return GQA_ERR_INVALID_ARG;
    if (o.path < 0 || o.path > GQA_PATH_TCGEN05 || o.window < 0) return GQA_ERR_INVALID_ARG;
    if (!r.own_ws && (!r.ws || !aligned(r.ws, 256) || r.ws_bytes < workspace_bytes_for(B, H, G, d, Lmax)))
        return GQA_ERR_WORKSPACE;

    const int n = H / G;
    const int path = o.path ? o.path : auto_path(H, G, d);
    if (path == GQA_PATH_SIMT && n > gqa::simt_max_heads()) return GQA_ERR_UNSUPPORTED;
    if (path == GQA_PATH_TCGEN05 && n > gqa::tc_max_heads()) return GQA_ERR_UNSUPPORTED;
    // the CUDA-core path reads a contiguous cache, every valid position
    if (path == GQA_PATH_SIMT && (r.block_table || r.k_new || o.window > 0)) return GQA_ERR_UNSUPPORTED;

    s = device_info(dev_out);
    if (s != GQA_OK) return s;
    *path_out = path;
    return GQA_OK;
}

gqa_status decode_impl(const DecodeRequest &r) {
    int path = 0;
    DeviceInfo dev;
    const gqa_status s = validate(r, &path, &dev);
    if (s != GQA_OK) return s;
    const int B = r.B, H = r.H, G = r.G, d = r.d, Lmax = r.Lmax;
    const int n = H / G;
    gqa_decode_options o{};
    if (r.opts) o = *r.opts;

    const bool paired = path == GQA_PATH_TCGEN05 && gqa::tc_paired(d, Lmax, n);
    const int tile_pos = paired ? 2 * gqa::kTile : gqa::kTile;
    // One CTA per SM, never more than there are tiles.
    const long long tiles_max = (long long)B * G * ((Lmax + tile_pos - 1) / tile_pos);
    long long ctas = o.num_ctas ? o.num_ctas : dev.sms;
    if (ctas > GQA_MAX_CTAS) ctas = GQA_MAX_CTAS;
    if (ctas > tiles_max) ctas = tiles_max;
    if (ctas < 1) ctas = 1;

    uint8_t *ws = static_cast<uint8_t *>(r.ws);
    DecodeParams p;
    p.q = static_cast<const __nv_bfloat16 *>(r.q);
    p.seq_lens = r.seq_lens;
    p.window = o.window;
    p.block_table = r.block_table;
    p.page_shift = 0;
    while (r.block_table && (1 << p.page_shift) < r.page_size) ++p.page_shift;
    p.max_pages = r.max_pages;
    p.num_pages = r.num_pages;
    p.k_new = static_cast<const __nv_bfloat16 *>(r.k_new);
    p.v_new = static_cast<const __nv_bfloat16 *>(r.v_new);
    p.k_dst = r.k_new ? static_cast<__nv_bfloat16 *>(const_cast<void *>(r.k)) : nullptr;
    p.v_dst = r.v_new ? static_cast<__nv_bfloat16 *>(const_cast<void *>(r.v)) : nullptr;
    p.out = r.out;
#ifdef GQA_TEST_HOOKS
    p.withhold_k = g_withhold_k.exchange(-1);
#else
    p.withhold_k = -1;
#endif
    p.flags = reinterpret_cast<unsigned int *>(ws);
    p.ticket = reinterpret_cast<unsigned int *>(ws + 4);
    p.fails = reinterpret_cast<unsigned int *>(ws + 8);
    // The CUDA-core path splits statically; so does the paired d=64 tcgen05 form, whose
    // piece ends (two GEMM parts per tile) cost more than per-SM balancing wins back.
    p.dyn_cap = (path == GQA_PATH_TCGEN05 && !paired) ? dyn_cap_for(B, G, Lmax) : 0;
    p.tile_shift = paired ? 8 : 7;
    p.partials = reinterpret_cast<float *>(ws + zero_prefix_bytes(B, G));
    p.B = B;
    p.H = H;
    p.G = G;
    p.n = n;
    p.Lmax = Lmax;
    p.scale_log2 = resolve_scale(r.scale, d) * 1.4426950408889634f;

    CUtensorMap tk, tv;
    const bool maps_ok = r.block_table
                             ? make_page_map(&tk, r.k, r.num_pages, G, d, r.page_size, paired) &&
                                   make_page_map(&tv, r.v, r.num_pages, G, d, r.page_size, paired)
                             : make_cache_map(&tk, r.k, B, G, d, Lmax, paired) &&
                                   make_cache_map(&tv, r.v, B, G, d, Lmax, paired);
    if (!maps_ok) return GQA_ERR_LAUNCH;
    cudaStream_t st = static_cast<cudaStream_t>(r.stream);
    cudaError_t e;
    if (path == GQA_PATH_SIMT) {
        e = gqa::launch_decode_simt(tk, tv, p, d, (int)ctas, st);
    } else {
        const int rows = gqa::tc_rows_for(n);
        CUtensorMap tq;
        if (!make_q_map(&tq, r.q, B, H, d, rows)) return GQA_ERR_LAUNCH;
        gqa::TailMaps tails;
        std::memset(&tails, 0, sizeof tails);
        const bool plain = !r.block_table && !r.k_new && o.window == 0;   // the instances that trim last tiles
        for (int t = 0; plain && t < 3; ++t)
            if (!make_cache_map(&tails.k[t], r.k, B, G, d, Lmax, paired, 64 >> t) ||
                !make_cache_map(&tails.v[t], r.v, B, G, d, Lmax, paired, 64 >> t))
                return GQA_ERR_LAUNCH;
        e = gqa::launch_decode_tc(tk, tv, tq, tails, p, d, paired, (int)ctas, st);
    }
    if (e == cudaErrorNotSupported) return GQA_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return GQA_ERR_LAUNCH;
    // merge the segments the work split cut across CTAs (a no-op grid when none is)
    e = gqa::launch_split_combine(p, d, (int)ctas, st);
    return e == cudaSuccess ? GQA_OK : GQA_ERR_LAUNCH;
}

}  // namespace

namespace gqa {
size_t decode_workspace_zero_prefix(int B, int G) { return zero_prefix_bytes(B, G); }

gqa_status decode_check(const void *q, const void *k_cache, const void *v_cache, const int32_t *seq_lens,
                        float *out, void *workspace, size_t workspace_bytes, int B, int H, int G, int d, int Lmax,
                        float scale) {
    DecodeRequest r;
    r.q = q;
    r.k = k_cache;
    r.v = v_cache;
    r.seq_lens = seq_lens;
    r.out = out;
    r.ws = workspace;
    r.ws_bytes = workspace_bytes;
    r.own_ws = workspace == nullptr;
    r.B = B, r.H = H, r.G = G, r.d = d, r.Lmax = Lmax;
    r.scale = scale;
    int path = 0;
    DeviceInfo dev;
    return validate(r, &path, &dev);
}
}  // namespace gqa

extern "C" {

const char *gqa_status_string(int status) {
    switch (status) {
        case GQA_OK: return "GQA_OK";
        case GQA_ERR_INVALID_ARG: return "GQA_ERR_INVALID_ARG: invalid argument";
        case GQA_ERR_UNSUPPORTED: return "GQA_ERR_UNSUPPORTED: shape or option not supported by this build";
        case GQA_ERR_WORKSPACE: return "GQA_ERR_WORKSPACE: workspace missing, misaligned or too small";
        case GQA_ERR_LAUNCH: return "GQA_ERR_LAUNCH: a CUDA call or kernel launch failed";
        case GQA_ERR_DEVICE: return "GQA_ERR_DEVICE: no usable sm_103 CUDA device";
        default: return "unknown gqa_status";
    }
}

int gqa_abi_version(void) { return GQA_ABI_VERSION; }

gqa_status gqa_decode_workspace_size(int B, int H, int G, int d, int Lmax, size_t *bytes) {
    if (!bytes) return GQA_ERR_INVALID_ARG;
    const gqa_status s = check_shape(B, H, G, d, Lmax);
    if (s != GQA_OK) return s;
    *bytes = workspace_bytes_for(B, H, G, d, Lmax);
    return GQA_OK;
}

int gqa_decode_select_path(int B, int H, int G, int d, int Lmax) {
    const gqa_status s = check_shape(B, H, G, d, Lmax);
    if (s != GQA_OK) return -(int)s;
    return auto_path(H, G, d);
}

gqa_status gqa_decode_ex(const void *q, const void *k_cache, const void *v_cache, const int32_t *seq_lens,
                         float *out, void *workspace, size_t workspace_bytes, int B, int H, int G, int d, int Lmax,
                         float scale, void *stream, const gqa_decode_options *opts) {
    DecodeRequest r;
    r.q = q;
    r.k = k_cache;
    r.v = v_cache;
    r.seq_lens = seq_lens;
    r.out = out;
    r.ws = workspace;
    r.ws_bytes = workspace_bytes;
    r.B = B, r.H = H, r.G = G, r.d = d, r.Lmax = Lmax;
    r.scale = scale;
    r.stream = stream;
    r.opts = opts;
    return decode_impl(r);
}

gqa_status gqa_decode(const void *q, const void *k_cache, const void *v_cache, const int32_t *seq_lens, float *out,
                      void *workspace, size_t workspace_bytes, int B, int H, int G, int d, int Lmax, float scale,
                      void *stream) {
    return gqa_decode_ex(q, k_cache, v_cache, seq_lens, out, workspace, workspace_bytes, B, H, G, d, Lmax, scale,
                         stream, nullptr);
}

gqa_status gqa_decode_append(const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                             const int32_t *seq_lens, float *out, void *workspace, size_t workspace_bytes, int B,
                             int H, int G, int d, int Lmax, float scale, void *stream,
                             const gqa_decode_options *opts) {
    if (!k_new || !v_new || !seq_lens) return GQA_ERR_INVALID_ARG;
    DecodeRequest r;
    r.q = q;
    r.k = k_cache;
    r.v = v_cache;
    r.k_new = k_new;
    r.v_new = v_new;
    r.seq_lens = seq_lens;
    r.out = out;
    r.ws = workspace;
    r.ws_bytes = workspace_bytes;
    r.B = B, r.H = H, r.G = G, r.d = d, r.Lmax = Lmax;
    r.scale = scale;
    r.stream = stream;
    r.opts = opts;
    return decode_impl(r);
}

gqa_status gqa_decode_paged(const void *q, void *k_pages, void *v_pages, const int32_t *block_table,
                            const int32_t *seq_lens, const void *k_new, const void *v_new, float *out,
                            void *workspace, size_t workspace_bytes, int B, int H, int G, int d, int page_size,
                            int max_pages, int num_pages, float scale, void *stream,
                            const gqa_decode_options *opts) {
    if (!block_table || (!k_new) != (!v_new) || (k_new && !seq_lens)) return GQA_ERR_INVALID_ARG;
    if (page_size < kMinPage || page_size > kMaxPage || (page_size & (page_size - 1)) != 0 || max_pages <= 0 ||
        num_pages <= 0)
        return GQA_ERR_INVALID_ARG;
    if ((long long)max_pages * page_size > kMaxLmax || (long long)num_pages * G >= kMaxPoolRows)
        return GQA_ERR_UNSUPPORTED;
    DecodeRequest r;
    r.q = q;
    r.k = k_pages;
    r.v = v_pages;
    r.k_new = k_new;
    r.v_new = v_new;
    r.block_table = block_table;
    r.page_size = page_size;
    r.max_pages = max_pages;
    r.num_pages = num_pages;
    r.seq_lens = seq_lens;
    r.out = out;
    r.ws = workspace;
    r.ws_bytes = workspace_bytes;
    r.B = B, r.H = H, r.G = G, r.d = d, r.Lmax = max_pages * page_size;
    r.scale = scale;
    r.stream = stream;
    r.opts = opts;
    return decode_impl(r);
}

#ifdef GQA_TEST_HOOKS
void gqa_debug_withhold_copy(int tile) { g_withhold_k.store(tile < 0 ? -1 : tile); }
#endif

gqa_status gqa_decode_read_flags(void *workspace, uint32_t *flags, int clear, void *stream) {
    if (!workspace || !flags || !aligned(workspace, 256)) return GQA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t host = 0;
    if (cudaMemcpyAsync(&host, workspace, sizeof host, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        (clear && cudaMemsetAsync(workspace, 0, sizeof host, st) != cudaSuccess) ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        cudaGetLastError();
        return GQA_ERR_LAUNCH;
    }
    *flags = host;
    return GQA_OK;
}

gqa_status gqa_meanpool_kv_strided(const float *w_in, float *w_out, int64_t outer, int H, int G, int64_t inner,
                                   void *stream) {
    if (!w_in || !w_out) return GQA_ERR_INVALID_ARG;
    if (outer <= 0 || inner <= 0 || H <= 0 || G <= 0 || G > H || H % G != 0) return GQA_ERR_INVALID_ARG;
    if (!aligned(w_in, 4) || !aligned(w_out, 4)) return GQA_ERR_INVALID_ARG;
    DeviceInfo dev;
    const gqa_status s = device_info(&dev);
    if (s != GQA_OK) return s;
    const cudaError_t e = gqa::launch_meanpool(w_in, w_out, outer, H, G, inner, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GQA_OK : GQA_ERR_LAUNCH;
}

gqa_status gqa_meanpool_kv(const float *w_in, float *w_out, int H, int G, int h, int d_model, void *stream) {
    if (h <= 0 || d_model <= 0) return GQA_ERR_INVALID_ARG;
    return gqa_meanpool_kv_strided(w_in, w_out, 1, H, G, (int64_t)h * d_model, stream);
}

}  // extern "C"
