/*
 * gqa.h — C ABI of the B300 (sm_103a) grouped-query attention decode library.
 *
 * Grouped-query attention (GQA): the H query heads are split into G groups and
 * every query head of group g attends with that group's single key head and
 * value head, so the KV cache holds G instead of H K/V heads per token.
 * G = 1 is multi-query attention, G = H is multi-head attention.
 * ["Grouped-query attention (GQA)" concept page, "Overview" and "Choosing the
 *  group count G"; arxiv:2305.13245 §2.2]
 *
 * Conventions shared by every entry point:
 *   - G counts K/V heads, as in the GQA paper (GQA-8 has 8 K/V heads).  It is
 *     not Gemma 2's `num_groups` (query heads per K/V head).  [same page,
 *     "Contradictions"]
 *   - Query head i belongs to group g(i) = i / (H/G) (contiguous blocks; the
 *     paper leaves the map open and the page's conversion sketch assumes
 *     blocks).
 *   - Device pointers are CUDA global-memory addresses on the current device.
 *     bf16 tensors are passed as `const void*` holding IEEE bfloat16 values.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call
 *     only enqueues work on `stream` and never synchronises; results are ready
 *     when the stream reaches that point.
 *   - The library never allocates device memory and keeps no per-call state on
 *     the host.  The caller owns every buffer.
 *   - Host-checkable errors return before anything is enqueued.  A failed
 *     launch returns GQA_ERR_LAUNCH.
 *   - Thread safety: calls from several host threads are safe; two calls that
 *     share a workspace must not overlap on the device (calls on one stream
 *     never do).
 *   - Per-device facts (SM count, kernel attributes, the no-alloc scratch
 *     address) are looked up on the first call on each device and kept for the
 *     life of the process: do not use the library across a cudaDeviceReset.
 */
#ifndef GQA_B300_GQA_H
#define GQA_B300_GQA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GQA_ABI_VERSION 2

/* scale value that selects 1/sqrt(d) (see gqa_decode). */
#define GQA_SCALE_DEFAULT 0.0f

/* Leading bytes of a decode workspace that hold its counters (see
 * gqa_decode_workspace_size); the same for every shape. */
#define GQA_WORKSPACE_HEADER_BYTES 256u

typedef enum gqa_status {
    GQA_OK = 0,
    GQA_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, H % G != 0, bad stride */
    GQA_ERR_UNSUPPORTED = 2,   /* valid but not built: head dim, H/G, batch or size limits */
    GQA_ERR_WORKSPACE = 3,     /* workspace null or smaller than gqa_decode_workspace_size() */
    GQA_ERR_LAUNCH = 4,        /* a CUDA call or kernel launch failed */
    GQA_ERR_DEVICE = 5         /* no usable CUDA device, or not an sm_103 device */
} gqa_status;

/* Bits the decode kernel ORs into the workspace's flag word (see gqa_decode_read_flags). */
#define GQA_FLAG_SEQ_LEN_CLAMPED 0x1u  /* some seq_lens[b] was < 0 or > Lmax; it was clamped */
#define GQA_FLAG_WAIT_TIMEOUT    0x2u  /* a pipeline wait ran out; that call's output is invalid */
#define GQA_FLAG_BAD_PAGE        0x4u  /* a block-table entry needed by gqa_decode_paged was not a page
                                          of the pool; its rows were read as zeros */

/* Kernel variants of gqa_decode_ex. */
#define GQA_PATH_AUTO    0   /* pick per shape (the default of gqa_decode) */
#define GQA_PATH_SIMT    1   /* CUDA-core dot products and online softmax, H/G <= 8 */
#define GQA_PATH_TCGEN05 2   /* fifth-generation tensor cores (tcgen05, TMEM), H/G <= 64 */

/* Limits of this build. */
#define GQA_MAX_BATCH 1024
#define GQA_MAX_CTAS 1024

/* Human-readable name of a status code.  Never NULL. */
const char *gqa_status_string(int status);

/* GQA_ABI_VERSION of the loaded library. */
int gqa_abi_version(void);

/*
 * Bytes of device workspace gqa_decode needs for this shape.  The value does not
 * depend on seq_lens or on the device; it grows with B*G and with Lmax (slots
 * for the dynamically claimed part of long work lists, at most 8192 of them).
 * Writes *bytes and returns GQA_OK, or returns the status gqa_decode would
 * return for the same shape.
 *
 * Layout: GQA_WORKSPACE_HEADER_BYTES of counters (the flag word, the claim
 * ticket and the failed-claim count of the dynamic work pool), then the
 * split-combine partial results (one (m, l, acc) triple per query head per
 * piece of a sequence).
 * It MUST be zero-filled before its first use (for example
 * cudaMemsetAsync(ws, 0, bytes, stream)) so that the counters start clear.
 * Every call leaves the two pool counters at zero again, so nothing needs resetting
 * between calls, whatever their shapes (one workspace of the largest size
 * serves them all) — except after a call that set GQA_FLAG_WAIT_TIMEOUT: zero
 * the first GQA_WORKSPACE_HEADER_BYTES again before the next call.  The flag
 * word is only ever OR-ed into.
 */
gqa_status gqa_decode_workspace_size(int B, int H, int G, int d, int Lmax, size_t *bytes);

/*
 * One GQA decode step over a bf16 KV cache.
 * ["Grouped-query attention (GQA)" concept page, "Implementation sketch", the
 *  decode-step pseudocode; arxiv:2305.13245 §2.2]
 *
 * For every sequence b and query head i, with g = i / (H/G) and
 * T = seq_lens[b]:
 *   s_t        = scale * sum_j q[b,i,j] * k_cache[b,g,t,j]      t = 0 .. T-1
 *   out[b,i,:] = sum_t softmax(s)_t * v_cache[b,g,t,:]
 * The token being decoded must already be in the cache (the page appends the new
 * key and value before attending), so T counts it.  There is no mask inside the
 * T positions.  Positions t >= T are never used; they may hold anything,
 * including NaN.  T = 0 gives out = 0.
 *
 * q         device, bf16 [B, H, d], contiguous (row b*H+i holds head i of sequence b)
 * k_cache   device, bf16 [B, G, Lmax, d], contiguous; 16-byte aligned
 * v_cache   device, bf16 [B, G, Lmax, d], contiguous; 16-byte aligned
 * seq_lens  device, int32 [B]; expected 0 <= seq_lens[b] <= Lmax.  Values outside
 *           are clamped into that range on the device and GQA_FLAG_SEQ_LEN_CLAMPED
 *           is set in the workspace flag word.
 *           NULL: every sequence has all Lmax positions valid.  This is decoder
 *           cross-attention over a fixed-length encoder cache, where GQA applies
 *           as it does to self-attention ["Grouped-query attention (GQA)"
 *           concept page, "When to use which", last row; arxiv:2305.13245 §3.1].
 * out       device, float32 [B, H, d], contiguous.  Must not overlap any input.
 * workspace device, zero-filled before first use, >= gqa_decode_workspace_size bytes,
 *           256-byte aligned.  Used by one call at a time.
 * B         1 .. GQA_MAX_BATCH
 * H, G      H >= G >= 1, H % G == 0, H/G <= 64
 * d         head dimension: 64 or 128
 * Lmax      >= 1, cache capacity per sequence, at most 2^24; B*G*ceil(Lmax/128) <= 2^30
 * scale     score scale (fp32), finite.  GQA_SCALE_DEFAULT (0) selects 1/sqrt(d),
 *           the pages' scale ["Grouped-query attention (GQA)" concept page,
 *           "Implementation sketch": scores divided by sqrt(h)], rounded once to
 *           fp32; any other value is used as given.
 *
 * Arithmetic: exact bf16 products accumulated in fp32, softmax in fp32 with a
 * running maximum, fp32 output.  Measured against a float64 evaluation of the
 * definition: max abs error <= 1e-2 and, per output row, max error <= 2e-3 of
 * the row's largest |value| on the benchmark workloads.
 *
 * Two kernels are enqueued: the split decode kernel and the split-combine
 * kernel that merges the sequences the work split cut across thread blocks.
 * Both use programmatic stream serialisation: each may start its on-chip
 * set-up while the previous kernel on `stream` drains (the split-combine sits
 * beside the decode kernel's blocks, the next decode beside the split-combine's),
 * and touches global memory only after that kernel has completed.
 */
gqa_status gqa_decode(const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *seq_lens, float *out,
                      void *workspace, size_t workspace_bytes,
                      int B, int H, int G, int d, int Lmax, float scale, void *stream);

/* Knobs for tests and tuning.  Zero-initialise, then set what you need. */
typedef struct gqa_decode_options {
    int path;          /* GQA_PATH_*; 0 = automatic */
    int num_ctas;      /* CTAs of the split kernel; 0 = automatic (1..GQA_MAX_CTAS) */
    int window;        /* sliding window: > 0 attends to the last `window` valid
                          positions of each sequence only, max(0, T - window) <= t < T;
                          0 = every valid position.  Mistral 7B pairs GQA with a
                          sliding window ["Grouped-query attention (GQA)" concept
                          page, "Variants", "Decoder-only models with GQA"]; the
                          pages give no size, so it is the caller's.  Tensor-core
                          path only. */
    int reserved[5];   /* must be zero */
} gqa_decode_options;

/* gqa_decode with explicit options (opts may be NULL = defaults).  A path that
 * does not support the shape returns GQA_ERR_UNSUPPORTED. */
gqa_status gqa_decode_ex(const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *seq_lens, float *out,
                         void *workspace, size_t workspace_bytes,
                         int B, int H, int G, int d, int Lmax, float scale, void *stream,
                         const gqa_decode_options *opts);

/*
 * Decode step with the cache append fused in.
 * ["Grouped-query attention (GQA)" concept page, "Implementation sketch": the
 *  decode step appends the new token's key and value to the cache, then attends]
 *
 * For every sequence b with T = seq_lens[b] >= 1 and K/V head g, the new rows
 * k_new[b, g, :] and v_new[b, g, :] are written to k_cache[b, g, T-1, :] and
 * v_cache[b, g, T-1, :], and the decode of gqa_decode_ex runs over the T
 * positions with those rows in place (the written rows are the ones attended
 * to; the caches' old contents at T-1 are never used).  Sequences with T = 0 are
 * not written and give out = 0.  One launch pair, as gqa_decode.
 *
 * k_new, v_new  device, bf16 [B, G, d], contiguous, 16-byte aligned
 * k_cache, v_cache  as gqa_decode, but written (row T-1 of each sequence)
 * seq_lens  device, int32 [B], required (counts the new token)
 * Other arguments as gqa_decode_ex.  Tensor-core path only.
 */
gqa_status gqa_decode_append(const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                             const int32_t *seq_lens, float *out, void *workspace, size_t workspace_bytes,
                             int B, int H, int G, int d, int Lmax, float scale, void *stream,
                             const gqa_decode_options *opts);

/*
 * Decode step over a paged KV cache.
 * [paged attention is named on the GQA paper's page, "How researchers see this
 *  paper", where a citing serving paper lists it beside GQA; the layout is this
 *  library's choice]
 *
 * The cache is a pool of num_pages pages; page p holds page_size consecutive
 * positions of all G K/V heads:
 *   k_pages, v_pages  device, bf16 [num_pages, G, page_size, d], 16-byte aligned
 *   block_table       device, int32 [B, max_pages]: position t of sequence b is
 *                     row t % page_size of page block_table[b, t / page_size]
 * Only the entries of attended positions are read (t < seq_lens[b], and inside
 * the window if one is set).  An entry outside [0, num_pages) reads zeros and
 * sets GQA_FLAG_BAD_PAGE.
 * page_size   a power of two, 16 .. 2^20
 * max_pages   >= 1; the cache capacity per sequence is Lmax = max_pages * page_size
 *             (workspace: gqa_decode_workspace_size(B, H, G, d, Lmax))
 * num_pages   >= 1, num_pages * G < 2^31
 * k_new, v_new  optional (both or neither): fused append as gqa_decode_append,
 *             written into the page that holds position seq_lens[b] - 1
 * seq_lens    as gqa_decode (NULL: every sequence has Lmax positions; not with
 *             k_new)
 * Computes exactly what gqa_decode_ex computes on the contiguous cache
 * [b, g, t, :] = pages[block_table[b, t / page_size], g, t % page_size, :].
 * Tensor-core path only.
 */
gqa_status gqa_decode_paged(const void *q, void *k_pages, void *v_pages, const int32_t *block_table,
                            const int32_t *seq_lens, const void *k_new, const void *v_new, float *out,
                            void *workspace, size_t workspace_bytes, int B, int H, int G, int d, int page_size,
                            int max_pages, int num_pages, float scale, void *stream,
                            const gqa_decode_options *opts);

/* The path gqa_decode would take for this shape (GQA_PATH_SIMT or
 * GQA_PATH_TCGEN05), or a negative gqa_status if the shape is rejected. */
int gqa_decode_select_path(int B, int H, int G, int d, int Lmax);

#ifdef GQA_TEST_HOOKS
/*
 * Test hook for the failure path, exported only by the test-hooks build of the
 * library (compiled with -DGQA_TEST_HOOKS; the product build has neither the
 * symbol nor the check in its kernels).  In the next decode call on the
 * tensor-core path (any thread, any entry point), thread block 0 skips its K
 * copy number `tile` (counted from 0 in its own copy order): nothing ever
 * arrives on that copy's barrier, so the score GEMM's bounded wait runs out
 * after about one second, the block abandons its work, GQA_FLAG_WAIT_TIMEOUT is
 * set in the workspace flag word and the call's output is invalid.  The context
 * stays usable; zero the workspace before the next call.  A negative `tile`
 * cancels a pending request.
 */
void gqa_debug_withhold_copy(int tile);
#endif

/*
 * Copy the workspace flag word (GQA_FLAG_* bits, OR-ed by earlier decode calls)
 * to *flags.  Enqueued on `stream` and then synchronises that stream.
 * With clear != 0 the word is reset to zero afterwards (also on `stream`).
 */
gqa_status gqa_decode_read_flags(void *workspace, uint32_t *flags, int clear, void *stream);

/*
 * gqa_decode for callers that cannot allocate device memory.
 * The pages have no counterpart: this is a packaging variant of gqa_decode.
 *
 * Who needs it: callers with no way to hand over a workspace, for example a
 * plugin that only receives its input and output tensors from a host framework
 * that owns all device memory, a runtime that reserves its memory once at
 * start-up and may not allocate afterwards, or a latency-critical loop that
 * cannot pay for cudaMalloc's implicit device synchronisation.
 *
 * Instead of a caller workspace it uses a scratch array compiled into the
 * library: GQA_NOALLOC_WORKSPACE_BYTES of device memory that every GPU loading
 * the library holds until the process exits.  Arguments, layouts, results and
 * error codes are those of gqa_decode, except:
 *   - shapes whose gqa_decode_workspace_size exceeds GQA_NOALLOC_WORKSPACE_BYTES
 *     return GQA_ERR_WORKSPACE and enqueue nothing;
 *   - every argument check of gqa_decode runs first: a rejected call enqueues
 *     nothing and leaves the scratch alone;
 *   - the first call on a device looks up the scratch address on that device
 *     (make it before any stream capture on that device);
 *   - every call clears the scratch's header and piece counts on `stream`
 *     before the kernel (cudaMemsetAsync, no allocation): the flag word, the
 *     dynamic-pool counters and the per-segment counts.  A call that ran into a
 *     wait limit leaves those counters where its aborted blocks stopped; the
 *     next call starts clean without anything to do for the caller.  The flag
 *     word cannot be read back through this entry point;
 *   - all calls share the one array: calls that overlap on the GPU (other
 *     streams, other host threads) race and corrupt each other's results, so
 *     order them on one stream or synchronise between them.
 * It never calls cudaMalloc, cudaFree or any allocating routine.
 */
#define GQA_NOALLOC_WORKSPACE_BYTES (8u << 20)

gqa_status gqa_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                              const int32_t *seq_lens, float *out,
                              int B, int H, int G, int d, int Lmax, float scale, void *stream);

/*
 * Mean-pool conversion of K (or V) projection heads into G groups.
 * ["Grouped-query attention (GQA)" concept page, "Converted and uptrained
 *  checkpoints" and the conversion pseudocode; arxiv:2305.13245 §2.1]
 *
 * w_in   device, float32 [H, h, d_model], head-major (head i's projection slice)
 * w_out  device, float32 [G, h, d_model]
 * w_out[g, r, c] = ((w_in[g*n, r, c] + w_in[g*n+1, r, c]) + ... + w_in[g*n+n-1, r, c]) / n
 * with n = H/G, each addition and the division rounded in fp32 (IEEE, round to
 * nearest), in that order: the result is bit-identical to that sequence.
 * Call it once for W_K and once for W_V; the query and output projections are
 * left unchanged by the conversion.
 *
 * Asynchronous on `stream` (one kernel, no allocation, no synchronisation).
 * w_in and w_out must not overlap.  Rows of 16-byte aligned pointers with
 * h*d_model a multiple of 4 are read and written 16 bytes at a time; any
 * 4-byte aligned layout is accepted.
 * Returns GQA_ERR_INVALID_ARG (nothing enqueued) for a NULL pointer, H, G, h or
 * d_model <= 0, G > H, H not a multiple of G, or a pointer that is not 4-byte
 * aligned; GQA_ERR_DEVICE if no CUDA device is current; GQA_ERR_LAUNCH if the
 * kernel launch fails.
 */
gqa_status gqa_meanpool_kv(const float *w_in, float *w_out, int H, int G, int h, int d_model,
                           void *stream);

/*
 * The same pooling for any layout with heads on a middle axis:
 * w_in [outer, H, inner] -> w_out [outer, G, inner].  The head-major layout is
 * outer = 1, inner = h*d_model; the pages' [d_model, H*h] projection (head i in
 * columns i*h .. (i+1)*h-1) is outer = d_model, inner = h.
 */
gqa_status gqa_meanpool_kv_strided(const float *w_in, float *w_out, int64_t outer, int H, int G,
                                   int64_t inner, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GQA_B300_GQA_H */
