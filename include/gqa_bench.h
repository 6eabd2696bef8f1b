/*
 * gqa_bench.h — measurement helper of the B300 GQA decode library (a separate
 * shared object, libgqa_b300_bench.so; not part of the decode ABI in gqa.h).
 *
 * The decode step is bound by reading the KV cache ["Grouped-query attention
 * (GQA)" concept page, "Overview": decoding reads the whole key and value cache
 * for every new token, so memory bandwidth limits speed].  This helper measures
 * the read bandwidth that access pattern can reach on the device, as a ceiling
 * for the decode kernel beside the copy bandwidth: one thread block per SM
 * streams a contiguous range of a bf16 buffer through shared memory with the
 * decode kernel's TMA boxes (64 columns x 128 rows, 128-byte swizzle, two boxes
 * per 32 KiB tile, a six-stage ring) and does nothing with the data.
 */
#ifndef GQA_B300_GQA_BENCH_H
#define GQA_B300_GQA_BENCH_H

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Reads the whole buffer once, asynchronously on `stream`.
 *   buf      device, bf16 [z, rows, 128] (256-byte rows), 16-byte aligned
 *   z, rows  >= 1; rows a multiple of 128
 *   ctas     thread blocks (0: one per SM)
 *   flags    device, one uint32 (zero before the call): bit 0x2 is OR-ed in if a
 *            pipeline wait ran out (bounded at about one second), as in the decode
 *            library's flag word
 * Returns 0, or a nonzero code for an invalid argument (1), no usable device (5)
 * or a failed launch (4); nothing is enqueued on an error.
 */
int gqa_bench_stream_read(const void *buf, long long z, long long rows, int ctas, unsigned int *flags,
                          void *stream);

/*
 * The same read with every 32 KiB tile fetched as pages, as the decode kernel
 * fetches a paged cache whose pages are smaller than its 128-position tile: the
 * per-box cost of small pages.
 *   page_rows  16, 32, 64 or 128: each tile is 128/page_rows pages, two boxes of
 *              64 columns x page_rows rows each
 *   lanes      1..32: lanes of the issuing warp that issue a tile's boxes (lane l
 *              issues boxes l, l + lanes, ...)
 *   scatter    nonzero: page q of the stream is read from page slot q * A mod
 *              npages (A odd, npages = z * rows / page_rows, which must then be a
 *              power of two), so consecutive pages sit far apart as in a pool;
 *              zero: in order
 *   one_box    zero: two boxes per page (64 columns x page_rows rows each);
 *              nonzero: one box per page, through a five-dimensional tensor map
 *              (64 columns, 8 rows, 2 column halves, page_rows / 8 row groups,
 *              pages) that lands the page as [row group][half][8 rows][128 bytes]
 *   warps      1 or 2: issuing warps, taking alternate tiles
 * Other arguments as for gqa_bench_stream_read; returns 0, 1 (invalid argument),
 * 4 (launch failed or the three-dimensional map refused), 5 (no usable device) or
 * 6 (the driver refused the five-dimensional map).
 */
int gqa_bench_stream_read_pages(const void *buf, long long z, long long rows, int page_rows, int lanes, int scatter,
                                int one_box, int warps, int ctas, unsigned int *flags, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GQA_B300_GQA_BENCH_H */
