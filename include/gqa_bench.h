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

#ifdef __cplusplus
}
#endif

#endif /* GQA_B300_GQA_BENCH_H */
