/*
 * CPU oracle for grouped-query attention (GQA) decode and for the K/V
 * mean-pool checkpoint conversion.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path links,
 * loads or calls this file.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header or constant
 * with the CUDA library.
 *
 * It is the plain definition, written out in float64 loops with no blocking,
 * fusion or reordering, so it can be checked against the pages by eye.
 *
 * Decode step  ["Grouped-query attention (GQA)" concept page, "Implementation
 * sketch", the decode-step pseudocode; arxiv:2305.13245 §2.2]:
 *   the H query heads are split into G groups; query head i uses the single
 *   key head and value head of its group g(i);
 *     scores_t = q[i] . K[t, g] / sqrt(h)        for every cached token t
 *     probs    = softmax(scores)
 *     out[i]   = sum_t probs_t * V[t, g]
 *   The pages leave the head-to-group map open; the same listing assumes
 *   contiguous blocks, so g(i) = i / (H/G).
 *   The scale is the caller's fp32 value (1/sqrt(h) in the pages), widened.
 *   Subtracting the row maximum before exp does not change the softmax.
 *   A sequence with no valid positions has an empty sum: its output is 0
 *   (this library's reading; the pages never decode an empty cache).
 *
 * Variants of the decode step (same definition, other inputs):
 *   - cross-attention: seq_lens NULL, every one of the Lmax positions is valid;
 *   - sliding window: only the last `window` valid positions are attended;
 *   - paged cache: oracle_gather_pages turns a page pool + block table into the
 *     contiguous cache, which the decode then reads;
 *   - fused append: oracle_append_row writes the new token's K (or V) row at
 *     position seq_lens[b] - 1 before the decode.
 *   Each function's comment names the passage it follows.
 *
 * Mean-pool conversion  [same page, "Implementation sketch", the conversion
 * pseudocode, and "Converted and uptrained checkpoints"; arxiv:2305.13245 §2.1]:
 *   the K (and, separately, V) projection of group g is the mean of the
 *   projections of the H/G heads in that group.  Reading: sum the members in
 *   increasing head order, then divide by H/G once.  The fp32 version does
 *   exactly that in fp32 (for a bit-exact comparison); the fp64 version is its
 *   twin in double.
 *
 * Parity pins: every function here is pinned by the CPU tests (independent
 * MHA/MQA formulations, replication, closed forms, brute force in high
 * precision, invariances).  No function is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the top half of an IEEE float32; widening is exact. */
static double bf16_value(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Head-to-group map: contiguous blocks of H/G query heads. */
int oracle_group_of(int i, int H, int G) { return i / (H / G); }

/*
 * The positions sequence b attends to: t0 <= t < T.
 *   T  = seq_lens[b]; with seq_lens == NULL every sequence holds Lmax valid
 *        positions.  That is decoder cross-attention over an encoder cache of
 *        fixed length, where GQA applies as it does to decoder self-attention
 *        ["Grouped-query attention (GQA)" concept page, "When to use which",
 *        last row; arxiv:2305.13245 §3.1].
 *   t0 = T - window when 0 < window < T, else 0: sliding-window attention, the
 *        last `window` positions only (the same page, "Variants", "Decoder-only
 *        models with GQA": Mistral 7B pairs GQA with a sliding window).  The
 *        pages give no window size; it is the caller's parameter.
 */
static void attended_range(const int32_t *seq_lens, int b, int Lmax, int window, int *t0, int *T) {
    *T = seq_lens ? seq_lens[b] : Lmax;
    *t0 = (window > 0 && *T > window) ? *T - window : 0;
}

/*
 * q        [B, H, d]        bf16 bits
 * k, v     [B, G, Lmax, d]  bf16 bits
 * seq_lens [B]              valid cache length per sequence, 0 <= . <= Lmax;
 *                           NULL: every sequence has Lmax valid positions
 * window   0: attend to every valid position; > 0: to the last `window` only
 * out      [B, H, d]        float64; only the requested rows are written
 * rows     optional list of flat row ids (b * H + i); NULL means every row
 * Returns 0, or -1 on a bad argument.
 */
int oracle_gqa_decode_window_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                 const int32_t *seq_lens, int window, double *out,
                                 int B, int H, int G, int d, int Lmax, float scale,
                                 const int64_t *rows, int64_t nrows) {
    if (B < 0 || H <= 0 || G <= 0 || d <= 0 || Lmax < 0 || H % G != 0 || window < 0) return -1;
    if (seq_lens)
        for (int b = 0; b < B; ++b)
            if (seq_lens[b] < 0 || seq_lens[b] > Lmax) return -1;
    const int64_t total = rows ? nrows : (int64_t)B * H;
    const double sc = (double)scale;
    int bad = 0;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < total; ++r) {
        const int64_t row = rows ? rows[r] : r;
        const int b = (int)(row / H);
        const int i = (int)(row % H);
        const int g = oracle_group_of(i, H, G);
        int t0, T;
        attended_range(seq_lens, b, Lmax, window, &t0, &T);
        const uint16_t *qi = q + ((int64_t)b * H + i) * d;
        const uint16_t *kg = k + ((int64_t)b * G + g) * Lmax * d;
        const uint16_t *vg = v + ((int64_t)b * G + g) * Lmax * d;
        double *o = out + row * d;

        if (T == 0) {
            for (int j = 0; j < d; ++j) o[j] = 0.0;
            continue;
        }
        double *s = (double *)malloc(sizeof(double) * (size_t)T);
        if (!s) {
#pragma omp atomic write
            bad = 1;
            continue;
        }
        /* scores_t = scale * sum_j q[i, j] * k[t, g, j] */
        for (int t = t0; t < T; ++t) {
            double dot = 0.0;
            for (int j = 0; j < d; ++j)
                dot += bf16_value(qi[j]) * bf16_value(kg[(int64_t)t * d + j]);
            s[t] = sc * dot;
        }
        /* softmax over t, with the maximum subtracted */
        double m = s[t0];
        for (int t = t0 + 1; t < T; ++t)
            if (s[t] > m) m = s[t];
        double l = 0.0;
        for (int t = t0; t < T; ++t) {
            s[t] = exp(s[t] - m);
            l += s[t];
        }
        /* out = (sum_t p_t * v_t) / l */
        for (int j = 0; j < d; ++j) {
            double acc = 0.0;
            for (int t = t0; t < T; ++t)
                acc += s[t] * bf16_value(vg[(int64_t)t * d + j]);
            o[j] = acc / l;
        }
        free(s);
    }
    return bad ? -1 : 0;
}

/* The decode step over every valid position (no window). */
int oracle_gqa_decode_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          const int32_t *seq_lens, double *out,
                          int B, int H, int G, int d, int Lmax, float scale,
                          const int64_t *rows, int64_t nrows) {
    return oracle_gqa_decode_window_f64(q, k, v, seq_lens, 0, out, B, H, G, d, Lmax, scale, rows, nrows);
}

/*
 * Paged cache -> contiguous cache.  A paged cache stores each sequence's
 * positions in fixed-size pages drawn from a shared pool and lists them in a
 * block table, the layout of paged attention (named on the GQA paper's page,
 * "How researchers see this paper": a citing serving paper lists it beside
 * GQA as a way to cut decode memory).  Layout read here: one page holds page_size consecutive positions of
 * all G K/V heads, head-major inside the page.
 *   pages  [num_pages, G, page_size, d]  bf16 bits
 *   table  [B, max_pages]                page of positions p*page_size .. of sequence b
 *   out    [B, G, Lmax, d]               out[b, g, t] = pages[table[b, t / page_size], g, t % page_size]
 *                                        for t < T_b (seq_lens NULL: T_b = Lmax); rows t >= T_b untouched
 * Only the table entries of valid positions are read.  Returns -1 on a bad
 * argument or when such an entry is not a page of the pool.
 */
int oracle_gather_pages(const uint16_t *pages, const int32_t *table, const int32_t *seq_lens, uint16_t *out,
                        int B, int G, int d, int page_size, int max_pages, int num_pages, int Lmax) {
    if (B < 0 || G <= 0 || d <= 0 || page_size <= 0 || max_pages < 0 || num_pages < 0 || Lmax < 0) return -1;
    if ((int64_t)max_pages * page_size < Lmax) return -1;
    for (int b = 0; b < B; ++b) {
        const int T = seq_lens ? seq_lens[b] : Lmax;
        if (T < 0 || T > Lmax) return -1;
        for (int t = 0; t < T; ++t) {
            const int page = table[(int64_t)b * max_pages + t / page_size];
            if (page < 0 || page >= num_pages) return -1;
            for (int g = 0; g < G; ++g) {
                const uint16_t *src = pages + (((int64_t)page * G + g) * page_size + t % page_size) * d;
                uint16_t *dst = out + (((int64_t)b * G + g) * Lmax + t) * d;
                memcpy(dst, src, sizeof(uint16_t) * (size_t)d);
            }
        }
    }
    return 0;
}

/*
 * Cache append of the decode step: the new token's key and value (one row per
 * K/V head) go to position T_b - 1 of each sequence, the position the decode
 * then attends to last ("Grouped-query attention (GQA)" concept page,
 * "Implementation sketch", the decode-step pseudocode appends to the cache
 * before attending; T_b counts the new token).  Sequences with T_b = 0 are
 * left alone.
 *   cache [B, G, Lmax, d] bf16 bits (K or V), updated in place
 *   row   [B, G, d]       bf16 bits
 */
int oracle_append_row(uint16_t *cache, const uint16_t *row, const int32_t *seq_lens, int B, int G, int d, int Lmax) {
    if (B < 0 || G <= 0 || d <= 0 || Lmax < 0 || !seq_lens) return -1;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] < 0 || seq_lens[b] > Lmax) return -1;
    for (int b = 0; b < B; ++b) {
        const int T = seq_lens[b];
        if (T == 0) continue;
        for (int g = 0; g < G; ++g)
            memcpy(cache + (((int64_t)b * G + g) * Lmax + (T - 1)) * d, row + ((int64_t)b * G + g) * d,
                   sizeof(uint16_t) * (size_t)d);
    }
    return 0;
}

/*
 * Mean-pool of head projections within each group.
 * w   [outer, H, inner]  fp32   (inner = h * d_model for the head-major
 *                                [H, h, d_model] layout with outer = 1; for the
 *                                pages' [d_model, H*h] layout, outer = d_model
 *                                and inner = h)
 * out [outer, G, inner]  fp32
 * out[o, g, x] = ((w[o, g*n, x] + w[o, g*n+1, x]) + ... + w[o, g*n+n-1, x]) / n
 */
int oracle_meanpool_f32(const float *w, float *out, int64_t outer, int H, int G,
                        int64_t inner) {
    if (outer < 0 || H <= 0 || G <= 0 || inner < 0 || H % G != 0) return -1;
    const int n = H / G;
    for (int64_t o = 0; o < outer; ++o)
        for (int g = 0; g < G; ++g)
            for (int64_t x = 0; x < inner; ++x) {
                float acc = w[(o * H + (int64_t)g * n) * inner + x];
                for (int j = 1; j < n; ++j)
                    acc = acc + w[(o * H + (int64_t)g * n + j) * inner + x];
                out[(o * G + g) * inner + x] = acc / (float)n;
            }
    return 0;
}

int oracle_meanpool_f64(const float *w, double *out, int64_t outer, int H, int G,
                        int64_t inner) {
    if (outer < 0 || H <= 0 || G <= 0 || inner < 0 || H % G != 0) return -1;
    const int n = H / G;
    for (int64_t o = 0; o < outer; ++o)
        for (int g = 0; g < G; ++g)
            for (int64_t x = 0; x < inner; ++x) {
                double acc = (double)w[(o * H + (int64_t)g * n) * inner + x];
                for (int j = 1; j < n; ++j)
                    acc = acc + (double)w[(o * H + (int64_t)g * n + j) * inner + x];
                out[(o * G + g) * inner + x] = acc / (double)n;
            }
    return 0;
}
