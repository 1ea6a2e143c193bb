/*
 * pa_oracle.c -- plain CPU oracle for decode-step attention over a
 * block-paged KV cache, in double precision.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA path.
 *
 * Sources (four web pages on paged KV caches; cited by title and section):
 *   [BM]  "KV Cache and BlockManager" (dpshk.com/news/5906718)
 *   [KB]  vLLM memory-management course, ch. 3 "KV Block design"
 *   [BUG] "A strange KV Cache bug" (dpshk.com/news/5937191)
 *   [PG]  "KV Cache paging in LLM inference" (intelliparadigm.com)
 *
 * What it computes, step by step, with no blocking, fusion or reordering:
 *   1. validate a sequence's valid length and its block_table entries;
 *   2. gather the sequence's K and V rows through block_table into contiguous
 *      double arrays (the contiguous "valid KV" form of [BUG] s4.1);
 *   3. textbook softmax attention of one query row over those rows, masked
 *      to the valid length only ([BUG] s2.4, s4.2).
 * Plus the write path (append one token's K/V into the slot block_table
 * assigns, [BM] s4.4 and [BUG] s4.1), per-partition partial softmax sums
 * ([PG] s2.2 block-decomposed attention) and their merge.
 *
 * Pool layout: element (blk, kv_head, slot, d) of a pool sits at
 *   blk*block_stride + kv_head*block_size*head_dim + slot*head_dim + d
 * which is the per-layer slice of the [num_blocks][2][heads][block_size]
 * [head_dim] cache of [BM] s5.1 (K and V co-located, [KB] s3.2) when the
 * V pointer is the K pointer plus heads*block_size*head_dim and
 * block_stride = 2*heads*block_size*head_dim; separate K and V pools use
 * block_stride = heads*block_size*head_dim.
 *
 * Every pin of this file lives in tests/test_oracle.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { PAO_F32 = 0, PAO_F16 = 1, PAO_BF16 = 2 };

/* per-sequence status bits written to seq_err[b] */
enum { PAO_SEQ_BAD_LEN = 1, PAO_SEQ_BAD_BLOCK = 2, PAO_SEQ_BAD_POS = 4 };

/* ------------------------------------------------------------------------ */
/* element decoding: IEEE binary16 and bfloat16 bit patterns to double       */
/* ------------------------------------------------------------------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double f16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);            /* zero or subnormal */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + frac), expo - 25);
    }
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
static double bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int pao_dtype_bytes(int dtype)
{
    return dtype == PAO_F32 ? 4 : 2;
}

double pao_element(const void *base, int64_t idx, int dtype)
{
    if (dtype == PAO_F32) {
        float f;
        memcpy(&f, (const char *)base + idx * 4, 4);
        return (double)f;
    }
    uint16_t h;
    memcpy(&h, (const char *)base + idx * 2, 2);
    return dtype == PAO_F16 ? f16_to_double(h) : bf16_to_double(h);
}

void pao_convert(const void *src, int64_t n, int dtype, double *dst)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = pao_element(src, i, dtype);
}

/* ------------------------------------------------------------------------ */
/* block bookkeeping ([BM] s1 and s2)                                        */
/* ------------------------------------------------------------------------ */

/* Number of fixed-size blocks a sequence of `len` tokens occupies: the last
 * block may be partly filled, so this is the ceiling of len/block_size. */
int64_t pao_blocks_needed(int64_t len, int64_t block_size)
{
    return (len + block_size - 1) / block_size;
}

/* KV-cache bytes per layer: one K and one V vector of head_dim elements per
 * token and per head ([BM] s1, the "2 x batch x heads x tokens x head_dim x
 * dtype_bytes" formula, with tokens counted per sequence). */
int64_t pao_kv_bytes(int64_t seqs, int64_t heads, int64_t tokens_per_seq,
                     int64_t head_dim, int64_t dtype_bytes)
{
    return 2 * seqs * heads * tokens_per_seq * head_dim * dtype_bytes;
}

/* ------------------------------------------------------------------------ */
/* validation                                                                */
/* ------------------------------------------------------------------------ */

/* A sequence is usable iff 0 <= len <= max_blocks_per_seq*block_size and
 * each of its first ceil(len/block_size) table entries names a pool block
 * (entries past that are never read and may hold the -1 "unallocated"
 * marker of [BM] s5.1).  Returns the status bits. */
static int validate_sequence(int64_t len, int bs, int MB, int64_t NB,
                             const int32_t *table_row)
{
    if (len < 0 || len > (int64_t)MB * bs)
        return PAO_SEQ_BAD_LEN;
    int64_t nblk = pao_blocks_needed(len, bs);
    for (int64_t j = 0; j < nblk; ++j)
        if (table_row[j] < 0 || (int64_t)table_row[j] >= NB)
            return PAO_SEQ_BAD_BLOCK;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* gather: paged -> contiguous                                               */
/* ------------------------------------------------------------------------ */

/* Logical token t of a sequence lives in logical block t / block_size at
 * in-block slot t % block_size; block_table maps the logical block to a
 * physical one ([BM] s2, [KB] s3.3).  Writes K and V of kv head `hk` for
 * tokens [0, len) into Kc[t*D + d] and Vc[t*D + d]. */
void pao_gather(int D, int bs, int Hkv, int64_t block_stride, int dtype,
                const void *k_pool, const void *v_pool,
                const int32_t *table_row, int hk, int64_t len,
                double *Kc, double *Vc)
{
    (void)Hkv;
    for (int64_t t = 0; t < len; ++t) {
        int64_t blk = table_row[t / bs];
        int64_t slot = t % bs;
        int64_t base = blk * block_stride + (int64_t)hk * bs * D + slot * D;
        for (int d = 0; d < D; ++d) {
            Kc[t * D + d] = pao_element(k_pool, base + d, dtype);
            Vc[t * D + d] = pao_element(v_pool, base + d, dtype);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* textbook attention of one query over contiguous K/V                       */
/* ------------------------------------------------------------------------ */

/* o[d] = sum_t w_t V[t][d] / sum_t w_t with w_t = exp(x_t - max_u x_u) and
 * x_t = scale * sum_d q[d] K[t][d], over t in [0, len) only.  len == 0 gives
 * o = 0 (nothing to attend to). */
void pao_attention_contiguous(int64_t len, int D, const double *q,
                              const double *Kc, const double *Vc,
                              double scale, double *o)
{
    for (int d = 0; d < D; ++d)
        o[d] = 0.0;
    if (len == 0)
        return;
    double *x = (double *)malloc((size_t)len * sizeof(double));
    double m = -INFINITY;
    for (int64_t t = 0; t < len; ++t) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += q[d] * Kc[t * D + d];
        x[t] = scale * dot;
        if (x[t] > m)
            m = x[t];
    }
    double wsum = 0.0;
    for (int64_t t = 0; t < len; ++t) {
        double w = exp(x[t] - m);
        wsum += w;
        for (int d = 0; d < D; ++d)
            o[d] += w * Vc[t * D + d];
    }
    for (int d = 0; d < D; ++d)
        o[d] /= wsum;
    free(x);
}

/* ------------------------------------------------------------------------ */
/* decode attention over the paged cache                                     */
/* ------------------------------------------------------------------------ */

/* For every sequence b and query head h: out[b][h][:] = attention of
 * q[b][h][:] over the valid tokens [0, seq_lens[b]) of kv head
 * h / (H/Hkv), gathered through block_table[b][:].  A sequence that fails
 * validation gets out = 0 and its status bits in seq_err[b].
 * q is [B][H][D] of `dtype`; out is [B][H][D] double.  Returns the OR of
 * all status bits. */
int pao_attention_decode(int B, int H, int Hkv, int D, int bs, int MB,
                         int64_t NB, int64_t block_stride, int dtype,
                         const void *q, const void *k_pool,
                         const void *v_pool, const int32_t *block_table,
                         const int32_t *seq_lens, double scale, double *out,
                         int32_t *seq_err, int nthreads)
{
    int group = H / Hkv;
    int any = 0;
    for (int b = 0; b < B; ++b) {
        seq_err[b] = validate_sequence(seq_lens[b], bs, MB, NB,
                                       block_table + (int64_t)b * MB);
        any |= seq_err[b];
    }
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t u = 0; u < (int64_t)B * Hkv; ++u) {
        int b = (int)(u / Hkv);
        int hk = (int)(u % Hkv);
        int64_t len = seq_lens[b];
        if (seq_err[b]) {
            for (int h = hk * group; h < (hk + 1) * group; ++h)
                for (int d = 0; d < D; ++d)
                    out[((int64_t)b * H + h) * D + d] = 0.0;
            continue;
        }
        size_t n = (size_t)(len > 0 ? len : 1) * D;
        double *Kc = (double *)malloc(n * sizeof(double));
        double *Vc = (double *)malloc(n * sizeof(double));
        double *qd = (double *)malloc((size_t)D * sizeof(double));
        pao_gather(D, bs, Hkv, block_stride, dtype, k_pool, v_pool,
                   block_table + (int64_t)b * MB, hk, len, Kc, Vc);
        for (int h = hk * group; h < (hk + 1) * group; ++h) {
            for (int d = 0; d < D; ++d)
                qd[d] = pao_element(q, ((int64_t)b * H + h) * D + d, dtype);
            pao_attention_contiguous(len, D, qd, Kc, Vc, scale,
                                     out + ((int64_t)b * H + h) * D);
        }
        free(Kc);
        free(Vc);
        free(qd);
    }
    return any;
}

/* ------------------------------------------------------------------------ */
/* partial softmax sums over a token range, and their merge ([PG] s2.2)      */
/* ------------------------------------------------------------------------ */

/* For tokens t in [t_begin, min(t_end, len)) of each (b, h):
 *   m   = max_t x_t
 *   l   = sum_t exp(x_t - m)
 *   acc = sum_t exp(x_t - m) V[t][:]
 * (an empty range gives m = -inf, l = 0, acc = 0).  Merging the ranges of a
 * partition of [0, len) with pao_merge_partials gives the full attention.
 * m, l are [B][H]; acc is [B][H][D]. */
int pao_attention_partial(int B, int H, int Hkv, int D, int bs, int MB,
                          int64_t NB, int64_t block_stride, int dtype,
                          const void *q, const void *k_pool,
                          const void *v_pool, const int32_t *block_table,
                          const int32_t *seq_lens, double scale,
                          int64_t t_begin, int64_t t_end, double *m,
                          double *l, double *acc, int32_t *seq_err,
                          int nthreads)
{
    int group = H / Hkv;
    int any = 0;
    for (int b = 0; b < B; ++b) {
        seq_err[b] = validate_sequence(seq_lens[b], bs, MB, NB,
                                       block_table + (int64_t)b * MB);
        any |= seq_err[b];
    }
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t bh = 0; bh < (int64_t)B * H; ++bh) {
        int b = (int)(bh / H);
        int h = (int)(bh % H);
        int64_t len = seq_lens[b];
        int64_t lo = t_begin;
        int64_t hi = t_end < len ? t_end : len;
        m[bh] = -INFINITY;
        l[bh] = 0.0;
        for (int d = 0; d < D; ++d)
            acc[bh * D + d] = 0.0;
        if (seq_err[b] || hi <= lo)
            continue;
        int hk = h / group;
        double *Kc = (double *)malloc((size_t)len * D * sizeof(double));
        double *Vc = (double *)malloc((size_t)len * D * sizeof(double));
        pao_gather(D, bs, Hkv, block_stride, dtype, k_pool, v_pool,
                   block_table + (int64_t)b * MB, hk, len, Kc, Vc);
        double *x = (double *)malloc((size_t)(hi - lo) * sizeof(double));
        for (int64_t t = lo; t < hi; ++t) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += pao_element(q, bh * D + d, dtype) * Kc[t * D + d];
            x[t - lo] = scale * dot;
            if (x[t - lo] > m[bh])
                m[bh] = x[t - lo];
        }
        for (int64_t t = lo; t < hi; ++t) {
            double w = exp(x[t - lo] - m[bh]);
            l[bh] += w;
            for (int d = 0; d < D; ++d)
                acc[bh * D + d] += w * Vc[t * D + d];
        }
        free(x);
        free(Kc);
        free(Vc);
    }
    return any;
}

/* Merge n partial results (m_p, l_p, acc_p[D]) of one (b, h):
 *   M = max_p m_p,  o = sum_p acc_p exp(m_p - M) / sum_p l_p exp(m_p - M).
 * Partials with m_p = -inf are empty and contribute nothing; if all are
 * empty, o = 0. */
void pao_merge_partials(int n, int D, const double *m, const double *l,
                        const double *acc, double *o)
{
    double M = -INFINITY;
    for (int p = 0; p < n; ++p)
        if (m[p] > M)
            M = m[p];
    for (int d = 0; d < D; ++d)
        o[d] = 0.0;
    if (M == -INFINITY)
        return;
    double lsum = 0.0;
    for (int p = 0; p < n; ++p) {
        if (m[p] == -INFINITY)
            continue;
        double w = exp(m[p] - M);
        lsum += w * l[p];
        for (int d = 0; d < D; ++d)
            o[d] += w * acc[(int64_t)p * D + d];
    }
    for (int d = 0; d < D; ++d)
        o[d] /= lsum;
}

/* ------------------------------------------------------------------------ */
/* append: write one new token's K/V row per (sequence, kv head)             */
/* ------------------------------------------------------------------------ */

/* Token position pos = positions[b] (the length before the append) goes to
 * logical block pos / block_size, slot pos % block_size, so tokens inside a
 * block keep their logical order ([BM] s4.4) and the cache grows exactly as
 * the contiguous append of [BUG] s4.1 does.  k_new, v_new are [B][Hkv][D].
 * The copy is byte for byte.  A sequence whose position lies outside
 * [0, max_blocks_per_seq*block_size) or whose target table entry names no
 * pool block is skipped and flagged in seq_err[b].  Returns the OR of all
 * status bits. */
int pao_kv_append(int B, int Hkv, int D, int bs, int MB, int64_t NB,
                  int64_t block_stride, int dtype, const void *k_new,
                  const void *v_new, void *k_pool, void *v_pool,
                  const int32_t *block_table, const int32_t *positions,
                  int32_t *seq_err)
{
    int s = pao_dtype_bytes(dtype);
    int any = 0;
    for (int b = 0; b < B; ++b) {
        int64_t pos = positions[b];
        seq_err[b] = 0;
        if (pos < 0 || pos >= (int64_t)MB * bs) {
            seq_err[b] = PAO_SEQ_BAD_POS;
            any |= seq_err[b];
            continue;
        }
        int64_t blk = block_table[(int64_t)b * MB + pos / bs];
        if (blk < 0 || blk >= NB) {
            seq_err[b] = PAO_SEQ_BAD_BLOCK;
            any |= seq_err[b];
            continue;
        }
        for (int hk = 0; hk < Hkv; ++hk) {
            int64_t dst = blk * block_stride + (int64_t)hk * bs * D +
                          (pos % bs) * D;
            int64_t src = ((int64_t)b * Hkv + hk) * D;
            memcpy((char *)k_pool + dst * s, (const char *)k_new + src * s,
                   (size_t)D * s);
            memcpy((char *)v_pool + dst * s, (const char *)v_new + src * s,
                   (size_t)D * s);
        }
    }
    return any;
}

/* ------------------------------------------------------------------------ */
/* multi-token append: the prompt (prefill) write                            */
/* ------------------------------------------------------------------------ */

/* For every sequence b, tokens t < counts[b] of k_new/v_new [B][T][Hkv][D]
 * (a padded batch: rows t >= counts[b] are padding and are never written,
 * the valid-length rule of [BUG] s2.3-2.4) go to positions positions[b] + t,
 * each through the table exactly as the one-token append places it.
 * counts[b] outside [0, T] flags PAO_SEQ_BAD_LEN and skips the sequence;
 * positions[b] < 0 or positions[b] + counts[b] past the table row flags
 * PAO_SEQ_BAD_POS and skips it; a token whose target entry names no pool
 * block is skipped and flags PAO_SEQ_BAD_BLOCK (the other tokens are
 * written).  Returns the OR of all status bits. */
int pao_kv_append_tokens(int B, int T, int Hkv, int D, int bs, int MB, int64_t NB,
                         int64_t block_stride, int dtype, const void *k_new,
                         const void *v_new, void *k_pool, void *v_pool,
                         const int32_t *block_table, const int32_t *positions,
                         const int32_t *counts, int32_t *seq_err)
{
    int s = pao_dtype_bytes(dtype);
    int any = 0;
    for (int b = 0; b < B; ++b) {
        seq_err[b] = 0;
        int64_t n = counts[b];
        int64_t start = positions[b];
        if (n < 0 || n > T) {
            seq_err[b] = PAO_SEQ_BAD_LEN;
        } else if (start < 0 || start + n > (int64_t)MB * bs) {
            seq_err[b] = PAO_SEQ_BAD_POS;
        } else {
            for (int64_t t = 0; t < n; ++t) {
                int64_t pos = start + t;
                int64_t blk = block_table[(int64_t)b * MB + pos / bs];
                if (blk < 0 || blk >= NB) {
                    seq_err[b] |= PAO_SEQ_BAD_BLOCK;
                    continue;
                }
                for (int hk = 0; hk < Hkv; ++hk) {
                    int64_t dst = blk * block_stride + (int64_t)hk * bs * D + (pos % bs) * D;
                    int64_t src = (((int64_t)b * T + t) * Hkv + hk) * D;
                    memcpy((char *)k_pool + dst * s, (const char *)k_new + src * s, (size_t)D * s);
                    memcpy((char *)v_pool + dst * s, (const char *)v_new + src * s, (size_t)D * s);
                }
            }
        }
        any |= seq_err[b];
    }
    return any;
}

/* ------------------------------------------------------------------------ */
/* sliding-window decode ([BUG] s5.3: keep only the most recent tokens)      */
/* ------------------------------------------------------------------------ */

/* As pao_attention_decode, but each query attends only to the last `window`
 * valid tokens [max(0, L - window), L) of its sequence.  window must be
 * positive; a window of at least L gives the full attention. */
int pao_attention_decode_window(int B, int H, int Hkv, int D, int bs, int MB, int64_t NB,
                                int64_t block_stride, int dtype, const void *q,
                                const void *k_pool, const void *v_pool,
                                const int32_t *block_table, const int32_t *seq_lens,
                                double scale, int64_t window, double *out,
                                int32_t *seq_err, int nthreads)
{
    int group = H / Hkv;
    int any = 0;
    for (int b = 0; b < B; ++b) {
        seq_err[b] = validate_sequence(seq_lens[b], bs, MB, NB,
                                       block_table + (int64_t)b * MB);
        any |= seq_err[b];
    }
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t u = 0; u < (int64_t)B * Hkv; ++u) {
        int b = (int)(u / Hkv);
        int hk = (int)(u % Hkv);
        int64_t len = seq_lens[b];
        if (seq_err[b]) {
            for (int h = hk * group; h < (hk + 1) * group; ++h)
                for (int d = 0; d < D; ++d)
                    out[((int64_t)b * H + h) * D + d] = 0.0;
            continue;
        }
        int64_t first = len > window ? len - window : 0;
        size_t n = (size_t)(len > 0 ? len : 1) * D;
        double *Kc = (double *)malloc(n * sizeof(double));
        double *Vc = (double *)malloc(n * sizeof(double));
        double *qd = (double *)malloc((size_t)D * sizeof(double));
        pao_gather(D, bs, Hkv, block_stride, dtype, k_pool, v_pool,
                   block_table + (int64_t)b * MB, hk, len, Kc, Vc);
        for (int h = hk * group; h < (hk + 1) * group; ++h) {
            for (int d = 0; d < D; ++d)
                qd[d] = pao_element(q, ((int64_t)b * H + h) * D + d, dtype);
            pao_attention_contiguous(len - first, D, qd, Kc + first * D, Vc + first * D,
                                     scale, out + ((int64_t)b * H + h) * D);
        }
        free(Kc);
        free(Vc);
        free(qd);
    }
    return any;
}

/* ------------------------------------------------------------------------ */
/* int8 cache blocks with per-block scales                                   */
/* ------------------------------------------------------------------------ */

/* The pages name quantised cache blocks (int8 blocks in the semantic
 * compression scheme of [BM] s6.3, a "quantized" element size in the block
 * sizing rule of [BM] s3) but fix no scheme.  The reading used here, the
 * plainest one that matches "int8 blocks with per-block scales":
 *   - a cached K (or V) element is a signed code c in [-127, 127] that
 *     stands for the value c * s, where s is the fp32 scale of its
 *     (physical block, kv head) for K (or for V);
 *   - scales are stored as kv_scales[(blk*2 + 0)*Hkv + hk] (K) and
 *     kv_scales[(blk*2 + 1)*Hkv + hk] (V), set by whoever allocates the
 *     block;
 *   - writing a value x gives c = clamp(round_half_even(x / s), -127, 127),
 *     the division and the rounding taken in IEEE binary32 (the precision
 *     in which the GPU decides the integer); a NaN quotient gives 0.
 * Pools hold one byte per element, laid out like the 16-bit pools. */

signed char pao_quantize_i8(float x, float s)
{
    volatile float q = x / s;   /* binary32 division, round to nearest even */
    float r = rintf(q);         /* nearest integer, ties to even */
    if (r != r)
        return 0;
    if (r > 127.0f)
        r = 127.0f;
    if (r < -127.0f)
        r = -127.0f;
    return (signed char)r;
}

void pao_quantize_i8_array(const float *x, int64_t n, float s, signed char *codes)
{
    for (int64_t i = 0; i < n; ++i)
        codes[i] = pao_quantize_i8(x[i], s);
}

/* As pao_kv_append, but the new rows (k_new, v_new of `dtype`) are written
 * as int8 codes with the scale of their target (block, kv head). */
int pao_kv_append_i8(int B, int Hkv, int D, int bs, int MB, int64_t NB,
                     int64_t block_stride, int dtype, const void *k_new,
                     const void *v_new, signed char *k_pool, signed char *v_pool,
                     const float *kv_scales, const int32_t *block_table,
                     const int32_t *positions, int32_t *seq_err)
{
    int any = 0;
    for (int b = 0; b < B; ++b) {
        int64_t pos = positions[b];
        seq_err[b] = 0;
        if (pos < 0 || pos >= (int64_t)MB * bs) {
            seq_err[b] = PAO_SEQ_BAD_POS;
            any |= seq_err[b];
            continue;
        }
        int64_t blk = block_table[(int64_t)b * MB + pos / bs];
        if (blk < 0 || blk >= NB) {
            seq_err[b] = PAO_SEQ_BAD_BLOCK;
            any |= seq_err[b];
            continue;
        }
        for (int hk = 0; hk < Hkv; ++hk) {
            int64_t dst = blk * block_stride + (int64_t)hk * bs * D + (pos % bs) * D;
            int64_t src = ((int64_t)b * Hkv + hk) * D;
            float sk = kv_scales[(blk * 2 + 0) * Hkv + hk];
            float sv = kv_scales[(blk * 2 + 1) * Hkv + hk];
            for (int d = 0; d < D; ++d) {
                k_pool[dst + d] = pao_quantize_i8((float)pao_element(k_new, src + d, dtype), sk);
                v_pool[dst + d] = pao_quantize_i8((float)pao_element(v_new, src + d, dtype), sv);
            }
        }
    }
    return any;
}

/* Gather of an int8 cache: the values c * s of kv head hk, tokens [0, len). */
void pao_gather_i8(int D, int bs, int Hkv, int64_t block_stride,
                   const signed char *k_pool, const signed char *v_pool,
                   const float *kv_scales, const int32_t *table_row, int hk,
                   int64_t len, double *Kc, double *Vc)
{
    for (int64_t t = 0; t < len; ++t) {
        int64_t blk = table_row[t / bs];
        int64_t base = blk * block_stride + (int64_t)hk * bs * D + (t % bs) * D;
        double sk = kv_scales[(blk * 2 + 0) * Hkv + hk];
        double sv = kv_scales[(blk * 2 + 1) * Hkv + hk];
        for (int d = 0; d < D; ++d) {
            Kc[t * D + d] = (double)k_pool[base + d] * sk;
            Vc[t * D + d] = (double)v_pool[base + d] * sv;
        }
    }
}

/* Decode attention over an int8 cache: the textbook attention of
 * pao_attention_decode over the values the codes stand for.  q is [B][H][D]
 * of `dtype`. */
int pao_attention_decode_i8(int B, int H, int Hkv, int D, int bs, int MB,
                            int64_t NB, int64_t block_stride, int dtype,
                            const void *q, const signed char *k_pool,
                            const signed char *v_pool, const float *kv_scales,
                            const int32_t *block_table, const int32_t *seq_lens,
                            double scale, double *out, int32_t *seq_err,
                            int nthreads)
{
    int group = H / Hkv;
    int any = 0;
    for (int b = 0; b < B; ++b) {
        seq_err[b] = validate_sequence(seq_lens[b], bs, MB, NB,
                                       block_table + (int64_t)b * MB);
        any |= seq_err[b];
    }
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t u = 0; u < (int64_t)B * Hkv; ++u) {
        int b = (int)(u / Hkv);
        int hk = (int)(u % Hkv);
        int64_t len = seq_lens[b];
        if (seq_err[b]) {
            for (int h = hk * group; h < (hk + 1) * group; ++h)
                for (int d = 0; d < D; ++d)
                    out[((int64_t)b * H + h) * D + d] = 0.0;
            continue;
        }
        size_t n = (size_t)(len > 0 ? len : 1) * D;
        double *Kc = (double *)malloc(n * sizeof(double));
        double *Vc = (double *)malloc(n * sizeof(double));
        double *qd = (double *)malloc((size_t)D * sizeof(double));
        pao_gather_i8(D, bs, Hkv, block_stride, k_pool, v_pool, kv_scales,
                      block_table + (int64_t)b * MB, hk, len, Kc, Vc);
        for (int h = hk * group; h < (hk + 1) * group; ++h) {
            for (int d = 0; d < D; ++d)
                qd[d] = pao_element(q, ((int64_t)b * H + h) * D + d, dtype);
            pao_attention_contiguous(len, D, qd, Kc, Vc, scale,
                                     out + ((int64_t)b * H + h) * D);
        }
        free(Kc);
        free(Vc);
        free(qd);
    }
    return any;
}

/* ------------------------------------------------------------------------ */
/* fp8 (E4M3) cache blocks with per-block scales                             */
/* ------------------------------------------------------------------------ */

/* The second reading of "quantised blocks with per-block scales": a cached
 * element is an 8-bit floating-point code in the OCP FP8 E4M3 format (sign
 * bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds
 * the subnormals m * 2^-9; no infinities; 0x7F and 0xFF are NaN, so the
 * largest finite magnitude is 448) that stands for value(c) * s, with the
 * scales laid out as for int8.  Writing a value x gives the code of x / s
 * (the division in IEEE binary32) rounded to the nearest E4M3 value, ties to
 * the even code, magnitudes beyond 448 saturating to 448 (infinities
 * included); a NaN quotient gives the NaN code 0x7F. */

/* The value an E4M3 code stands for. */
double pao_e4m3_value(unsigned char c)
{
    int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);          /* subnormal: m/8 * 2^-6 */
    else
        v = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* The E4M3 code of a binary32 value: nearest, ties to even, saturating. */
unsigned char pao_e4m3_encode(float x)
{
    unsigned char sign;
    double a, r;
    int e2, E;
    if (x != x)
        return 0x7F;
    sign = signbit(x) ? 0x80 : 0x00;
    a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: multiples of 2^-9; 8 * 2^-9 is the smallest
         * normal, code 0x08, so the code is the multiple itself */
        r = nearbyint(a / ldexp(1.0, -9));   /* exact quotient; ties to even */
        return sign | (unsigned char)r;
    }
    frexp(a, &e2);          /* a in [2^(e2-1), 2^e2) */
    E = e2 - 1;             /* a in [2^E, 2^(E+1)), E in [-6, 8] */
    r = nearbyint(a / ldexp(1.0, E - 3));   /* in [8, 16]: 8 + mantissa */
    if (r == 16.0) {        /* rounded up to the next power of two */
        r = 8.0;
        E += 1;
    }
    return sign | (unsigned char)(((E + 7) << 3) | ((int)r - 8));
}

unsigned char pao_quantize_fp8(float x, float s)
{
    volatile float q = x / s;   /* binary32 division, round to nearest even */
    return pao_e4m3_encode(q);
}

void pao_quantize_fp8_array(const float *x, int64_t n, float s, unsigned char *codes)
{
    for (int64_t i = 0; i < n; ++i)
        codes[i] = pao_quantize_fp8(x[i], s);
}

/* As pao_kv_append_i8, with E4M3 codes. */
int pao_kv_append_fp8(int B, int Hkv, int D, int bs, int MB, int64_t NB,
                      int64_t block_stride, int dtype, const void *k_new,
                      const void *v_new, unsigned char *k_pool, unsigned char *v_pool,
                      const float *kv_scales, const int32_t *block_table,
                      const int32_t *positions, int32_t *seq_err)
{
    int any = 0;
    for (int b = 0; b < B; ++b) {
        int64_t pos = positions[b];
        seq_err[b] = 0;
        if (pos < 0 || pos >= (int64_t)MB * bs) {
            seq_err[b] = PAO_SEQ_BAD_POS;
            any |= seq_err[b];
            continue;
        }
        int64_t blk = block_table[(int64_t)b * MB + pos / bs];
        if (blk < 0 || blk >= NB) {
            seq_err[b] = PAO_SEQ_BAD_BLOCK;
            any |= seq_err[b];
            continue;
        }
        for (int hk = 0; hk < Hkv; ++hk) {
            int64_t dst = blk * block_stride + (int64_t)hk * bs * D + (pos % bs) * D;
            int64_t src = ((int64_t)b * Hkv + hk) * D;
            float sk = kv_scales[(blk * 2 + 0) * Hkv + hk];
            float sv = kv_scales[(blk * 2 + 1) * Hkv + hk];
            for (int d = 0; d < D; ++d) {
                k_pool[dst + d] = pao_quantize_fp8((float)pao_element(k_new, src + d, dtype), sk);
                v_pool[dst + d] = pao_quantize_fp8((float)pao_element(v_new, src + d, dtype), sv);
            }
        }
    }
    return any;
}

/* Gather of an fp8 cache: the values value(c) * s of kv head hk, tokens
 * [0, len). */
void pao_gather_fp8(int D, int bs, int Hkv, int64_t block_stride,
                    const unsigned char *k_pool, const unsigned char *v_pool,
                    const float *kv_scales, const int32_t *table_row, int hk,
                    int64_t len, double *Kc, double *Vc)
{
    for (int64_t t = 0; t < len; ++t) {
        int64_t blk = table_row[t / bs];
        int64_t base = blk * block_stride + (int64_t)hk * bs * D + (t % bs) * D;
        double sk = kv_scales[(blk * 2 + 0) * Hkv + hk];
        double sv = kv_scales[(blk * 2 + 1) * Hkv + hk];
        for (int d = 0; d < D; ++d) {
            Kc[t * D + d] = pao_e4m3_value(k_pool[base + d]) * sk;
            Vc[t * D + d] = pao_e4m3_value(v_pool[base + d]) * sv;
        }
    }
}

/* Decode attention over an fp8 cache: the textbook attention of
 * pao_attention_decode over the values the codes stand for. */
int pao_attention_decode_fp8(int B, int H, int Hkv, int D, int bs, int MB,
                             int64_t NB, int64_t block_stride, int dtype,
                             const void *q, const unsigned char *k_pool,
                             const unsigned char *v_pool, const float *kv_scales,
                             const int32_t *block_table, const int32_t *seq_lens,
                             double scale, double *out, int32_t *seq_err,
                             int nthreads)
{
    int group = H / Hkv;
    int any = 0;
    for (int b = 0; b < B; ++b) {
        seq_err[b] = validate_sequence(seq_lens[b], bs, MB, NB,
                                       block_table + (int64_t)b * MB);
        any |= seq_err[b];
    }
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t u = 0; u < (int64_t)B * Hkv; ++u) {
        int b = (int)(u / Hkv);
        int hk = (int)(u % Hkv);
        int64_t len = seq_lens[b];
        if (seq_err[b]) {
            for (int h = hk * group; h < (hk + 1) * group; ++h)
                for (int d = 0; d < D; ++d)
                    out[((int64_t)b * H + h) * D + d] = 0.0;
            continue;
        }
        size_t n = (size_t)(len > 0 ? len : 1) * D;
        double *Kc = (double *)malloc(n * sizeof(double));
        double *Vc = (double *)malloc(n * sizeof(double));
        double *qd = (double *)malloc((size_t)D * sizeof(double));
        pao_gather_fp8(D, bs, Hkv, block_stride, k_pool, v_pool, kv_scales,
                       block_table + (int64_t)b * MB, hk, len, Kc, Vc);
        for (int h = hk * group; h < (hk + 1) * group; ++h) {
            for (int d = 0; d < D; ++d)
                qd[d] = pao_element(q, ((int64_t)b * H + h) * D + d, dtype);
            pao_attention_contiguous(len, D, qd, Kc, Vc, scale,
                                     out + ((int64_t)b * H + h) * D);
        }
        free(Kc);
        free(Vc);
        free(qd);
    }
    return any;
}
