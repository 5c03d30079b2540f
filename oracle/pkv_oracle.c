/*
 * pkv_oracle.c -- float64 CPU oracle for paged-KV-cache decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no source, header, table or helper with the
 * CUDA library in paged_kv_cache_278_gb300/csrc.
 *
 * Every routine is the plain definition, written as loops, in float64:
 *
 *   - KV-cache size: 2 x L x H x D x S x bytes per element
 *       ("推理优化这件事，为什么值得反复复盘", sec. 4.1, the size formula and its
 *        32-layer / 32-head / 128-dim / 4096-token worked example);
 *       with a batch factor as in "LLM推理优化：从硬件瓶颈到KV Cache的工程实践",
 *       sec. 4.1.
 *   - Paged storage: the cache is cut into fixed-size blocks addressed through
 *     a per-request block table ("为什么“推理优化”不是锦上添花", sec. 3.2, scheme 1;
 *     "推理优化这件事，为什么值得反复复盘", sec. 4.2 and 4.3).
 *   - Append: the new token's K/V is written in place into its slot, nothing
 *     is reallocated or recomputed ("为什么“推理优化”不是锦上添花", sec. 3.1;
 *     "LLM推理优化：从硬件瓶颈到KV Cache的工程实践", sec. 4.3).
 *   - Decode: one step reads every cached K/V of the request, scores it
 *     against q, normalises with softmax and takes the weighted sum of V
 *     ("LLM推理优化：从硬件瓶颈到KV Cache的工程实践", sec. 4.2).
 *
 * Readings where the pages are silent (each one is listed in the design
 * notes of the repository):
 *   - cache layout [num_blocks][num_kv_heads][block_size][head_dim], fp16;
 *   - query head h reads kv head h / (num_q_heads / num_kv_heads);
 *   - context_lens[b] counts every cached token including the one appended
 *     in this step; block_tables entries past ceil(ctx/bs) are never read;
 *   - a negative slot in the slot mapping means "no token": it is skipped;
 *   - an empty context yields a zero output row;
 *   - split-context partitions and their log-sum-exp merge are not on the
 *     pages: they are the softmax identity exp(s - M) = exp(s - m_p) exp(m_p - M)
 *     applied to consecutive token ranges, so merge(partition(x)) must equal
 *     decode(x).
 *
 *   - Key-only int8 cache: the pages advise quantising K alone and keeping V
 *     in full precision ("推理优化这件事，为什么值得反复复盘", sec. 4.4; the
 *     int8 halving of cache memory also in "LLM推理优化：从硬件瓶颈到KV Cache的工程实践",
 *     sec. 4.2).  They give no scheme; the reading taken is symmetric int8 with
 *     one float32 scale per (token, kv head): s = max_d |k_d| / 127 and
 *     code_d = round-half-even(k_d / s), both in float32, so that the integer
 *     decision is taken in the precision the kernels use; an all-zero row has
 *     s = 0 and zero codes.  Attention then uses k_d = code_d * s exactly.
 *     The optional int8 K + V cache quantises value rows by the same scheme.
 *
 * fp16 values are carried as raw uint16 bit patterns and decoded to double by
 * the IEEE-754 binary16 definition (sign, 5-bit exponent with bias 15, 10-bit
 * fraction, subnormals, inf/nan) in oracle_half_to_double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* IEEE-754 binary16 -> double, from the format's definition. */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);              /* subnormal: frac * 2^-14 * 2^-10 */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + frac), expo - 25); /* (1 + frac/1024) * 2^(expo-15) */
    }
    return sign ? -v : v;
}

/* Elementwise binary16 -> double over an array. */
void oracle_halves_to_doubles(double *out, const uint16_t *in, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_half_to_double(in[i]);
}

/* Bytes of K plus V for L layers, H kv heads, head_dim D, S tokens, per batch
 * of `batch` requests, at `elem_bytes` bytes per element. */
int64_t oracle_kv_cache_bytes(int64_t batch, int64_t L, int64_t H, int64_t D, int64_t S,
                              int64_t elem_bytes)
{
    return 2 * batch * L * H * D * S * elem_bytes;
}

/* slot of a token at logical position pos of request b:
 *   block_tables[b][pos / bs] * bs + pos % bs;  pos < 0 gives slot -1. */
void oracle_slot_mapping(int64_t *slots, const int32_t *block_tables, const int32_t *positions,
                         int num_seqs, int max_blocks_per_seq, int block_size)
{
    for (int b = 0; b < num_seqs; ++b) {
        int pos = positions[b];
        if (pos < 0) {
            slots[b] = -1;
            continue;
        }
        int32_t phys = block_tables[(int64_t)b * max_blocks_per_seq + pos / block_size];
        slots[b] = (int64_t)phys * block_size + pos % block_size;
    }
}

static int64_t cache_index(int64_t phys, int j, int off, int d, int Hkv, int bs, int D)
{
    return ((phys * Hkv + j) * bs + off) * D + d;
}

/* In-place append: k_cache[slot] <- k_new[t], v_cache[slot] <- v_new[t] for
 * every kv head; a raw copy of the 16-bit patterns.  Negative slots skip. */
void oracle_append(uint16_t *k_cache, uint16_t *v_cache, const int64_t *slot_mapping,
                   const uint16_t *k_new, const uint16_t *v_new,
                   int num_tokens, int num_kv_heads, int head_dim, int block_size)
{
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        int64_t blk = slot / block_size;
        int off = (int)(slot % block_size);
        for (int j = 0; j < num_kv_heads; ++j) {
            for (int d = 0; d < head_dim; ++d) {
                int64_t src = ((int64_t)t * num_kv_heads + j) * head_dim + d;
                int64_t dst = cache_index(blk, j, off, d, num_kv_heads, block_size, head_dim);
                k_cache[dst] = k_new[src];
                v_cache[dst] = v_new[src];
            }
        }
    }
}

/* Copy-on-write of whole blocks: k_cache[dst[i]] <- k_cache[src[i]] and the same for V,
 * every kv head and slot of the block, as raw 16-bit patterns (copying a shared page
 * before a request appends into it; the pages share prefix blocks between requests:
 * "推理优化这件事，为什么值得反复复盘", sec. 4.2). */
void oracle_copy_blocks(uint16_t *k_cache, uint16_t *v_cache, const int32_t *src, const int32_t *dst, int n,
                        int num_kv_heads, int head_dim, int block_size)
{
    int64_t per_block = (int64_t)num_kv_heads * block_size * head_dim;
    for (int i = 0; i < n; ++i) {
        for (int64_t e = 0; e < per_block; ++e) {
            k_cache[(int64_t)dst[i] * per_block + e] = k_cache[(int64_t)src[i] * per_block + e];
            v_cache[(int64_t)dst[i] * per_block + e] = v_cache[(int64_t)src[i] * per_block + e];
        }
    }
}

/* Whole blocks from one pool to another (swap out / swap in, "LLM推理优化：从硬件瓶颈到KV Cache的工程实践",
 * sec. 3.2: pages move in and out at page granularity): dst_k[dst[i]] <- src_k[src[i]] and the
 * same for V, raw 16-bit patterns; both pools [blocks][num_kv_heads][block_size][head_dim]. */
void oracle_copy_blocks_between(uint16_t *dst_k, uint16_t *dst_v, const uint16_t *src_k, const uint16_t *src_v,
                                const int32_t *src, const int32_t *dst, int n, int num_kv_heads, int head_dim,
                                int block_size)
{
    int64_t elems = (int64_t)num_kv_heads * block_size * head_dim;
    for (int i = 0; i < n; ++i) {
        for (int64_t e = 0; e < elems; ++e) {
            dst_k[(int64_t)dst[i] * elems + e] = src_k[(int64_t)src[i] * elems + e];
            dst_v[(int64_t)dst[i] * elems + e] = src_v[(int64_t)src[i] * elems + e];
        }
    }
}

/* scores s_p = scale * q . K[p] for p in [p0, p1) of request b, kv head j. */
static void scores_range(double *s, const uint16_t *q_row, const uint16_t *k_cache,
                         const int32_t *bt_row, int p0, int p1, int j,
                         int Hkv, int D, int bs, double scale)
{
    for (int p = p0; p < p1; ++p) {
        int64_t phys = bt_row[p / bs];
        int off = p % bs;
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += oracle_half_to_double(q_row[d]) *
                   oracle_half_to_double(k_cache[cache_index(phys, j, off, d, Hkv, bs, D)]);
        s[p - p0] = scale * dot;
    }
}

/* Softmax-weighted sum of V over [p0, p1) given the scores s: writes
 * o = sum_p exp(s_p - m) v_p / l with m = max s_p, l = sum_p exp(s_p - m),
 * and returns m and l. */
static void softmax_weighted_sum(double *o, double *m_out, double *l_out, const double *s,
                                 const uint16_t *v_cache, const int32_t *bt_row,
                                 int p0, int p1, int j, int Hkv, int D, int bs)
{
    double m = -INFINITY;
    for (int p = p0; p < p1; ++p)
        if (s[p - p0] > m)
            m = s[p - p0];
    double l = 0.0;
    for (int d = 0; d < D; ++d)
        o[d] = 0.0;
    for (int p = p0; p < p1; ++p) {
        double w = exp(s[p - p0] - m);
        int64_t phys = bt_row[p / bs];
        int off = p % bs;
        l += w;
        for (int d = 0; d < D; ++d)
            o[d] += w * oracle_half_to_double(v_cache[cache_index(phys, j, off, d, Hkv, bs, D)]);
    }
    for (int d = 0; d < D; ++d)
        o[d] /= l;
    *m_out = m;
    *l_out = l;
}

/* out[b][h][:] = softmax(scale * q[b][h] . K^T) V over the ctx_b cached
 * positions of request b, gathered through its block table.  out is float64
 * [num_seqs][num_q_heads][head_dim]; an empty context gives zeros. */
void oracle_decode(double *out, const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                   const int32_t *block_tables, const int32_t *context_lens,
                   int num_seqs, int max_blocks_per_seq, int num_q_heads, int num_kv_heads,
                   int head_dim, int block_size, double scale)
{
    int group = num_q_heads / num_kv_heads;
    for (int b = 0; b < num_seqs; ++b) {
        int ctx = context_lens[b];
        const int32_t *bt_row = block_tables + (int64_t)b * max_blocks_per_seq;
        double *s = (double *)malloc(sizeof(double) * (ctx > 0 ? ctx : 1));
        for (int h = 0; h < num_q_heads; ++h) {
            int j = h / group;
            double *o = out + ((int64_t)b * num_q_heads + h) * head_dim;
            if (ctx <= 0) {
                for (int d = 0; d < head_dim; ++d)
                    o[d] = 0.0;
                continue;
            }
            const uint16_t *q_row = q + ((int64_t)b * num_q_heads + h) * head_dim;
            double m, l;
            scores_range(s, q_row, k_cache, bt_row, 0, ctx, j, num_kv_heads, head_dim,
                         block_size, scale);
            softmax_weighted_sum(o, &m, &l, s, v_cache, bt_row, 0, ctx, j, num_kv_heads,
                                 head_dim, block_size);
        }
        free(s);
    }
}

/* Symmetric int8 quantisation of one K row of D binary16 values, in float32:
 * scale = max |k| / 127, code_d = round-half-even(k_d / scale) in [-127, 127].
 * The float32 division and rintf (round to nearest even in the default mode)
 * are the IEEE-754 operations; an all-zero row gives scale 0 and zero codes. */
void oracle_quantize_k_row(int8_t *codes, float *scale, const uint16_t *k_row, int D)
{
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) {
        float a = fabsf((float)oracle_half_to_double(k_row[d]));
        if (a > amax)
            amax = a;
    }
    float s = amax / 127.0f;
    *scale = s;
    for (int d = 0; d < D; ++d) {
        if (s == 0.0f) {
            codes[d] = 0;
            continue;
        }
        float r = rintf((float)oracle_half_to_double(k_row[d]) / s);
        if (r > 127.0f)
            r = 127.0f;
        if (r < -127.0f)
            r = -127.0f;
        codes[d] = (int8_t)r;
    }
}

/* Append into the K-int8 / V-fp16 cache: for each token t with a slot >= 0 and
 * each kv head j, k_codes[slot][j] and k_scale[slot][j] receive the quantised
 * K row and v_cache[slot][j] the raw V row.  Layouts: k_codes int8 and v_cache
 * fp16 [num_blocks][num_kv_heads][block_size][head_dim], k_scale float32
 * [num_blocks][num_kv_heads][block_size]. */
void oracle_append_quant_k(int8_t *k_codes, float *k_scale, uint16_t *v_cache, const int64_t *slot_mapping,
                           const uint16_t *k_new, const uint16_t *v_new, int num_tokens,
                           int num_kv_heads, int head_dim, int block_size)
{
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        int64_t blk = slot / block_size;
        int off = (int)(slot % block_size);
        for (int j = 0; j < num_kv_heads; ++j) {
            int64_t row = (blk * num_kv_heads + j) * block_size + off;
            const uint16_t *src = k_new + ((int64_t)t * num_kv_heads + j) * head_dim;
            oracle_quantize_k_row(k_codes + row * head_dim, k_scale + row, src, head_dim);
            for (int d = 0; d < head_dim; ++d)
                v_cache[row * head_dim + d] = v_new[((int64_t)t * num_kv_heads + j) * head_dim + d];
        }
    }
}

/* Decode attention over the K-int8 / V-fp16 cache: the plain definition with
 * every key dequantised, k_d = code_d * scale (float64), and V as stored.  Same
 * shapes, table and context rules as oracle_decode. */
void oracle_decode_quant_k(double *out, const uint16_t *q, const int8_t *k_codes, const float *k_scale,
                           const uint16_t *v_cache, const int32_t *block_tables, const int32_t *context_lens,
                           int num_seqs, int max_blocks_per_seq, int num_q_heads, int num_kv_heads,
                           int head_dim, int block_size, double scale)
{
    int group = num_q_heads / num_kv_heads;
    for (int b = 0; b < num_seqs; ++b) {
        int ctx = context_lens[b];
        const int32_t *bt_row = block_tables + (int64_t)b * max_blocks_per_seq;
        double *s = (double *)malloc(sizeof(double) * (ctx > 0 ? ctx : 1));
        for (int h = 0; h < num_q_heads; ++h) {
            int kvh = h / group;
            double *o = out + ((int64_t)b * num_q_heads + h) * head_dim;
            if (ctx <= 0) {
                for (int d = 0; d < head_dim; ++d)
                    o[d] = 0.0;
                continue;
            }
            const uint16_t *q_row = q + ((int64_t)b * num_q_heads + h) * head_dim;
            for (int p = 0; p < ctx; ++p) {
                int64_t row = ((int64_t)bt_row[p / block_size] * num_kv_heads + kvh) * block_size + p % block_size;
                double dot = 0.0;
                for (int d = 0; d < head_dim; ++d)
                    dot += oracle_half_to_double(q_row[d]) * ((double)k_codes[row * head_dim + d] * k_scale[row]);
                s[p] = scale * dot;
            }
            double m, l;
            softmax_weighted_sum(o, &m, &l, s, v_cache, bt_row, 0, ctx, kvh, num_kv_heads, head_dim,
                                 block_size);
        }
        free(s);
    }
}

/* Several new tokens per request (a verified draft or a prefill chunk): request b
 * owns query rows query_start[b] .. query_start[b + 1] - 1 of q and out
 * ([total_q][num_q_heads][head_dim]); its n_b = query_start[b + 1] - query_start[b]
 * new tokens are already appended, so context_lens[b] counts them, and query row i
 * sits at logical position ctx_b - n_b + i.  Causally, it attends to positions
 * 0 .. ctx_b - n_b + i: the plain decode definition over that prefix of the
 * request's cache.  (The pages list chunked prefill and speculative decoding as
 * decode-side techniques over the same cache: "LLM推理优化：从硬件瓶颈到KV Cache的工程实践",
 * sec. 3.2.) */
void oracle_decode_multi(double *out, const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                         const int32_t *block_tables, const int32_t *context_lens, const int32_t *query_start,
                         int num_seqs, int max_blocks_per_seq, int num_q_heads, int num_kv_heads,
                         int head_dim, int block_size, double scale)
{
    int group = num_q_heads / num_kv_heads;
    for (int b = 0; b < num_seqs; ++b) {
        int n = query_start[b + 1] - query_start[b];
        int ctx = context_lens[b];
        const int32_t *bt_row = block_tables + (int64_t)b * max_blocks_per_seq;
        double *s = (double *)malloc(sizeof(double) * (ctx > 0 ? ctx : 1));
        for (int i = 0; i < n; ++i) {
            int visible = ctx - n + i + 1;
            int64_t t = query_start[b] + i;
            for (int h = 0; h < num_q_heads; ++h) {
                int kvh = h / group;
                double *o = out + (t * num_q_heads + h) * head_dim;
                const uint16_t *q_row = q + (t * num_q_heads + h) * head_dim;
                double m, l;
                scores_range(s, q_row, k_cache, bt_row, 0, visible, kvh, num_kv_heads, head_dim,
                             block_size, scale);
                softmax_weighted_sum(o, &m, &l, s, v_cache, bt_row, 0, visible, kvh, num_kv_heads,
                                     head_dim, block_size);
            }
        }
        free(s);
    }
}

/* Append into the int8 K + V cache: both rows quantised by oracle_quantize_k_row
 * (the same symmetric per-row scheme for values), codes and scales stored at the
 * slot.  Layouts as oracle_append_quant_k, with v_codes / v_scale like the keys'. */
void oracle_append_quant_kv(int8_t *k_codes, float *k_scale, int8_t *v_codes, float *v_scale,
                            const int64_t *slot_mapping, const uint16_t *k_new, const uint16_t *v_new,
                            int num_tokens, int num_kv_heads, int head_dim, int block_size)
{
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        int64_t blk = slot / block_size;
        int off = (int)(slot % block_size);
        for (int j = 0; j < num_kv_heads; ++j) {
            int64_t row = blk * num_kv_heads * block_size + (int64_t)j * block_size + off;
            int64_t src = ((int64_t)t * num_kv_heads + j) * head_dim;
            oracle_quantize_k_row(k_codes + row * head_dim, k_scale + row, k_new + src, head_dim);
            oracle_quantize_k_row(v_codes + row * head_dim, v_scale + row, v_new + src, head_dim);
        }
    }
}

/* Decode attention over the int8 K + V cache: keys and values dequantised,
 * code * scale (float64), then the plain definition.  Same shapes and rules as
 * oracle_decode. */
void oracle_decode_quant_kv(double *out, const uint16_t *q, const int8_t *k_codes, const float *k_scale,
                            const int8_t *v_codes, const float *v_scale, const int32_t *block_tables,
                            const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                            int num_q_heads, int num_kv_heads, int head_dim, int block_size, double scale)
{
    int group = num_q_heads / num_kv_heads;
    for (int b = 0; b < num_seqs; ++b) {
        int ctx = context_lens[b];
        const int32_t *bt_row = block_tables + (int64_t)b * max_blocks_per_seq;
        double *s = (double *)malloc(sizeof(double) * (ctx > 0 ? ctx : 1));
        for (int h = 0; h < num_q_heads; ++h) {
            int head_kv = h / group;
            double *o = out + ((int64_t)b * num_q_heads + h) * head_dim;
            for (int d = 0; d < head_dim; ++d)
                o[d] = 0.0;
            if (ctx <= 0)
                continue;
            const uint16_t *q_row = q + ((int64_t)b * num_q_heads + h) * head_dim;
            double m = -INFINITY;
            for (int p = 0; p < ctx; ++p) {
                int64_t row = ((int64_t)bt_row[p / block_size] * num_kv_heads + head_kv) * block_size + p % block_size;
                double dot = 0.0;
                for (int d = 0; d < head_dim; ++d)
                    dot += oracle_half_to_double(q_row[d]) * ((double)k_scale[row] * k_codes[row * head_dim + d]);
                s[p] = scale * dot;
                if (s[p] > m)
                    m = s[p];
            }
            double l = 0.0;
            for (int p = 0; p < ctx; ++p) {
                int64_t row = ((int64_t)bt_row[p / block_size] * num_kv_heads + head_kv) * block_size + p % block_size;
                double w = exp(s[p] - m);
                l = l + w;
                for (int d = 0; d < head_dim; ++d)
                    o[d] += w * ((double)v_codes[row * head_dim + d] * v_scale[row]);
            }
            for (int d = 0; d < head_dim; ++d)
                o[d] /= l;
        }
        free(s);
    }
}

/* Split-context partial results.  Partition p of request b covers the
 * positions [p * partition_size, min(ctx_b, (p + 1) * partition_size)).  For
 * each such partition and q head: m = max score, l = sum exp(s - m),
 * o = sum exp(s - m) v / l.  Layouts: o [num_seqs][num_q_heads][max_partitions][head_dim],
 * m and l [num_seqs][num_q_heads][max_partitions].  Partitions past the end of
 * the context get m = -inf, l = 0, o = 0. */
void oracle_decode_partition(double *o_part, double *m_part, double *l_part,
                             const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                             const int32_t *block_tables, const int32_t *context_lens,
                             int num_seqs, int max_blocks_per_seq, int num_q_heads,
                             int num_kv_heads, int head_dim, int block_size, double scale,
                             int partition_size, int max_partitions)
{
    int group = num_q_heads / num_kv_heads;
    double *s = (double *)malloc(sizeof(double) * partition_size);
    for (int b = 0; b < num_seqs; ++b) {
        int ctx = context_lens[b];
        const int32_t *bt_row = block_tables + (int64_t)b * max_blocks_per_seq;
        for (int h = 0; h < num_q_heads; ++h) {
            int j = h / group;
            const uint16_t *q_row = q + ((int64_t)b * num_q_heads + h) * head_dim;
            for (int p = 0; p < max_partitions; ++p) {
                int64_t row = ((int64_t)b * num_q_heads + h) * max_partitions + p;
                double *o = o_part + row * head_dim;
                int p0 = p * partition_size;
                int p1 = p0 + partition_size < ctx ? p0 + partition_size : ctx;
                if (p0 >= p1) {
                    for (int d = 0; d < head_dim; ++d)
                        o[d] = 0.0;
                    m_part[row] = -INFINITY;
                    l_part[row] = 0.0;
                    continue;
                }
                scores_range(s, q_row, k_cache, bt_row, p0, p1, j, num_kv_heads, head_dim,
                             block_size, scale);
                softmax_weighted_sum(o, &m_part[row], &l_part[row], s, v_cache, bt_row, p0, p1,
                                     j, num_kv_heads, head_dim, block_size);
            }
        }
    }
    free(s);
}

/* Log-sum-exp merge of the partitions of each (request, q head):
 *   M = max_p m_p,  w_p = l_p exp(m_p - M),  out = sum_p w_p o_p / sum_p w_p
 * over the ceil(ctx_b / partition_size) partitions; an empty context gives
 * zeros. */
void oracle_merge(double *out, const double *o_part, const double *m_part, const double *l_part,
                  const int32_t *context_lens, int num_seqs, int num_q_heads, int head_dim,
                  int partition_size, int max_partitions)
{
    for (int b = 0; b < num_seqs; ++b) {
        int ctx = context_lens[b];
        int np = ctx > 0 ? (ctx + partition_size - 1) / partition_size : 0;
        for (int h = 0; h < num_q_heads; ++h) {
            double *o = out + ((int64_t)b * num_q_heads + h) * head_dim;
            int64_t row0 = ((int64_t)b * num_q_heads + h) * max_partitions;
            for (int d = 0; d < head_dim; ++d)
                o[d] = 0.0;
            if (np == 0)
                continue;
            double M = -INFINITY;
            for (int p = 0; p < np; ++p)
                if (m_part[row0 + p] > M)
                    M = m_part[row0 + p];
            double wsum = 0.0;
            for (int p = 0; p < np; ++p) {
                double w = l_part[row0 + p] * exp(m_part[row0 + p] - M);
                wsum += w;
                for (int d = 0; d < head_dim; ++d)
                    o[d] += w * o_part[(row0 + p) * head_dim + d];
            }
            for (int d = 0; d < head_dim; ++d)
                o[d] /= wsum;
        }
    }
}

/*
 * fp8 K + V cache.  The pages compress the cache to 8 bits per element (int8 in
 * "推理优化这件事，为什么值得反复复盘", sec. 4.4, and "LLM推理优化：从硬件瓶颈到KV Cache的工程实践",
 * sec. 4.2) and name FP8 as the 8-bit number format the hardware handles natively
 * ("LLM推理优化：从硬件瓶颈到KV Cache的工程实践", sec. 2).  The reading taken for an 8-bit
 * floating-point cache: every element is an E4M3 code (1 sign bit, 4 exponent bits
 * with bias 7, 3 fraction bits; exponent field 0 holds subnormals; S.1111.111 is
 * NaN; no infinities; largest finite magnitude 448), with one float32 scale per
 * (token, kv head) row as for int8: s = max_d |x_d| / 448 and code_d = the E4M3
 * value nearest to x_d / s (ties to the even code), both in float32, clamped to
 * +-448; an all-zero row has s = 0 and zero codes.  Attention then uses
 * x_d = value(code_d) * s exactly.
 */

/* Value of one E4M3 code, from the format's definition. */
double oracle_e4m3_to_double(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int expo = (c >> 3) & 0xf;
    int frac = c & 0x7;
    double v;
    if (expo == 0xf && frac == 0x7)
        v = NAN;
    else if (expo == 0)
        v = ldexp((double)frac, -9);                 /* subnormal: frac/8 * 2^(1-7) */
    else
        v = ldexp((double)(8 + frac), expo - 10);    /* (1 + frac/8) * 2^(expo-7) */
    return sign ? -v : v;
}

/* The E4M3 code whose value is nearest to y (ties: the code with an even fraction),
 * |y| clamped to 448 first; the sign bit is y's, as in any IEEE rounding (a negative y
 * that rounds to zero gives -0, code 0x80).  The finite non-negative codes 0 .. 0x7E
 * have increasing values, so "even fraction" is "even code" and the nearest code is
 * one of the two neighbours of |y| in that sorted table, found by bisection. */
static double e4m3_table[0x7f];                /* value of codes 0 .. 0x7E, filled once */
static int e4m3_table_ready;

static double e4m3_value(int c)
{
    if (!e4m3_table_ready) {
        for (int i = 0; i < 0x7f; ++i)
            e4m3_table[i] = oracle_e4m3_to_double((uint8_t)i);
        e4m3_table_ready = 1;
    }
    return e4m3_table[c];
}

uint8_t oracle_e4m3_from_float(float y)
{
    double a = fabs((double)y);
    if (a > 448.0)
        a = 448.0;
    int lo = 0, hi = 0x7e;                     /* invariant: value(lo) <= a */
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (e4m3_value(mid) <= a)
            lo = mid;
        else
            hi = mid - 1;
    }
    int best = lo;
    if (lo < 0x7e) {
        double below = a - e4m3_value(lo);
        double above = e4m3_value(lo + 1) - a;
        if (above < below || (above == below && ((lo + 1) & 1) == 0))
            best = lo + 1;
    }
    return (uint8_t)(signbit(y) ? (best | 0x80) : best);
}

/* One row of D binary16 values -> E4M3 codes and the row's float32 scale. */
void oracle_quantize_fp8_row(uint8_t *codes, float *scale, const uint16_t *row, int D)
{
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) {
        float a = fabsf((float)oracle_half_to_double(row[d]));
        if (a > amax)
            amax = a;
    }
    float s = amax / 448.0f;
    *scale = s;
    for (int d = 0; d < D; ++d)
        codes[d] = s == 0.0f ? 0 : oracle_e4m3_from_float((float)oracle_half_to_double(row[d]) / s);
}

/* Append into the fp8 K + V cache: both rows quantised by oracle_quantize_fp8_row and
 * stored with their scales at the slot.  Layouts: codes uint8
 * [num_blocks][num_kv_heads][block_size][head_dim], scales float32
 * [num_blocks][num_kv_heads][block_size].  Negative slots skip. */
void oracle_append_fp8_kv(uint8_t *k_codes, float *k_scale, uint8_t *v_codes, float *v_scale,
                          const int64_t *slot_mapping, const uint16_t *k_new, const uint16_t *v_new,
                          int num_tokens, int num_kv_heads, int head_dim, int block_size)
{
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        int64_t blk = slot / block_size;
        int off = (int)(slot % block_size);
        for (int j = 0; j < num_kv_heads; ++j) {
            int64_t row = (int64_t)(blk * num_kv_heads + j) * block_size + off;
            int64_t src = ((int64_t)t * num_kv_heads + j) * head_dim;
            oracle_quantize_fp8_row(k_codes + row * head_dim, k_scale + row, k_new + src, head_dim);
            oracle_quantize_fp8_row(v_codes + row * head_dim, v_scale + row, v_new + src, head_dim);
        }
    }
}

/* Decode attention over the fp8 K + V cache: every key and value dequantised,
 * value(code) * scale in float64, then the plain definition (scores, softmax,
 * weighted sum).  Same shapes, table and context rules as oracle_decode. */
void oracle_decode_fp8_kv(double *out, const uint16_t *q, const uint8_t *k_codes, const float *k_scale,
                          const uint8_t *v_codes, const float *v_scale, const int32_t *block_tables,
                          const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                          int num_q_heads, int num_kv_heads, int head_dim, int block_size, double scale)
{
    int group = num_q_heads / num_kv_heads;
    for (int b = 0; b < num_seqs; ++b) {
        int ctx = context_lens[b];
        const int32_t *bt_row = block_tables + (int64_t)b * max_blocks_per_seq;
        double *s = (double *)malloc(sizeof(double) * (ctx > 0 ? ctx : 1));
        for (int h = 0; h < num_q_heads; ++h) {
            int kvh = h / group;
            double *o = out + ((int64_t)b * num_q_heads + h) * head_dim;
            for (int d = 0; d < head_dim; ++d)
                o[d] = 0.0;
            if (ctx <= 0)
                continue;
            const uint16_t *q_row = q + ((int64_t)b * num_q_heads + h) * head_dim;
            double m = -INFINITY;
            for (int p = 0; p < ctx; ++p) {
                int64_t row = ((int64_t)bt_row[p / block_size] * num_kv_heads + kvh) * block_size + p % block_size;
                double dot = 0.0;
                for (int d = 0; d < head_dim; ++d)
                    dot += oracle_half_to_double(q_row[d]) *
                           (oracle_e4m3_to_double(k_codes[row * head_dim + d]) * k_scale[row]);
                s[p] = scale * dot;
                if (s[p] > m)
                    m = s[p];
            }
            double l = 0.0;
            for (int p = 0; p < ctx; ++p) {
                int64_t row = ((int64_t)bt_row[p / block_size] * num_kv_heads + kvh) * block_size + p % block_size;
                double w = exp(s[p] - m);
                l += w;
                for (int d = 0; d < head_dim; ++d)
                    o[d] += w * (oracle_e4m3_to_double(v_codes[row * head_dim + d]) * v_scale[row]);
            }
            for (int d = 0; d < head_dim; ++d)
                o[d] /= l;
        }
        free(s);
    }
}
