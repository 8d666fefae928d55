/*
 * Oracle for the paged decode path -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of what the path computes.  Only the
 * tests, the smoke check and the benchmark's CPU-baseline leg may load it;
 * the library under test never does.  It shares no code, header or table
 * with the CUDA path.
 *
 * Sources (page title, then section / equation):
 *   - "vLLM & PagedAttention: Efficient Memory Management for LLM Serving",
 *     §I attention equation: a_ij = exp(q_i.k_j/sqrt d) / sum_{t<=i} exp(q_i.k_t/sqrt d),
 *     o_i = sum_j a_ij v_j.
 *   - same page, §III blockwise equation: the same sum grouped by blocks
 *     K_j = (k_{(j-1)B+1} .. k_{jB}); blocks need not be adjacent in memory.
 *   - "PagedAttention and vLLM, annotated" §4.1: the paged result is identical
 *     to attending over one contiguous array; §4.2: the block table maps a
 *     logical block to a physical block.
 *   - "vLLM & PagedAttention" §X: fused reshape + block write (new K/V written
 *     at block-table positions) and fused block copy (copy-on-write copies of
 *     scattered blocks).
 *   - same page, §VIII: swapping copies an evicted group's blocks to a CPU
 *     pool and back (block copies between two pools).
 *
 * Layouts (the pages leave the "read-optimized layout" open; this is the
 * reading the whole build uses):
 *   key/value        [T][Hkv][d]            16-bit (fp16 or bf16 bit patterns)
 *   key/value cache  [NB][Hkv][B][d]        16-bit
 *   query            [S][H][d]              16-bit
 *   block_tables     [S][max_blocks]        int32 physical block ids
 *   context_lens     [S]                    int32, includes the decode token
 *   out              [S][H][d]              double
 * The query head h reads kv head g = h / (H / Hkv) (contiguous grouping).
 *
 * Every function returns 0 on success, a negative code on bad input:
 *   -1 bad size argument, -2 index out of range.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- 16-bit float decoding, from the formats' definitions -------------- */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double half_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                   /* subnormal: f * 2^-14 * 2^-10 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 1024), e - 15 - 10);  /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE 754 binary32. */
static double bfloat16_bits_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float x;
    memcpy(&x, &u, sizeof x);
    return (double)x;
}

static double to_double(uint16_t bits, int is_bf16)
{
    return is_bf16 ? bfloat16_bits_to_double(bits) : half_bits_to_double(bits);
}

/* Exposed so that the decoding can be pinned against the standard library
 * conversions on its own. */
void oracle_decode16(const uint16_t *bits, int64_t n, int is_bf16, double *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = to_double(bits[i], is_bf16);
}

/* ---- block-table gather ------------------------------------------------- */

/* Token t (0-based) of a sequence lives in logical block t / B at offset
 * t % B; the block table row maps the logical block to a physical one. */
static void locate(const int32_t *table_row, int B, int64_t t, int32_t *phys, int32_t *off)
{
    *phys = table_row[t / B];
    *off = (int32_t)(t % B);
}

/* The (physical block, offset) of each of the first ctx tokens. */
int oracle_locate_tokens(const int32_t *table_row, int B, int64_t ctx,
                         int32_t *phys, int32_t *off)
{
    if (B <= 0 || ctx < 0)
        return -1;
    for (int64_t t = 0; t < ctx; t++)
        locate(table_row, B, t, &phys[t], &off[t]);
    return 0;
}

/* ---- slot-mapped cache write ("fused reshape + block write") ----------- */

/* For each token t with slot s = slots[t] >= 0: block s / B, offset s % B;
 * copy the raw 16-bit patterns of key[t][h][:] and value[t][h][:] there.
 * A negative slot marks a padding token and is skipped. */
int oracle_cache_write(const uint16_t *key, const uint16_t *value,
                       uint16_t *key_cache, uint16_t *value_cache,
                       const int64_t *slots, int T, int Hkv, int d, int B, int NB)
{
    if (T < 0 || Hkv <= 0 || d <= 0 || B <= 0 || NB < 0)
        return -1;
    for (int t = 0; t < T; t++) {
        int64_t s = slots[t];
        if (s < 0)
            continue;
        if (s >= (int64_t)NB * B)
            return -2;
        int64_t blk = s / B, off = s % B;
        for (int h = 0; h < Hkv; h++) {
            for (int i = 0; i < d; i++) {
                int64_t src = ((int64_t)t * Hkv + h) * d + i;
                int64_t dst = ((blk * Hkv + h) * B + off) * d + i;
                key_cache[dst] = key[src];
                value_cache[dst] = value[src];
            }
        }
    }
    return 0;
}

/* ---- block copy ("fused block copy", copy-on-write) -------------------- */

/* For each pair (src, dst): the whole dst block := the whole src block.
 * block_elems = Hkv * B * d 16-bit elements. */
int oracle_copy_blocks(uint16_t *cache, const int32_t *pairs, int n,
                       int64_t block_elems, int NB)
{
    if (n < 0 || block_elems <= 0 || NB < 0)
        return -1;
    for (int p = 0; p < n; p++) {
        int32_t src = pairs[2 * p], dst = pairs[2 * p + 1];
        if (src < 0 || src >= NB || dst < 0 || dst >= NB)
            return -2;
        for (int64_t i = 0; i < block_elems; i++)
            cache[(int64_t)dst * block_elems + i] = cache[(int64_t)src * block_elems + i];
    }
    return 0;
}

/* Copies between two pools (swapping, "vLLM & PagedAttention" §VIII): for
 * each pair, block dst_pool[pairs[i][1]] := src_pool[pairs[i][0]]; every
 * other block of dst_pool is untouched. */
int oracle_copy_blocks_between(uint16_t *dst_pool, const uint16_t *src_pool, const int32_t *pairs, int n,
                               int64_t block_elems, int src_blocks, int dst_blocks)
{
    if (n < 0 || block_elems <= 0)
        return -1;
    for (int p = 0; p < n; p++) {
        int32_t src = pairs[2 * p], dst = pairs[2 * p + 1];
        if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks)
            return -2;
        for (int64_t i = 0; i < block_elems; i++)
            dst_pool[(int64_t)dst * block_elems + i] = src_pool[(int64_t)src * block_elems + i];
    }
    return 0;
}

/* ---- decode attention over the paged cache ------------------------------ */

static int check_row(const int32_t *table_row, int max_blocks, int B, int64_t ctx, int NB)
{
    if (ctx > (int64_t)max_blocks * B)
        return -1;
    for (int64_t j = 0; j * B < ctx; j++)
        if (table_row[j] < 0 || table_row[j] >= NB)
            return -2;
    return 0;
}

/* One (sequence, query head): the attention equation of §I, over tokens
 * [t0, t1) gathered through the block table.  Writes the scores' maximum m,
 * the sum of exp(x_t - m) and the un-normalised sum of exp(x_t - m) v_t.
 * An empty range gives m = -inf, l = 0, o = 0. */
static void attend_range(const uint16_t *q, const uint16_t *key_cache,
                         const uint16_t *value_cache, const int32_t *table_row,
                         int64_t t0, int64_t t1, int B, int Hkv, int g, int d,
                         double scale, int is_bf16, double *m_out, double *l_out,
                         double *o_out, double *x /* scratch, t1 - t0 */)
{
    double m = -INFINITY;
    for (int64_t t = t0; t < t1; t++) {
        int32_t p, off;
        locate(table_row, B, t, &p, &off);
        const uint16_t *k = key_cache + (((int64_t)p * Hkv + g) * B + off) * d;
        double dot = 0.0;
        for (int i = 0; i < d; i++)
            dot += to_double(q[i], is_bf16) * to_double(k[i], is_bf16);
        x[t - t0] = scale * dot;
        if (x[t - t0] > m)
            m = x[t - t0];
    }
    double l = 0.0;
    for (int i = 0; i < d; i++)
        o_out[i] = 0.0;
    for (int64_t t = t0; t < t1; t++) {
        int32_t p, off;
        locate(table_row, B, t, &p, &off);
        const uint16_t *v = value_cache + (((int64_t)p * Hkv + g) * B + off) * d;
        double w = exp(x[t - t0] - m);
        l += w;
        for (int i = 0; i < d; i++)
            o_out[i] += w * to_double(v[i], is_bf16);
    }
    *m_out = m;
    *l_out = l;
}

/* out[s][h][:] = sum_t softmax_t(scale * q.k_t) v_t over the context_lens[s]
 * tokens of sequence s.  An empty context gives zeros.
 * `which` lists (s, h) pairs to compute (n_which of them); NULL computes all,
 * and the other rows of out are left untouched. */
int oracle_paged_attention(double *out, const uint16_t *query,
                           const uint16_t *key_cache, const uint16_t *value_cache,
                           const int32_t *block_tables, const int32_t *context_lens,
                           int S, int max_blocks, int B, int H, int Hkv, int d,
                           double scale, int is_bf16, int NB,
                           const int32_t *which, int n_which)
{
    if (S < 0 || max_blocks < 0 || B <= 0 || H <= 0 || Hkv <= 0 || d <= 0 || H % Hkv)
        return -1;
    for (int s = 0; s < S; s++) {
        if (context_lens[s] < 0)
            return -1;
        int rc = check_row(block_tables + (int64_t)s * max_blocks, max_blocks, B,
                           context_lens[s], NB);
        if (rc)
            return rc;
    }
    int64_t max_ctx = 0;
    for (int s = 0; s < S; s++)
        if (context_lens[s] > max_ctx)
            max_ctx = context_lens[s];
    double *x = malloc(sizeof(double) * (size_t)(max_ctx > 0 ? max_ctx : 1));
    if (!x)
        return -1;
    int n = which ? n_which : S * H;
    for (int k = 0; k < n; k++) {
        int s = which ? which[2 * k] : k / H;
        int h = which ? which[2 * k + 1] : k % H;
        if (s < 0 || s >= S || h < 0 || h >= H) {
            free(x);
            return -2;
        }
        int g = h / (H / Hkv);
        double *o = out + ((int64_t)s * H + h) * d;
        double m, l;
        attend_range(query + ((int64_t)s * H + h) * d, key_cache, value_cache,
                     block_tables + (int64_t)s * max_blocks, 0, context_lens[s], B, Hkv,
                     g, d, scale, is_bf16, &m, &l, o, x);
        for (int i = 0; i < d; i++)
            o[i] = l > 0.0 ? o[i] / l : 0.0;
    }
    free(x);
    return 0;
}

/* ---- prompt phase: many query tokens per sequence, causal --------------- */

/* The prompt (prefill) phase ("vLLM & PagedAttention" §II and §V) takes a
 * sequence's new tokens all at once; with a shared prefix (§VII) those are the
 * request's own input after prefix blocks that are already cached.  Sequence
 * s has n_s = query_start[s+1] - query_start[s] new tokens, the last n_s of
 * its context_lens[s]; their keys and values are already in the cache.  New
 * token j sits at position p = context_lens[s] - n_s + j and, by the causal
 * sum of the §I attention equation (t <= i), attends tokens 0..p.
 *
 * Layouts: query and out [T][H][d] with T = query_start[S]; query_start [S+1]
 * non-decreasing from 0.  `which` lists (token, h) pairs to compute (n_which
 * of them); NULL computes all, and the other rows of out are left untouched.
 * A sequence with n_s = 0 has no rows.  n_s > context_lens[s] is a bad size. */
int oracle_paged_prefill(double *out, const uint16_t *query,
                         const uint16_t *key_cache, const uint16_t *value_cache,
                         const int32_t *block_tables, const int32_t *context_lens,
                         const int32_t *query_start, int S, int max_blocks, int B,
                         int H, int Hkv, int d, double scale, int is_bf16, int NB,
                         const int32_t *which, int n_which)
{
    if (S < 0 || max_blocks < 0 || B <= 0 || H <= 0 || Hkv <= 0 || d <= 0 || H % Hkv)
        return -1;
    if (S > 0 && query_start[0] != 0)
        return -1;
    int64_t max_ctx = 0;
    for (int s = 0; s < S; s++) {
        int64_t n = (int64_t)query_start[s + 1] - query_start[s];
        if (n < 0 || context_lens[s] < 0 || n > context_lens[s])
            return -1;
        int rc = check_row(block_tables + (int64_t)s * max_blocks, max_blocks, B,
                           context_lens[s], NB);
        if (rc)
            return rc;
        if (context_lens[s] > max_ctx)
            max_ctx = context_lens[s];
    }
    int64_t T = S > 0 ? query_start[S] : 0;
    double *x = malloc(sizeof(double) * (size_t)(max_ctx > 0 ? max_ctx : 1));
    if (!x)
        return -1;
    int64_t n_rows = which ? n_which : T * H;
    int s = 0;
    for (int64_t k = 0; k < n_rows; k++) {
        int64_t tok = which ? which[2 * k] : k / H;
        int h = which ? which[2 * k + 1] : (int)(k % H);
        if (tok < 0 || tok >= T || h < 0 || h >= H) {
            free(x);
            return -2;
        }
        /* the sequence holding new token `tok` */
        if (which || tok < query_start[s])
            s = 0;
        while (query_start[s + 1] <= tok)
            s++;
        int64_t n = (int64_t)query_start[s + 1] - query_start[s];
        int64_t p = context_lens[s] - n + (tok - query_start[s]);
        double *o = out + (tok * H + h) * d;
        double m, l;
        attend_range(query + (tok * H + h) * d, key_cache, value_cache,
                     block_tables + (int64_t)s * max_blocks, 0, p + 1, B, Hkv,
                     h / (H / Hkv), d, scale, is_bf16, &m, &l, o, x);
        for (int i = 0; i < d; i++)
            o[i] = l > 0.0 ? o[i] / l : 0.0;
    }
    free(x);
    return 0;
}

/* ---- split context: per-partition statistics and their merge ------------ */

/* For one (s, h): partition p covers tokens [p*P, min((p+1)*P, ctx)).
 * Writes m[p], l[p], o[p][:] (un-normalised) for p < ceil(ctx / P) and
 * returns that count (or a negative code). */
int oracle_partition_stats(const uint16_t *query, const uint16_t *key_cache,
                           const uint16_t *value_cache, const int32_t *block_tables,
                           const int32_t *context_lens, int S, int max_blocks, int B,
                           int H, int Hkv, int d, double scale, int is_bf16, int NB,
                           int s, int h, int P, double *m, double *l, double *o)
{
    if (P <= 0 || s < 0 || s >= S || h < 0 || h >= H || H % Hkv)
        return -1;
    int64_t ctx = context_lens[s];
    int rc = check_row(block_tables + (int64_t)s * max_blocks, max_blocks, B, ctx, NB);
    if (rc)
        return rc;
    double *x = malloc(sizeof(double) * (size_t)P);
    if (!x)
        return -1;
    int np = 0;
    for (int64_t t0 = 0; t0 < ctx; t0 += P, np++) {
        int64_t t1 = t0 + P < ctx ? t0 + P : ctx;
        attend_range(query + ((int64_t)s * H + h) * d, key_cache, value_cache,
                     block_tables + (int64_t)s * max_blocks, t0, t1, B, Hkv, h / (H / Hkv),
                     d, scale, is_bf16, &m[np], &l[np], o + (int64_t)np * d, x);
    }
    free(x);
    return np;
}

/* Log-sum-exp merge of n partitions: M = max_p m_p, L = sum_p l_p e^(m_p - M),
 * out = sum_p o_p e^(m_p - M) / L.  n = 0 gives zeros. */
void oracle_merge_partitions(const double *m, const double *l, const double *o,
                             int n, int d, double *out)
{
    double M = -INFINITY;
    for (int p = 0; p < n; p++)
        if (m[p] > M)
            M = m[p];
    double L = 0.0;
    for (int i = 0; i < d; i++)
        out[i] = 0.0;
    for (int p = 0; p < n; p++) {
        double w = exp(m[p] - M);
        L += l[p] * w;
        for (int i = 0; i < d; i++)
            out[i] += o[(int64_t)p * d + i] * w;
    }
    for (int i = 0; i < d; i++)
        out[i] = L > 0.0 ? out[i] / L : 0.0;
}
