/*
 * Paged KV-cache attention oracle: a plain, slow, fp64 CPU reference.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header or constant with the CUDA library; it defines its own copy of
 * the cache layout from the layout's written description.
 *
 * What it computes (the vLLM pages' statement of PagedAttention):
 *
 *  - Cache write ("vLLM internals: managing the KV cache like an OS manages
 *    memory", section 2.1; "continuous batching and PagedAttention"
 *    tutorial, section 3.3 "Data structures", step 2 of each decode): every
 *    new token t with slot_mapping[t] >= 0 is stored at physical block
 *    slot / block_size, offset slot % block_size.  It is a bit copy.
 *
 *  - Attention (tutorial section 3.6 "PagedAttention kernel"; "vLLM source
 *    reading" section 2.3): the query token at position p of request r
 *    attends to keys 0..p of its own request, key j being read from physical
 *    block block_tables[r][j / block_size] at offset j % block_size.  The
 *    result is plain softmax(scale * q.k_j) weighted sum of v_j, computed in
 *    two passes (maximum, then exponentials) in fp64.
 *
 * Cache layout (an independent statement of the library's documented
 * layout): bf16 [num_blocks][num_kv_heads][2][block_size][head_size], index 0
 * of the third axis holding K and 1 holding V.  bf16 values are taken as raw
 * 16-bit patterns and widened exactly to double.
 *
 * Positions: a request with seq_len L and query_len q has context c = L - q;
 * its i-th query token sits at position c + i (the new tokens are the last q
 * of the sequence, written before attention reads them).  Query head h reads
 * kv head h / (num_q_heads / num_kv_heads).
 *
 * FP8 cache option ("vLLM internals: managing the KV cache like an OS manages
 * memory", section 7.2, the KV cache itself can be stored in FP8; the
 * "continuous batching and PagedAttention" tutorial, sections 8.8, 10.3 and
 * the FAQ of 10.8: an FP8 KV cache halves its memory at almost no loss).  The
 * pages fix neither the 8-bit format nor the scaling; the reading taken is
 * the OCP E4M3 format (sign, 4 exponent bits with bias 7, 3 mantissa bits;
 * exponent 0 is subnormal; all-ones exponent and mantissa is NaN; no
 * infinities; largest finite 448) with one fp32 scale for all K and one for
 * all V: the stored code is E4M3(x / scale), the quotient an fp32 division
 * rounded to nearest and the code the nearest E4M3 value (ties to the even
 * code, magnitudes past 448 held at 448), and the cache then holds
 * code_value * scale.  The same layout holds one byte per element.
 *
 * Every function returns 0 on success and a negative code on invalid input.
 */

#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_EINVAL (-1)
#define ORACLE_ERANGE (-2)
#define ORACLE_EDUP (-3)
#define ORACLE_ENOMEM (-4)

static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* element offset of (block, kv head, k-or-v, offset-in-block, dim 0) */
static size_t cache_offset(int64_t block, int32_t kv_head, int32_t which, int32_t off,
                           int32_t num_kv_heads, int32_t block_size, int32_t head_size)
{
    size_t idx = (size_t)block;
    idx = idx * (size_t)num_kv_heads + (size_t)kv_head;
    idx = idx * 2u + (size_t)which;
    idx = idx * (size_t)block_size + (size_t)off;
    return idx * (size_t)head_size;
}

/* ---- E4M3 ------------------------------------------------------------------ */

/* The value of an E4M3 code, from the format's definition. */
double oracle_e4m3_decode(uint8_t code)
{
    const int sign = code >> 7;
    const int e = (code >> 3) & 15;
    const int m = code & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);               /* m/8 * 2^(1-7) */
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/*
 * The E4M3 code nearest to x (ties to the even code), magnitudes at or past
 * 448 held at 448, NaN to 0x7F.  The sign is kept, also for results that
 * round to zero.
 */
uint8_t oracle_e4m3_encode(float x)
{
    if (isnan(x))
        return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7E;
    int code;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: multiples of 2^-9; code = that multiple (0..8) */
        code = (int)nearbyint(ldexp(a, 9));     /* exact scaling; rounds half to even */
    } else {
        int ex;
        const double fr = frexp(a, &ex);        /* a = fr * 2^ex, fr in [0.5, 1) */
        const int e = ex - 1;                   /* a = (2 fr) * 2^e, 2 fr in [1, 2) */
        const int m = (int)nearbyint((2.0 * fr - 1.0) * 8.0);
        code = ((e + 7) << 3) + m;              /* m = 8 carries into the exponent */
    }
    return sign | (uint8_t)code;
}

/* fp32 quotient x / scale, rounded to nearest (the value that is encoded). */
static float quotient_f32(float x, float scale)
{
    volatile float q = x / scale;               /* a single IEEE fp32 division */
    return q;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static int cmp_i64(const void *a, const void *b)
{
    int64_t x = *(const int64_t *)a, y = *(const int64_t *)b;
    return (x > y) - (x < y);
}

/* Cache write.  key/value: bf16 [num_tokens][num_kv_heads][head_size]. */
int oracle_kv_write(uint16_t *cache, int64_t num_blocks, int32_t num_kv_heads,
                    int32_t head_size, int32_t block_size,
                    const uint16_t *key, const uint16_t *value,
                    const int64_t *slot_mapping, int32_t num_tokens)
{
    if (num_tokens < 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0 || num_blocks < 0)
        return ORACLE_EINVAL;
    if (num_tokens == 0)
        return 0;
    if (!cache || !key || !value || !slot_mapping)
        return ORACLE_EINVAL;
    const int64_t num_slots = num_blocks * (int64_t)block_size;

    /* a slot written twice in one call has no defined result: reject it */
    int64_t *sorted = (int64_t *)malloc(sizeof(int64_t) * (size_t)num_tokens);
    if (!sorted)
        return ORACLE_ENOMEM;
    int32_t n = 0;
    for (int32_t t = 0; t < num_tokens; ++t) {
        int64_t s = slot_mapping[t];
        if (s >= num_slots) {
            free(sorted);
            return ORACLE_ERANGE;
        }
        if (s >= 0)
            sorted[n++] = s;
    }
    qsort(sorted, (size_t)n, sizeof(int64_t), cmp_i64);
    for (int32_t i = 1; i < n; ++i) {
        if (sorted[i] == sorted[i - 1]) {
            free(sorted);
            return ORACLE_EDUP;
        }
    }
    free(sorted);

    const size_t row = (size_t)head_size * sizeof(uint16_t);
    for (int32_t t = 0; t < num_tokens; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue; /* padding token */
        const int64_t block = slot / block_size;
        const int32_t off = (int32_t)(slot % block_size);
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            const size_t src = ((size_t)t * (size_t)num_kv_heads + (size_t)h) * (size_t)head_size;
            memcpy(cache + cache_offset(block, h, 0, off, num_kv_heads, block_size, head_size),
                   key + src, row);
            memcpy(cache + cache_offset(block, h, 1, off, num_kv_heads, block_size, head_size),
                   value + src, row);
        }
    }
    return 0;
}

/*
 * Cache write into an FP8 cache: the same slots as oracle_kv_write, each
 * element stored as oracle_e4m3_encode(bf16 value / scale), k_scale for K
 * and v_scale for V.  cache: uint8 [num_blocks][num_kv_heads][2][block_size][head_size].
 */
int oracle_kv_write_fp8(uint8_t *cache, int64_t num_blocks, int32_t num_kv_heads,
                        int32_t head_size, int32_t block_size,
                        const uint16_t *key, const uint16_t *value,
                        const int64_t *slot_mapping, int32_t num_tokens,
                        float k_scale, float v_scale)
{
    if (num_tokens < 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0 || num_blocks < 0)
        return ORACLE_EINVAL;
    if (!(k_scale > 0.0f) || !(v_scale > 0.0f) || isinf(k_scale) || isinf(v_scale))
        return ORACLE_EINVAL;
    if (num_tokens == 0)
        return 0;
    if (!cache || !key || !value || !slot_mapping)
        return ORACLE_EINVAL;
    const int64_t num_slots = num_blocks * (int64_t)block_size;
    int64_t *sorted = (int64_t *)malloc(sizeof(int64_t) * (size_t)num_tokens);
    if (!sorted)
        return ORACLE_ENOMEM;
    int32_t n = 0;
    for (int32_t t = 0; t < num_tokens; ++t) {
        int64_t s = slot_mapping[t];
        if (s >= num_slots) {
            free(sorted);
            return ORACLE_ERANGE;
        }
        if (s >= 0)
            sorted[n++] = s;
    }
    qsort(sorted, (size_t)n, sizeof(int64_t), cmp_i64);
    for (int32_t i = 1; i < n; ++i) {
        if (sorted[i] == sorted[i - 1]) {
            free(sorted);
            return ORACLE_EDUP;
        }
    }
    free(sorted);

    for (int32_t t = 0; t < num_tokens; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        const int64_t block = slot / block_size;
        const int32_t off = (int32_t)(slot % block_size);
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            const size_t src = ((size_t)t * (size_t)num_kv_heads + (size_t)h) * (size_t)head_size;
            uint8_t *kd = cache + cache_offset(block, h, 0, off, num_kv_heads, block_size, head_size);
            uint8_t *vd = cache + cache_offset(block, h, 1, off, num_kv_heads, block_size, head_size);
            for (int32_t e = 0; e < head_size; ++e) {
                kd[e] = oracle_e4m3_encode(quotient_f32((float)bf16_bits_to_double(key[src + e]), k_scale));
                vd[e] = oracle_e4m3_encode(quotient_f32((float)bf16_bits_to_double(value[src + e]), v_scale));
            }
        }
    }
    return 0;
}

/*
 * Copy-on-write block copies ("continuous batching and PagedAttention"
 * tutorial, section 3.8): for every pair, the destination block receives a
 * bit copy of the source block (every kv head, K and V).  mapping: int64
 * [num_pairs][2] = {source, destination}.  Out-of-range ids are rejected.
 */
int oracle_copy_blocks(uint16_t *cache, int64_t num_blocks, int32_t num_kv_heads, int32_t head_size,
                       int32_t block_size, const int64_t *mapping, int32_t num_pairs)
{
    if (num_pairs < 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0)
        return ORACLE_EINVAL;
    if (num_pairs == 0)
        return 0;
    if (!cache || !mapping)
        return ORACLE_EINVAL;
    for (int32_t i = 0; i < num_pairs; ++i)
        if (mapping[2 * i] < 0 || mapping[2 * i] >= num_blocks || mapping[2 * i + 1] < 0 ||
            mapping[2 * i + 1] >= num_blocks)
            return ORACLE_ERANGE;
    const size_t block_elems = cache_offset(1, 0, 0, 0, num_kv_heads, block_size, head_size);
    for (int32_t i = 0; i < num_pairs; ++i) {
        const int64_t src = mapping[2 * i], dst = mapping[2 * i + 1];
        if (src == dst)
            continue;
        memcpy(cache + (size_t)dst * block_elems, cache + (size_t)src * block_elems,
               block_elems * sizeof(uint16_t));
    }
    return 0;
}

typedef struct {
    const uint16_t *query;
    const void *cache;          /* bf16 elements, or E4M3 bytes when fp8 */
    int64_t num_blocks;
    const int32_t *block_tables;
    int32_t max_blocks_per_seq;
    const int32_t *seq_lens;
    const int32_t *query_start_loc;
    int32_t num_seqs;
    int32_t num_q_heads, num_kv_heads, head_size, block_size;
    double scale;
    int fp8;                    /* 0: bf16 cache; 1: E4M3 cache */
    double k_scale, v_scale;    /* fp8 only: the value is code_value * scale */
} problem_t;

/* Element e of the K (which = 0) or V (which = 1) row at (block, kv head, offset). */
static double cache_elem(const problem_t *p, int64_t block, int32_t kv_head, int32_t which, int32_t off,
                         int32_t e)
{
    const size_t i = cache_offset(block, kv_head, which, off, p->num_kv_heads, p->block_size, p->head_size) +
                     (size_t)e;
    if (p->fp8)
        return oracle_e4m3_decode(((const uint8_t *)p->cache)[i]) * (which ? p->v_scale : p->k_scale);
    return bf16_bits_to_double(((const uint16_t *)p->cache)[i]);
}

static int check_problem(const problem_t *p)
{
    if (p->num_seqs < 0 || p->num_q_heads <= 0 || p->num_kv_heads <= 0 || p->head_size <= 0 ||
        p->block_size <= 0 || p->max_blocks_per_seq < 0)
        return ORACLE_EINVAL;
    if (p->num_q_heads % p->num_kv_heads)
        return ORACLE_EINVAL;
    if (p->num_seqs == 0)
        return 0;
    if (!p->query_start_loc || !p->seq_lens || !p->block_tables || !p->cache)
        return ORACLE_EINVAL;
    if (p->query_start_loc[0] != 0)
        return ORACLE_EINVAL;
    for (int32_t r = 0; r < p->num_seqs; ++r) {
        const int32_t q = p->query_start_loc[r + 1] - p->query_start_loc[r];
        const int32_t L = p->seq_lens[r];
        if (q < 0 || L < q)
            return ORACLE_EINVAL;
        const int64_t nblk = ((int64_t)L + p->block_size - 1) / p->block_size;
        if (nblk > p->max_blocks_per_seq)
            return ORACLE_ERANGE;
        if (q == 0)
            continue;
        for (int64_t b = 0; b < nblk; ++b) {
            const int32_t phys = p->block_tables[(size_t)r * (size_t)p->max_blocks_per_seq + (size_t)b];
            if (phys < 0 || phys >= p->num_blocks)
                return ORACLE_ERANGE;
        }
    }
    return 0;
}

/*
 * Attention of one query row (request r, its i-th query token, q head h)
 * over the keys j in [key_begin, key_end) that it may see (j <= its
 * position).  Writes the normalised output to out[head_size] and the natural
 * log-sum-exp of the scaled scores to *lse; with no visible key, out is all
 * zero and *lse is -inf.  When weights is not NULL it receives the
 * normalised softmax weight of every visible key, in key order.
 * scores: scratch of at least (key_end - key_begin) doubles.
 */
static void attend_row(const problem_t *p, int32_t r, int32_t i, int32_t h,
                       int64_t key_begin, int64_t key_end,
                       double *scores, double *out, double *lse, double *weights)
{
    const int32_t d = p->head_size;
    const int32_t B = p->block_size;
    const int32_t G = p->num_q_heads / p->num_kv_heads;
    const int32_t g = h / G;
    const int32_t q_len = p->query_start_loc[r + 1] - p->query_start_loc[r];
    const int64_t context = (int64_t)p->seq_lens[r] - q_len;
    const int64_t pos = context + i;
    const int64_t t = (int64_t)p->query_start_loc[r] + i;
    const int32_t *table = p->block_tables + (size_t)r * (size_t)p->max_blocks_per_seq;
    const uint16_t *q = p->query + ((size_t)t * (size_t)p->num_q_heads + (size_t)h) * (size_t)d;

    int64_t j0 = key_begin < 0 ? 0 : key_begin;
    int64_t j1 = key_end < pos + 1 ? key_end : pos + 1;
    for (int32_t e = 0; e < d; ++e)
        out[e] = 0.0;
    if (j1 <= j0) {
        *lse = -INFINITY;
        return;
    }

    /* pass 1: scores and their maximum */
    double m = -INFINITY;
    for (int64_t j = j0; j < j1; ++j) {
        const int32_t phys = table[j / B];
        double dot = 0.0;
        for (int32_t e = 0; e < d; ++e)
            dot += bf16_bits_to_double(q[e]) * cache_elem(p, phys, g, 0, (int32_t)(j % B), e);
        const double s = p->scale * dot;
        scores[j - j0] = s;
        if (s > m)
            m = s;
    }
    /* pass 2: exponentials, their sum, and the weighted sum of values */
    double z = 0.0;
    for (int64_t j = j0; j < j1; ++j) {
        const double w = exp(scores[j - j0] - m);
        scores[j - j0] = w;
        z += w;
        const int32_t phys = table[j / B];
        for (int32_t e = 0; e < d; ++e)
            out[e] += w * cache_elem(p, phys, g, 1, (int32_t)(j % B), e);
    }
    for (int32_t e = 0; e < d; ++e)
        out[e] /= z;
    *lse = m + log(z);
    if (weights)
        for (int64_t j = j0; j < j1; ++j)
            weights[j - j0] = scores[j - j0] / z;
}

static int64_t longest_seq(const problem_t *p)
{
    int64_t mx = 1;
    for (int32_t r = 0; r < p->num_seqs; ++r)
        if (p->seq_lens[r] > mx)
            mx = p->seq_lens[r];
    return mx;
}

/*
 * Full attention step.  out: double [num_tokens][num_q_heads][head_size];
 * lse: double [num_tokens][num_q_heads] (may be NULL).  Rows are
 * independent; num_threads <= 0 uses every available thread.
 */
static int paged_attn_all(const problem_t *pp, double *out, double *lse, int32_t num_threads);

int oracle_paged_attn(double *out, double *lse, const uint16_t *query,
                      const uint16_t *cache, int64_t num_blocks,
                      const int32_t *block_tables, int32_t max_blocks_per_seq,
                      const int32_t *seq_lens, const int32_t *query_start_loc, int32_t num_seqs,
                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                      int32_t block_size, float scale, int32_t num_threads)
{
    problem_t p = {query, cache, num_blocks, block_tables, max_blocks_per_seq, seq_lens,
                   query_start_loc, num_seqs, num_q_heads, num_kv_heads, head_size,
                   block_size, (double)scale, 0, 1.0, 1.0};
    return paged_attn_all(&p, out, lse, num_threads);
}

/* The same attention over an E4M3 cache: K and V values are code_value * scale. */
int oracle_paged_attn_fp8(double *out, double *lse, const uint16_t *query,
                          const uint8_t *cache, int64_t num_blocks,
                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                          const int32_t *seq_lens, const int32_t *query_start_loc, int32_t num_seqs,
                          int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                          int32_t block_size, float scale, float k_scale, float v_scale,
                          int32_t num_threads)
{
    if (!(k_scale > 0.0f) || !(v_scale > 0.0f) || isinf(k_scale) || isinf(v_scale))
        return ORACLE_EINVAL;
    problem_t p = {query, cache, num_blocks, block_tables, max_blocks_per_seq, seq_lens,
                   query_start_loc, num_seqs, num_q_heads, num_kv_heads, head_size,
                   block_size, (double)scale, 1, (double)k_scale, (double)v_scale};
    return paged_attn_all(&p, out, lse, num_threads);
}

static int paged_attn_all(const problem_t *pp, double *out, double *lse, int32_t num_threads)
{
    const problem_t p = *pp;
    const int32_t num_seqs = p.num_seqs, num_q_heads = p.num_q_heads, head_size = p.head_size;
    const int32_t *query_start_loc = p.query_start_loc, *seq_lens = p.seq_lens;
    const uint16_t *query = p.query;
    int rc = check_problem(&p);
    if (rc)
        return rc;
    if (num_seqs == 0)
        return 0;
    const int64_t num_tokens = query_start_loc[num_seqs];
    if (num_tokens == 0)
        return 0;
    if (!out || !query)
        return ORACLE_EINVAL;
    /* the request each query token belongs to, by a plain walk over requests */
    int32_t *owner = (int32_t *)malloc(sizeof(int32_t) * (size_t)num_tokens);
    if (!owner)
        return ORACLE_ENOMEM;
    for (int32_t r = 0; r < num_seqs; ++r)
        for (int32_t t = query_start_loc[r]; t < query_start_loc[r + 1]; ++t)
            owner[t] = r;
    const int64_t units = num_tokens * num_q_heads;
    const int64_t scratch_len = longest_seq(&p);
    int failed = 0;
#ifdef _OPENMP
    if (num_threads > 0)
        omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif
#pragma omp parallel
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)scratch_len);
        if (!scores) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t u = 0; u < units; ++u) {
            if (!scores)
                continue;
            const int64_t t = u / num_q_heads;
            const int32_t h = (int32_t)(u % num_q_heads);
            const int32_t r = owner[t];
            const int32_t i = (int32_t)(t - query_start_loc[r]);
            double l;
            attend_row(&p, r, i, h, 0, seq_lens[r], scores,
                       out + (size_t)u * (size_t)head_size, &l, NULL);
            if (lse)
                lse[u] = l;
        }
        free(scores);
    }
    free(owner);
    return failed ? ORACLE_ENOMEM : 0;
}

/*
 * One row restricted to keys [key_begin, key_end): the partial result that a
 * split of the key range produces.  out: double [head_size]; weights (may be
 * NULL): double [key_end - key_begin], filled for the visible keys.
 * Returns the number of visible keys (>= 0) or a negative code.
 */
int oracle_attn_row(double *out, double *lse, double *weights, const uint16_t *query,
                    const uint16_t *cache, int64_t num_blocks,
                    const int32_t *block_tables, int32_t max_blocks_per_seq,
                    const int32_t *seq_lens, const int32_t *query_start_loc, int32_t num_seqs,
                    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                    int32_t block_size, float scale,
                    int32_t request, int32_t query_index, int32_t q_head,
                    int64_t key_begin, int64_t key_end)
{
    problem_t p = {query, cache, num_blocks, block_tables, max_blocks_per_seq, seq_lens,
                   query_start_loc, num_seqs, num_q_heads, num_kv_heads, head_size,
                   block_size, (double)scale, 0, 1.0, 1.0};
    int rc = check_problem(&p);
    if (rc)
        return rc;
    if (request < 0 || request >= num_seqs || q_head < 0 || q_head >= num_q_heads)
        return ORACLE_EINVAL;
    const int32_t q_len = query_start_loc[request + 1] - query_start_loc[request];
    if (query_index < 0 || query_index >= q_len || !out || !lse || !query)
        return ORACLE_EINVAL;
    const int64_t pos = (int64_t)seq_lens[request] - q_len + query_index;
    int64_t j0 = key_begin < 0 ? 0 : key_begin;
    int64_t j1 = key_end < pos + 1 ? key_end : pos + 1;
    int64_t n = j1 > j0 ? j1 - j0 : 0;
    double *scores = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    if (!scores)
        return ORACLE_ENOMEM;
    attend_row(&p, request, query_index, q_head, key_begin, key_end, scores, out, lse, weights);
    free(scores);
    return (int)n;
}

/*
 * Merge of partial results over a partition of one row's keys:
 * lse = log(sum_s exp(lse_s)), out = sum_s exp(lse_s - lse) * out_s.
 * A part with lse_s = -inf (no visible key) has weight 0.
 * part_out: double [n_parts][head_size].
 */
int oracle_lse_combine(double *out, double *lse_out, const double *part_out,
                       const double *part_lse, int32_t n_parts, int32_t head_size)
{
    if (n_parts <= 0 || head_size <= 0 || !out || !part_out || !part_lse)
        return ORACLE_EINVAL;
    double m = -INFINITY;
    for (int32_t s = 0; s < n_parts; ++s)
        if (part_lse[s] > m)
            m = part_lse[s];
    if (m == -INFINITY)
        return ORACLE_EINVAL; /* no part saw any key */
    double z = 0.0;
    for (int32_t e = 0; e < head_size; ++e)
        out[e] = 0.0;
    for (int32_t s = 0; s < n_parts; ++s) {
        if (part_lse[s] == -INFINITY)
            continue;
        const double w = exp(part_lse[s] - m);
        z += w;
        for (int32_t e = 0; e < head_size; ++e)
            out[e] += w * part_out[(size_t)s * (size_t)head_size + (size_t)e];
    }
    for (int32_t e = 0; e < head_size; ++e)
        out[e] /= z;
    if (lse_out)
        *lse_out = m + log(z);
    return 0;
}
