/*
 * CPU oracle for paged decode attention and its KV scatter.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library calls this code; only the
 * tests, the smoke check and the benchmark's CPU-baseline leg load it.  It
 * shares no code, header or table with the CUDA path.
 *
 * What it computes, and where that is stated:
 *  - The KV cache is a pool of fixed-size blocks reached through a per
 *    sequence block table that maps logical block j to a physical block id;
 *    blocks need not be contiguous and may be shared between sequences
 *    (vLLM web pages, "vllm-project-vllm" review, §3 Q2; §6 "KV Cache Block
 *    Tables").  Token i of sequence s therefore lives in physical block
 *    block_tables[s][i / bs] at offset i % bs.
 *  - Decode attends one new query token per sequence over that sequence's
 *    whole cached context (same review, §7: decode reads the full KV cache of
 *    every layer for one token at a time).  The result is plain softmax
 *    attention, evaluated here in fp64 straight from its definition:
 *        z_i = scale * <q, k_i>,  out = sum_i exp(z_i - max z) v_i / sum_i exp(z_i - max z).
 *  - The split variant evaluates the same quantity per fixed-size token
 *    partition and merges the partial results by log-sum-exp; it must equal
 *    the unsplit result up to rounding.
 *  - The scatter writes each new token's K and V rows into the slot named by
 *    its slot id (a sequence's blocks grow by one token every decode step:
 *    same review, §6).
 *    FP8 E4M3 caches store round-to-nearest-even(x / kv_scale), saturated to
 *    the largest finite E4M3 value, and are read back as code * kv_scale.
 *
 * Number formats are decoded from their bit definitions: IEEE-754 binary16;
 * bfloat16 = the upper 16 bits of an IEEE-754 binary32; OCP FP8 E4M3 (1 sign,
 * 4 exponent bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 is
 * NaN, largest finite value 448).
 *
 * Build: gcc -O2 -std=c11 -fopenmp -ffp-contract=off -shared -fPIC.  No fast
 * math: every float operation is IEEE round-to-nearest-even.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_E4M3 = 2 };

/* ------------------------------------------------------------------ */
/* number formats                                                      */
/* ------------------------------------------------------------------ */

/* IEEE-754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double orc_f16_to_double(uint16_t h)
{
    int sign = h >> 15, e = (h >> 10) & 0x1F, f = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-14 * 2^-10 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);     /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: the upper half of an IEEE-754 binary32. */
double orc_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float x;
    memcpy(&x, &u, sizeof x);
    return (double)x;
}

/* OCP FP8 E4M3 (the "fn" variant): bias 7, S.1111.111 = NaN, no infinities. */
double orc_e4m3_to_double(uint8_t c)
{
    int sign = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);                  /* subnormal: (m/8) * 2^(1-7) */
    else
        v = ldexp((double)(8 + m), e - 10);        /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/*
 * E4M3 encoding of a float32, round to nearest with ties to the even code,
 * saturating: any magnitude at or above 448 (and +-inf) becomes +-448.  The
 * nearest code is found by searching the sorted table of the 127 non-negative
 * finite E4M3 values, so nothing here depends on bit tricks.  The sign is
 * kept (a negative value that rounds to zero gives -0 = 0x80).  NaN gives 0x7F.
 */
static double e4m3_pos_value[127];   /* value of code c, c = 0..126 */
static int e4m3_ready = 0;

static void e4m3_table(void)
{
    if (e4m3_ready)
        return;
    for (int c = 0; c < 127; ++c)
        e4m3_pos_value[c] = orc_e4m3_to_double((uint8_t)c);
    e4m3_ready = 1;
}

uint8_t orc_float_to_e4m3(float y)
{
    e4m3_table();
    if (isnan(y))
        return 0x7F;
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs((double)y);
    if (a >= 448.0)
        return sign | 0x7E;
    /* largest code lo with value(lo) <= a (binary search, values increase with the code) */
    int lo = 0, hi = 126;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (e4m3_pos_value[mid] <= a)
            lo = mid;
        else
            hi = mid - 1;
    }
    int code = lo;
    if (e4m3_pos_value[lo] != a) {              /* a lies strictly between lo and lo+1 */
        double below = a - e4m3_pos_value[lo];
        double above = e4m3_pos_value[lo + 1] - a;
        if (above < below || (above == below && ((lo + 1) & 1) == 0))
            code = lo + 1;
    }
    return sign | (uint8_t)code;
}

/*
 * Round an fp64 value to a binary floating format with `p` significant bits
 * and smallest normal exponent `emin` (quantum floor 2^(emin - p + 1)),
 * ties to even, returning the rounded value in fp64 (exact).  Used only to
 * round final outputs; the tests compare against the unrounded value.
 */
static double round_to_format(double x, int p, int emin)
{
    if (x == 0.0 || !isfinite(x))
        return x;
    int e;
    frexp(fabs(x), &e);                 /* |x| = f * 2^e, f in [0.5, 1): floor(log2|x|) = e - 1 */
    int q = (e - 1) - (p - 1);          /* exponent of the last significant bit */
    if (q < emin - (p - 1))
        q = emin - (p - 1);
    double n = ldexp(x, -q);            /* exact: scaling by a power of two */
    double r = nearbyint(n);            /* default rounding mode: nearest, ties to even */
    return ldexp(r, q);
}

uint16_t orc_double_to_f16(double x)
{
    if (isnan(x))
        return 0x7E00;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double r = fabs(round_to_format(x, 11, -14));
    if (r > 65504.0)
        return sign | 0x7C00;
    if (r == 0.0)
        return sign;
    int e;
    frexp(r, &e);
    int E = e - 1;                      /* floor(log2 r) */
    if (E < -14)                        /* subnormal: r = f * 2^-24 */
        return sign | (uint16_t)ldexp(r, 24);
    uint16_t f = (uint16_t)(ldexp(r, 10 - E) - 1024.0);
    return sign | (uint16_t)((E + 15) << 10) | f;
}

uint16_t orc_double_to_bf16(double x)
{
    if (isnan(x))
        return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double r = fabs(round_to_format(x, 8, -126));
    double maxv = ldexp(255.0, 120);    /* (2 - 2^-7) * 2^127 */
    if (r > maxv)
        return sign | 0x7F80;
    if (r == 0.0)
        return sign;
    int e;
    frexp(r, &e);
    int E = e - 1;
    if (E < -126)                       /* subnormal: r = f * 2^-133 */
        return sign | (uint16_t)ldexp(r, 133);
    uint16_t f = (uint16_t)(ldexp(r, 7 - E) - 128.0);
    return sign | (uint16_t)((E + 127) << 7) | f;
}

/* lookup tables for the 16-bit formats (built once, from the decoders above) */
static double *tab_f16 = 0, *tab_bf16 = 0;

void orc_init(void)
{
    e4m3_table();
    if (!tab_f16) {
        double *a = (double *)malloc(65536 * sizeof(double));
        double *b = (double *)malloc(65536 * sizeof(double));
        for (int i = 0; i < 65536; ++i) {
            a[i] = orc_f16_to_double((uint16_t)i);
            b[i] = orc_bf16_to_double((uint16_t)i);
        }
        tab_f16 = a;
        tab_bf16 = b;
    }
}

static double decode16(uint16_t bits, int dtype)
{
    return dtype == ORC_F16 ? tab_f16[bits] : tab_bf16[bits];
}

/* Value of cache element `idx` as the attention reads it (FP8: code * kv_scale). */
static double cache_value(const void *cache, int64_t idx, int cache_dtype, double kv_scale)
{
    if (cache_dtype == ORC_E4M3)
        return orc_e4m3_to_double(((const uint8_t *)cache)[idx]) * kv_scale;
    return decode16(((const uint16_t *)cache)[idx], cache_dtype);
}

/* ------------------------------------------------------------------ */
/* reshape_and_cache                                                   */
/* ------------------------------------------------------------------ */

/*
 * For each token t with slot = slot_mapping[t] >= 0: block = slot / bs,
 * offset = slot % bs, and for every kv head h and channel d
 *     k_cache[block][h][offset][d] = key[t][h][d]   (same for value/v_cache).
 * Same dtype: the 16-bit pattern is copied.  FP8 cache: x is widened to
 * float32 (exact), y = x / kv_scale in float32, stored = e4m3(y).
 * Returns the number of tokens whose slot lay outside the pool (skipped).
 */
int64_t orc_reshape_and_cache(const uint16_t *key, const uint16_t *value, int in_dtype,
                              int64_t num_tokens, int num_kv_heads, int head_dim,
                              void *k_cache, void *v_cache, int cache_dtype,
                              int64_t num_blocks, int block_size,
                              const int64_t *slot_mapping, float kv_scale)
{
    orc_init();
    int64_t bad = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= num_blocks * (int64_t)block_size) {
            ++bad;
            continue;
        }
        int64_t blk = slot / block_size, off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            for (int d = 0; d < head_dim; ++d) {
                int64_t src = ((int64_t)t * num_kv_heads + h) * head_dim + d;
                int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * head_dim + d;
                if (cache_dtype == in_dtype) {
                    ((uint16_t *)k_cache)[dst] = key[src];
                    ((uint16_t *)v_cache)[dst] = value[src];
                } else {
                    float xk = (float)decode16(key[src], in_dtype);     /* exact widening */
                    float xv = (float)decode16(value[src], in_dtype);
                    float yk = xk / kv_scale;                           /* IEEE float32 division */
                    float yv = xv / kv_scale;
                    ((uint8_t *)k_cache)[dst] = orc_float_to_e4m3(yk);
                    ((uint8_t *)v_cache)[dst] = orc_float_to_e4m3(yv);
                }
            }
        }
    }
    return bad;
}

/* ------------------------------------------------------------------ */
/* decode attention                                                    */
/* ------------------------------------------------------------------ */

typedef struct {
    const uint16_t *q;
    int q_dtype, num_q_heads, num_kv_heads, head_dim;
    const void *k_cache, *v_cache;
    int cache_dtype;
    int64_t num_blocks;
    int block_size;
    const int32_t *block_tables;
    int max_blocks_per_seq;
    double scale, kv_scale;
} orc_problem;

/*
 * Softmax attention of query head g of sequence s over its context tokens
 * [t0, t1), reached through the block table.  Produces the partial result of
 * that range: m = max_i z_i, l = sum_i exp(z_i - m), o[d] = sum_i exp(z_i - m) v_i[d].
 * An empty range gives m = -inf, l = 0, o = 0.
 */
static void attend_range(const orc_problem *P, int s, int g, int t0, int t1,
                         double *m_out, double *l_out, double *o, double *z)
{
    int D = P->head_dim, Hkv = P->num_kv_heads, bs = P->block_size;
    int G = P->num_q_heads / Hkv;
    int h = g / G;                                       /* query head g reads kv head g / G */
    const uint16_t *qrow = P->q + ((int64_t)s * P->num_q_heads + g) * D;
    for (int d = 0; d < D; ++d)
        o[d] = 0.0;
    *m_out = -INFINITY;
    *l_out = 0.0;
    if (t1 <= t0)
        return;

    double m = -INFINITY;
    for (int i = t0; i < t1; ++i) {
        int64_t phys = P->block_tables[(int64_t)s * P->max_blocks_per_seq + i / bs];
        int64_t base = ((phys * Hkv + h) * bs + i % bs) * (int64_t)D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += decode16(qrow[d], P->q_dtype) * cache_value(P->k_cache, base + d, P->cache_dtype, P->kv_scale);
        z[i - t0] = P->scale * dot;
        if (z[i - t0] > m)
            m = z[i - t0];
    }
    double l = 0.0;
    for (int i = t0; i < t1; ++i) {
        int64_t phys = P->block_tables[(int64_t)s * P->max_blocks_per_seq + i / bs];
        int64_t base = ((phys * Hkv + h) * bs + i % bs) * (int64_t)D;
        double w = exp(z[i - t0] - m);
        l += w;
        for (int d = 0; d < D; ++d)
            o[d] += w * cache_value(P->v_cache, base + d, P->cache_dtype, P->kv_scale);
    }
    *m_out = m;
    *l_out = l;
}

/*
 * out[s][g][d] (fp64, unrounded) for every sequence and query head.
 * A sequence with context length 0 gives all zeros.  Returns 0, or -1 when a
 * context length exceeds max_blocks_per_seq * block_size or a block id in use
 * lies outside the pool (nothing is computed then).
 */
int orc_decode(double *out, const uint16_t *q, int q_dtype, int num_seqs, int num_q_heads,
               int num_kv_heads, int head_dim, const void *k_cache, const void *v_cache,
               int cache_dtype, int64_t num_blocks, int block_size,
               const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
               double scale, double kv_scale, int partition_size, int num_threads)
{
    orc_init();
    orc_problem P = {q, q_dtype, num_q_heads, num_kv_heads, head_dim, k_cache, v_cache,
                     cache_dtype, num_blocks, block_size, block_tables, max_blocks_per_seq,
                     scale, cache_dtype == ORC_E4M3 ? kv_scale : 1.0};
    for (int s = 0; s < num_seqs; ++s) {
        int L = context_lens[s];
        if (L < 0 || L > max_blocks_per_seq * block_size)
            return -1;
        for (int j = 0; j < (L + block_size - 1) / block_size; ++j) {
            int32_t b = block_tables[(int64_t)s * max_blocks_per_seq + j];
            if (b < 0 || b >= num_blocks)
                return -1;
        }
    }
    if (num_threads < 1)
        num_threads = 1;
    int D = head_dim;
    int64_t tasks = (int64_t)num_seqs * num_q_heads;

#pragma omp parallel num_threads(num_threads)
    {
        int maxL = max_blocks_per_seq * block_size;
        double *z = (double *)malloc(sizeof(double) * (maxL > 0 ? maxL : 1));
        double *o = (double *)malloc(sizeof(double) * D);
        double *acc = (double *)malloc(sizeof(double) * D);
#pragma omp for schedule(dynamic, 1)
        for (int64_t task = 0; task < tasks; ++task) {
            int s = (int)(task / num_q_heads), g = (int)(task % num_q_heads);
            int L = context_lens[s];
            double *dst = out + task * D;
            if (L == 0) {
                for (int d = 0; d < D; ++d)
                    dst[d] = 0.0;
                continue;
            }
            if (partition_size <= 0) {
                double m, l;
                attend_range(&P, s, g, 0, L, &m, &l, o, z);
                for (int d = 0; d < D; ++d)
                    dst[d] = o[d] / l;
            } else {
                /* per-partition partials (m_p, l_p, o_p), then the log-sum-exp merge:
                   M = max_p m_p, Lsum = sum_p l_p e^(m_p - M), out = sum_p o_p e^(m_p - M) / Lsum */
                int np = (L + partition_size - 1) / partition_size;
                double *pm = (double *)malloc(sizeof(double) * np);
                double *pl = (double *)malloc(sizeof(double) * np);
                double *po = (double *)malloc(sizeof(double) * (size_t)np * D);
                double M = -INFINITY;
                for (int p = 0; p < np; ++p) {
                    int t0 = p * partition_size;
                    int t1 = t0 + partition_size < L ? t0 + partition_size : L;
                    attend_range(&P, s, g, t0, t1, &pm[p], &pl[p], po + (size_t)p * D, z);
                    if (pm[p] > M)
                        M = pm[p];
                }
                double Lsum = 0.0;
                for (int d = 0; d < D; ++d)
                    acc[d] = 0.0;
                for (int p = 0; p < np; ++p) {
                    double w = exp(pm[p] - M);
                    Lsum += pl[p] * w;
                    for (int d = 0; d < D; ++d)
                        acc[d] += po[(size_t)p * D + d] * w;
                }
                for (int d = 0; d < D; ++d)
                    dst[d] = acc[d] / Lsum;
                free(pm);
                free(pl);
                free(po);
            }
        }
        free(z);
        free(o);
        free(acc);
    }
    return 0;
}

/* Partial results of one token range, for the merge tests. */
void orc_attend_range(double *m, double *l, double *o, const uint16_t *q, int q_dtype,
                      int num_q_heads, int num_kv_heads, int head_dim, const void *k_cache,
                      const void *v_cache, int cache_dtype, int64_t num_blocks, int block_size,
                      const int32_t *block_tables, int max_blocks_per_seq, double scale,
                      double kv_scale, int s, int g, int t0, int t1)
{
    orc_init();
    orc_problem P = {q, q_dtype, num_q_heads, num_kv_heads, head_dim, k_cache, v_cache,
                     cache_dtype, num_blocks, block_size, block_tables, max_blocks_per_seq,
                     scale, cache_dtype == ORC_E4M3 ? kv_scale : 1.0};
    double *z = (double *)malloc(sizeof(double) * (t1 > t0 ? t1 - t0 : 1));
    attend_range(&P, s, g, t0, t1, m, l, o, z);
    free(z);
}

/* Array helpers for the tests (same arithmetic as above, element-wise). */
void orc_decode16_array(const uint16_t *bits, double *out, int64_t n, int dtype)
{
    orc_init();
    for (int64_t i = 0; i < n; ++i)
        out[i] = decode16(bits[i], dtype);
}

void orc_e4m3_decode_array(const uint8_t *codes, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_to_double(codes[i]);
}

void orc_e4m3_encode_array(const float *y, uint8_t *out, int64_t n)
{
    e4m3_table();
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_float_to_e4m3(y[i]);
}

void orc_round_array(const double *x, uint16_t *out, int64_t n, int dtype)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = dtype == ORC_F16 ? orc_double_to_f16(x[i]) : orc_double_to_bf16(x[i]);
}

/* ------------------------------------------------------------------ */
/* whole-block moves                                                   */
/* ------------------------------------------------------------------ */

/* Block b of a cache is bytes [b * block_bytes, (b + 1) * block_bytes).
 * Copy: for each pair in order, cache[dst] = cache[src] (K and V).
 * Gather: buf[i] = (k[ids[i]], v[ids[i]]).  Scatter: the inverse.
 * Ids outside [0, num_blocks) are skipped; each returns how many it skipped. */
int64_t orc_copy_blocks(uint8_t *k_cache, uint8_t *v_cache, int64_t block_bytes, const int64_t *pairs, int64_t n,
                        int64_t num_blocks)
{
    int64_t bad = 0;
    for (int64_t i = 0; i < n; ++i) {
        int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            ++bad;
            continue;
        }
        memmove(k_cache + dst * block_bytes, k_cache + src * block_bytes, (size_t)block_bytes);
        memmove(v_cache + dst * block_bytes, v_cache + src * block_bytes, (size_t)block_bytes);
    }
    return bad;
}

int64_t orc_gather_blocks(uint8_t *buf, const uint8_t *k_cache, const uint8_t *v_cache, int64_t block_bytes,
                          const int64_t *ids, int64_t n, int64_t num_blocks)
{
    int64_t bad = 0;
    for (int64_t i = 0; i < n; ++i) {
        int64_t b = ids[i];
        if (b < 0 || b >= num_blocks) {
            ++bad;
            continue;
        }
        memcpy(buf + (2 * i) * block_bytes, k_cache + b * block_bytes, (size_t)block_bytes);
        memcpy(buf + (2 * i + 1) * block_bytes, v_cache + b * block_bytes, (size_t)block_bytes);
    }
    return bad;
}

int64_t orc_scatter_blocks(uint8_t *k_cache, uint8_t *v_cache, const uint8_t *buf, int64_t block_bytes,
                           const int64_t *ids, int64_t n, int64_t num_blocks)
{
    int64_t bad = 0;
    for (int64_t i = 0; i < n; ++i) {
        int64_t b = ids[i];
        if (b < 0 || b >= num_blocks) {
            ++bad;
            continue;
        }
        memcpy(k_cache + b * block_bytes, buf + (2 * i) * block_bytes, (size_t)block_bytes);
        memcpy(v_cache + b * block_bytes, buf + (2 * i + 1) * block_bytes, (size_t)block_bytes);
    }
    return bad;
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
