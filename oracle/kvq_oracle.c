/*
 * kvq_oracle.c -- plain, slow, fp64 CPU oracle for the FP8 paged-KV decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no source, header, table or helper with the
 * CUDA library under fp8_quantised_paged_kv_gb300/csrc.
 *
 * What it follows ("Smaller, faster, safer: running Kimi and GLM at scale",
 * as mirrored on the four source pages):
 *   - KV cache stored as FP8 e4m3 instead of BF16, halving its size
 *     (page 1, section "Quantised KV cache"; page 3, "FP8 saves more than
 *     memory").  The e4m3 bit layout itself is not on the pages; it is the
 *     OCP 8-bit floating point "E4M3" format: 1 sign bit, 4 exponent bits
 *     with bias 7, 3 mantissa bits, no infinities, S.1111.111 is NaN,
 *     largest finite magnitude 448.
 *   - The FP8 attention kernel converts the values it reads (page 1,
 *     "Quantised KV cache"), so attention here runs on decode(code) * scale.
 *   - Each physical cache page carries a tag that changes on reallocation;
 *     every request records the (page, tag) pairs it expects; a separate
 *     batched check runs before decode reads and aborts the request on any
 *     mismatch (page 2, "KV cache integrity check"; page 3, "A shared cache
 *     that cannot be wrong").
 *   - KV size = requests x tokens x layers x KV heads x head_dim x 2 x
 *     bytes per element (page 4, "Why memory becomes the bottleneck"): the
 *     argument list below follows those dimensions.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - quantise as one IEEE fp32 round-to-nearest division x / scale, then
 *     round that fp32 value to e4m3, ties to even, saturating at +-448
 *     (infinities included); NaN keeps its sign and encodes as S.1111.111;
 *     zero keeps its sign;
 *   - per-layer, per-KV-head fp32 scale, separate for K and V;
 *   - query head h reads KV head h / (Hq / Hkv);
 *   - an aborted request, an empty request, a request longer than its block
 *     table, or one whose table holds a page id outside [0, num_pages)
 *     produces zeros and reads no page;
 *   - the tag check compares, for each of the ceil(L / page_size) table
 *     entries a request uses, the live tag of that page with the tag the
 *     request expects; out-of-range page ids also abort.
 *
 * Cache layout: cache[page][kv_head][slot][dim], page-major, one byte per
 * element for e4m3, two (bf16 bits) for the bf16 variant.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- formats */

static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static float bf16_bits_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* e4m3 -> real number, straight from the format definition. */
double oracle_e4m3_decode(uint8_t code)
{
    int sign = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);          /* subnormal: m/8 * 2^(1-7) */
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7); /* normal: (1 + m/8) * 2^(e-7) */
    return sign ? -mag : mag;
}

/* Code of a non-negative representable magnitude v (0 <= v <= 448). */
static uint8_t e4m3_code_of_magnitude(double v)
{
    if (v < ldexp(1.0, -6)) {
        /* subnormal binade: v = m * 2^-9, m in 0..7 (m == 8 is the first
         * normal, whose code 0x08 is also 8, so the formula carries over). */
        return (uint8_t)(v / ldexp(1.0, -9));
    }
    int ex;
    frexp(v, &ex);                  /* v in [2^(ex-1), 2^ex) */
    int e = ex - 1 + 7;             /* biased exponent */
    int m = (int)(v / ldexp(1.0, ex - 1 - 3)) - 8;
    return (uint8_t)((e << 3) | m);
}

/* real (given as fp32) -> e4m3: round to nearest, ties to even, saturate. */
uint8_t oracle_e4m3_encode(float y)
{
    uint32_t bits;
    memcpy(&bits, &y, sizeof bits);
    uint8_t sign = (bits >> 31) ? 0x80 : 0x00;
    if (isnan(y))
        return sign | 0x7F;
    double a = fabs((double)y);
    if (a >= 448.0)
        return sign | 0x7E;         /* satfinite: out of range and +-inf -> +-448 */
    double quantum;
    if (a < ldexp(1.0, -6)) {
        quantum = ldexp(1.0, -9);   /* subnormal spacing */
    } else {
        int ex;
        frexp(a, &ex);              /* a in [2^(ex-1), 2^ex): 3 fraction bits */
        quantum = ldexp(1.0, ex - 1 - 3);
    }
    /* a / quantum is exact in double; nearbyint rounds half to even in the
     * default rounding mode, which is what ties-to-even on the mantissa
     * means because the quantum is the weight of the mantissa's last bit. */
    double v = nearbyint(a / quantum) * quantum;
    if (v > 448.0)
        v = 448.0;
    return sign | e4m3_code_of_magnitude(v);
}

/* Array forms of the two codec functions (same arithmetic, one call). */
void oracle_e4m3_encode_n(const float *y, uint8_t *codes, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        codes[i] = oracle_e4m3_encode(y[i]);
}

void oracle_e4m3_decode_n(const uint8_t *codes, double *values, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        values[i] = oracle_e4m3_decode(codes[i]);
}

/* --------------------------------------------------------------- append */

/*
 * Write each new token's K and V into the cache slot slot_mapping[t].
 * Tokens with slot < 0, slot >= num_pages * page_size, or a set abort flag
 * are skipped.  For the e4m3 cache each element becomes
 * encode((float)x / scale[h]) with the division done once in fp32.
 */
void oracle_append(int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                   int32_t page_size, int32_t num_pages, int32_t cache_is_bf16,
                   const uint16_t *k_new, const uint16_t *v_new,
                   const int64_t *slot_mapping,
                   const float *k_scale, const float *v_scale,
                   const uint8_t *abort_flags,
                   void *k_cache, void *v_cache)
{
    const int64_t num_slots = (int64_t)num_pages * page_size;
    int32_t t;
    /* tokens write distinct slots (a caller mapping two tokens to one slot is
     * an error on both sides), so the token loop can run on several threads */
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (t = 0; t < num_tokens; ++t) {
        if (abort_flags && abort_flags[t])
            continue;
        int64_t slot = slot_mapping[t];
        if (slot < 0 || slot >= num_slots)
            continue;
        int64_t page = slot / page_size;
        int64_t off = slot % page_size;
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            int64_t src = ((int64_t)t * num_kv_heads + h) * head_dim;
            int64_t dst = ((page * num_kv_heads + h) * page_size + off) * head_dim;
            for (int32_t d = 0; d < head_dim; ++d) {
                if (cache_is_bf16) {
                    ((uint16_t *)k_cache)[dst + d] = k_new[src + d];
                    ((uint16_t *)v_cache)[dst + d] = v_new[src + d];
                } else {
                    float kq = bf16_bits_to_float(k_new[src + d]) / k_scale[h];
                    float vq = bf16_bits_to_float(v_new[src + d]) / v_scale[h];
                    ((uint8_t *)k_cache)[dst + d] = oracle_e4m3_encode(kq);
                    ((uint8_t *)v_cache)[dst + d] = oracle_e4m3_encode(vq);
                }
            }
        }
    }
}

/* ------------------------------------------------------------- tag check */

/*
 * abort[r] = 1 if any of the ceil(L_r / page_size) table entries request r
 * uses names a page outside [0, num_pages) or a page whose live tag differs
 * from the tag the request expects; also 1 if L_r needs more entries than
 * the table row has.  Otherwise 0.  Every flag is written.
 */
void oracle_tag_check(const int32_t *block_table, const uint32_t *expected_tags,
                      const int32_t *seq_lens, int32_t batch, int32_t max_pages_per_seq,
                      int32_t page_size, const uint32_t *page_tags, int32_t num_pages,
                      uint8_t *abort_flags)
{
    for (int32_t r = 0; r < batch; ++r) {
        int64_t len = seq_lens[r] > 0 ? seq_lens[r] : 0;
        int64_t used = (len + page_size - 1) / page_size;
        uint8_t bad = 0;
        if (used > max_pages_per_seq) {
            bad = 1;
            used = max_pages_per_seq;
        }
        for (int64_t i = 0; i < used; ++i) {
            int32_t p = block_table[(int64_t)r * max_pages_per_seq + i];
            if (p < 0 || p >= num_pages || page_tags[p] != expected_tags[(int64_t)r * max_pages_per_seq + i])
                bad = 1;
        }
        abort_flags[r] = bad;
    }
}

/* ------------------------------------------------------------- attention */

static double cache_value(const void *cache, int32_t cache_is_bf16, int64_t idx, double scale)
{
    if (cache_is_bf16)
        return bf16_bits_to_double(((const uint16_t *)cache)[idx]);
    return oracle_e4m3_decode(((const uint8_t *)cache)[idx]) * scale;
}

/*
 * Single-token decode attention over a paged cache, in fp64.
 * For request r, query head h, KV head kvh = h / (Hq / Hkv):
 *   s_j = softmax_scale * sum_d q[r][h][d] * K^[j][d],     j = 0 .. L_r - 1
 *   out[r][h][:] = sum_j exp(s_j - max s) V^[j] / sum_j exp(s_j - max s)
 * where token j lives at page block_table[r][j / page_size], slot
 * j % page_size, and K^ = decode(code) * k_scale[kvh] (bf16 cache: the bf16
 * value).  Requests that are aborted, empty, longer than their table row or
 * that name a page outside [0, num_pages) get zeros.
 */
void oracle_decode_attn(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                        int32_t head_dim, int32_t page_size, int32_t num_pages,
                        int32_t cache_is_bf16, const uint16_t *q,
                        const void *k_cache, const void *v_cache,
                        const float *k_scale, const float *v_scale,
                        const int32_t *block_table, int32_t max_pages_per_seq,
                        const int32_t *seq_lens, float softmax_scale,
                        const uint8_t *abort_flags, double *out)
{
    const int32_t group = num_q_heads / num_kv_heads;
    const double sigma = (double)softmax_scale;
    int64_t rh;
    const int64_t total = (int64_t)batch * num_q_heads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (rh = 0; rh < total; ++rh) {
        const int32_t r = (int32_t)(rh / num_q_heads);
        const int32_t h = (int32_t)(rh % num_q_heads);
        double *o = out + rh * head_dim;
        for (int32_t d = 0; d < head_dim; ++d)
            o[d] = 0.0;
        const int64_t len = seq_lens[r];
        if (len <= 0 || (abort_flags && abort_flags[r]))
            continue;
        const int64_t used = (len + page_size - 1) / page_size;
        if (used > max_pages_per_seq)
            continue;
        const int32_t *row = block_table + (int64_t)r * max_pages_per_seq;
        int valid = 1;
        for (int64_t i = 0; i < used; ++i)
            if (row[i] < 0 || row[i] >= num_pages)
                valid = 0;
        if (!valid)
            continue;

        const int32_t kvh = h / group;
        const double ks = cache_is_bf16 ? 1.0 : (double)k_scale[kvh];
        const double vs = cache_is_bf16 ? 1.0 : (double)v_scale[kvh];
        const uint16_t *qh = q + rh * head_dim;
        double *s = (double *)malloc((size_t)len * sizeof(double));
        double smax = -INFINITY;
        for (int64_t j = 0; j < len; ++j) {
            int64_t base = (((int64_t)row[j / page_size] * num_kv_heads + kvh) * page_size
                            + j % page_size) * head_dim;
            double dot = 0.0;
            for (int32_t d = 0; d < head_dim; ++d)
                dot += bf16_bits_to_double(qh[d]) * cache_value(k_cache, cache_is_bf16, base + d, ks);
            s[j] = sigma * dot;
            if (s[j] > smax)
                smax = s[j];
        }
        double den = 0.0;
        for (int64_t j = 0; j < len; ++j) {
            double w = exp(s[j] - smax);
            int64_t base = (((int64_t)row[j / page_size] * num_kv_heads + kvh) * page_size
                            + j % page_size) * head_dim;
            den += w;
            for (int32_t d = 0; d < head_dim; ++d)
                o[d] += w * cache_value(v_cache, cache_is_bf16, base + d, vs);
        }
        for (int32_t d = 0; d < head_dim; ++d)
            o[d] /= den;
        free(s);
    }
}

/*
 * Multi-token decode (several new query tokens per request, as in verifying
 * speculative drafts): the pages say nothing about it; the reading taken is
 * that the n new tokens are the request's last n positions, already in the
 * cache, and that each attends causally -- query token i of request r, at
 * position L_r - n + i, attends to positions 0 .. L_r - n + i, every one of
 * them through the block table, exactly as oracle_decode_attn attends a
 * single query to positions 0 .. L_r - 1.  A query with no position to
 * attend to (L_r - n + i < 0) gets zeros; so does every query of a request
 * that oracle_decode_attn would zero (aborted, empty, longer than its table,
 * or naming a page outside [0, num_pages)).
 *   q, out   [B][n_query][Hq][D] (bf16 bits in, fp64 out).
 */
void oracle_decode_attn_multi(int32_t batch, int32_t n_query, int32_t num_q_heads,
                              int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                              int32_t num_pages, int32_t cache_is_bf16, const uint16_t *q,
                              const void *k_cache, const void *v_cache,
                              const float *k_scale, const float *v_scale,
                              const int32_t *block_table, int32_t max_pages_per_seq,
                              const int32_t *seq_lens, float softmax_scale,
                              const uint8_t *abort_flags, double *out)
{
    const int32_t group = num_q_heads / num_kv_heads;
    const double sigma = (double)softmax_scale;
    int64_t rih;
    const int64_t total = (int64_t)batch * n_query * num_q_heads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (rih = 0; rih < total; ++rih) {
        const int32_t r = (int32_t)(rih / ((int64_t)n_query * num_q_heads));
        const int32_t i = (int32_t)((rih / num_q_heads) % n_query);
        const int32_t h = (int32_t)(rih % num_q_heads);
        double *o = out + rih * head_dim;
        for (int32_t d = 0; d < head_dim; ++d)
            o[d] = 0.0;
        const int64_t len = seq_lens[r];
        if (len <= 0 || (abort_flags && abort_flags[r]))
            continue;
        const int64_t used = (len + page_size - 1) / page_size;
        if (used > max_pages_per_seq)
            continue;
        const int32_t *row = block_table + (int64_t)r * max_pages_per_seq;
        int valid = 1;
        for (int64_t p = 0; p < used; ++p)
            if (row[p] < 0 || row[p] >= num_pages)
                valid = 0;
        if (!valid)
            continue;
        /* positions this query sees: 0 .. len - n_query + i */
        const int64_t seen = len - n_query + i + 1;
        if (seen <= 0)
            continue;

        const int32_t kvh = h / group;
        const double ks = cache_is_bf16 ? 1.0 : (double)k_scale[kvh];
        const double vs = cache_is_bf16 ? 1.0 : (double)v_scale[kvh];
        const uint16_t *qh = q + rih * head_dim;
        double *s = (double *)malloc((size_t)seen * sizeof(double));
        double smax = -INFINITY;
        for (int64_t j = 0; j < seen; ++j) {
            int64_t base = (((int64_t)row[j / page_size] * num_kv_heads + kvh) * page_size
                            + j % page_size) * head_dim;
            double dot = 0.0;
            for (int32_t d = 0; d < head_dim; ++d)
                dot += bf16_bits_to_double(qh[d]) * cache_value(k_cache, cache_is_bf16, base + d, ks);
            s[j] = sigma * dot;
            if (s[j] > smax)
                smax = s[j];
        }
        double den = 0.0;
        for (int64_t j = 0; j < seen; ++j) {
            double w = exp(s[j] - smax);
            int64_t base = (((int64_t)row[j / page_size] * num_kv_heads + kvh) * page_size
                            + j % page_size) * head_dim;
            den += w;
            for (int32_t d = 0; d < head_dim; ++d)
                o[d] += w * cache_value(v_cache, cache_is_bf16, base + d, vs);
        }
        for (int32_t d = 0; d < head_dim; ++d)
            o[d] /= den;
        free(s);
    }
}

/* Threads the attention loop runs on (1 without OpenMP). */
int32_t oracle_num_threads(void)
{
#ifdef _OPENMP
    return (int32_t)omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------ prefill -> decode */

/*
 * Per-KV-head scales of a set of bf16 pages: scale[h] = amax / 448 over
 * every element of head h in the listed pages (one fp32 division), 1 when
 * amax is 0.  K and V separately.  (Prefill keeps a BF16 cache and decode an
 * FP8 one: page 1 "量化KV缓存"; these scales are what the decode pool
 * quantises the handed-over pages with.)
 */
void oracle_amax_scales(int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                        const uint16_t *k_cache, const uint16_t *v_cache,
                        const int32_t *pages, int32_t n_pages,
                        float *k_scale, float *v_scale)
{
    for (int32_t h = 0; h < num_kv_heads; ++h) {
        float ka = 0.0f, va = 0.0f;
        for (int32_t i = 0; i < n_pages; ++i) {
            int64_t base = ((int64_t)pages[i] * num_kv_heads + h) * page_size * head_dim;
            for (int64_t e = 0; e < (int64_t)page_size * head_dim; ++e) {
                float kx = fabsf(bf16_bits_to_float(k_cache[base + e]));
                float vx = fabsf(bf16_bits_to_float(v_cache[base + e]));
                if (kx > ka)
                    ka = kx;
                if (vx > va)
                    va = vx;
            }
        }
        k_scale[h] = ka > 0.0f ? ka / 448.0f : 1.0f;
        v_scale[h] = va > 0.0f ? va / 448.0f : 1.0f;
    }
}

/*
 * Quantise whole bf16 pages into e4m3 pages: element (h, slot, d) of page
 * src_pages[i] becomes encode((float)x / scale[h]) at the same position of
 * page dst_pages[i] -- the append rule applied to every slot of the page.
 */
void oracle_quantize_pages(int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                           const uint16_t *k_src, const uint16_t *v_src, const int32_t *src_pages,
                           uint8_t *k_dst, uint8_t *v_dst, const int32_t *dst_pages, int32_t n,
                           const float *k_scale, const float *v_scale)
{
    const int64_t per_head = (int64_t)page_size * head_dim;
    for (int32_t i = 0; i < n; ++i) {
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            int64_t s = ((int64_t)src_pages[i] * num_kv_heads + h) * per_head;
            int64_t d = ((int64_t)dst_pages[i] * num_kv_heads + h) * per_head;
            for (int64_t e = 0; e < per_head; ++e) {
                k_dst[d + e] = oracle_e4m3_encode(bf16_bits_to_float(k_src[s + e]) / k_scale[h]);
                v_dst[d + e] = oracle_e4m3_encode(bf16_bits_to_float(v_src[s + e]) / v_scale[h]);
            }
        }
    }
}

/*
 * INT4 weight-only product for decode (the pages' second technique: weights
 * compressed from FP8 to 4-bit integers, expanded before the multiply;
 * page 1, section "Compressing model weights"; page 2, "Model weight
 * compression to lower latency").  The pages fix no format; the reading
 * taken here:
 *   - w[n][k] = q[n][k] * s[n][k / 128]: symmetric signed 4-bit integers
 *     q in [-8, 7] (two's complement), one bf16 scale per output column n
 *     and group of 128 consecutive k;
 *   - packing: byte k / 2 of row n of W (rows of K / 2 bytes) holds q[n][k]
 *     in its low nibble for even k, in its high nibble for odd k;
 *   - y[m][n] = sum_k x[m][k] * w[n][k], x bf16.
 * fp64 throughout; one output column per outer iteration.
 */
static int oracle_int4_nibble(uint8_t byte, int64_t k)
{
    int v = (k & 1) ? (byte >> 4) : (byte & 0x0F);
    return v >= 8 ? v - 16 : v;
}

void oracle_w4a16_gemm(int32_t m, int32_t n, int32_t k, const uint16_t *x, const uint8_t *w,
                       const uint16_t *scales, double *y)
{
    const int32_t groups = k / 128;
#pragma omp parallel for schedule(static)
    for (int32_t col = 0; col < n; ++col) {
        const uint8_t *wrow = w + (int64_t)col * (k / 2);
        for (int32_t row = 0; row < m; ++row) {
            double acc = 0.0;
            for (int64_t kk = 0; kk < k; ++kk) {
                double s = (double)bf16_bits_to_float(scales[(int64_t)col * groups + kk / 128]);
                double wv = (double)oracle_int4_nibble(wrow[kk / 2], kk) * s;
                acc += (double)bf16_bits_to_float(x[(int64_t)row * k + kk]) * wv;
            }
            y[(int64_t)row * n + col] = acc;
        }
    }
}
