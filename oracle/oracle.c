/*
 * oracle.c -- the plain CPU oracle for the KV-cache decode step.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke
 * check and the CPU-baseline leg of the benchmark load this file's library.
 * It shares no code, header, table or constant with the CUDA path under
 * kv_cache_decode_append_gb300/csrc, and includes none of it.
 *
 * Everything here is the plain definition, in double precision, with plain
 * loops and no blocking, fusion or reordering:
 *
 *   oracle_cache_bytes       the KV-cache size formula
 *                            [openai-hub.com/news/2435 "GPT-2缓存实测：千倍计算只快6倍",
 *                             section "GPT-2缓存要占多少显存" (how much memory the
 *                             GPT-2 cache takes), the size formula and its table]
 *   oracle_append            the cache update: the new K/V of N tokens goes to
 *                            slots P..P+N-1 of the time axis, i.e. the result of
 *                            concatenating old and new along the sequence axis
 *                            [gitcode.csdn.net miniONNXRuntime article, section
 *                             "Decode Shape 示例" (decode shape example);
 *                             openai-hub.com/news/2435, section "一个很容易漏掉的错误"
 *                             (an easy-to-miss error), the data-flow sketch]
 *                            written in place into preallocated slots
 *                            [jennyma11.github.io/infra/ch07-01 "7.1 自回归生成过程",
 *                             section "Decode 阶段", the note under code 1-2]
 *   oracle_decode_attention  scores = q.K^T * scale, softmax, .V for each new
 *                            query row i, over keys 0..P+i (the causal mask
 *                            with history offset)
 *                            [jennyma11.github.io/infra/ch07-01, code 1-2
 *                             "Decode 单步到底在算什么";
 *                             openai-hub.com/news/2435, section
 *                             "一个很容易漏掉的错误", the offset-mask paragraph]
 *   oracle_paged_append, oracle_paged_decode_attention
 *                            the same two operations on a paged cache: the
 *                            tokens of a sequence live in fixed-size pages
 *                            found through a per-sequence block table, and
 *                            new tokens are written into their page slots in
 *                            place [jennyma11.github.io/infra/ch07-01, the note
 *                            under code 1-2 (real engines write by slot, with
 *                            PagedAttention); openai-hub.com/news/2435, section
 *                            "显存测量最容易被分配器误导" (the allocator misleads
 *                            memory measurements), which names PagedAttention as
 *                            the remedy for reallocation]; defined here as the
 *                            contiguous operations applied to the cache gathered
 *                            through the block table
 *   oracle_append_e4m3, oracle_decode_attention_e4m3
 *                            the same two operations with an 8-bit floating-point
 *                            (E4M3) cache and per-tensor K and V scales: the pages
 *                            name FP8 among the cache precisions used in serving
 *                            and say quantization pays most at decode
 *                            [openai-hub.com/news/2435, section "实验到底测了什么"
 *                             (what the experiment measured), the paragraph after the
 *                             configuration table; jennyma11.github.io/infra/ch07-01,
 *                             section "Decode 阶段"];
 *                            they give no format, so the format and the scaling
 *                            are a reading (see the design notes)
 *   oracle_full_causal_attention
 *                            the uncached route: ordinary causal attention of
 *                            T query rows over T keys (row t sees keys 0..t)
 *                            [gitcode.csdn.net miniONNXRuntime article, section
 *                             "Baseline 重算开销" (baseline recompute cost);
 *                             openai-hub.com/news/2435, section "正确性先于性能",
 *                             test 2: cached vs uncached last-position outputs]
 *
 * Readings taken where the pages are silent (the same readings are listed in
 * the design notes of the repository):
 *   - layout [B, H, T, D] row-major for caches, [B, H, N, D] for q / new K/V / out;
 *   - GQA: query head hq uses KV head hq / (H_q / H_kv) (consecutive query
 *     heads share one KV head);
 *   - past_len[b] is the number of cached tokens BEFORE the append;
 *   - bf16 values are widened exactly (bf16 bits << 16 is the fp32 value);
 *     fp16 values exactly from the IEEE binary16 encoding; E4M3 codes (an
 *     8-bit cache format) exactly from their encoding, times a per-tensor scale.
 *
 * Paged layout (a reading: the pages do not fix one): pages are
 * [num_pages, H_kv, page_size, D] row-major; logical page j of sequence b is
 * physical page block_table[b * max_pages + j]; token t of (b, h) is row
 * t % page_size of head h in logical page t / page_size.
 *
 * Status codes: 0 = ok, 1 = invalid argument, 2 = capacity (P + N > T_max or
 * P < 0 for some sequence; that sequence is left untouched), 3 = a block-table
 * entry that a sequence needs is outside [0, num_pages) (that sequence is left
 * untouched / its output rows are NaN).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F16 = 2, ORACLE_E4M3 = 3 };

static int elem_bytes(int dtype)
{
    if (dtype == ORACLE_F32) return 4;
    if (dtype == ORACLE_BF16 || dtype == ORACLE_F16) return 2;
    return dtype == ORACLE_E4M3 ? 1 : 0;
}

/* An 8-bit E4M3 value (1 sign, 4 exponent, 3 fraction bits, bias 7; no
 * infinities, exponent 15 with fraction 7 is NaN, the largest finite value is
 * 448) as a double: normal numbers (8 + fraction) * 2^(exponent - 10),
 * subnormals fraction * 2^-9. */
static double e4m3_bits_to_double(uint8_t c)
{
    const int sign = c >> 7, expo = (c >> 3) & 0xf, frac = c & 0x7;
    double v;
    if (expo == 15 && frac == 7)
        v = NAN;
    else if (expo == 0)
        v = ldexp((double)frac, -9);
    else
        v = ldexp((double)(8 + frac), expo - 10);
    return sign ? -v : v;
}

/* An IEEE 754 binary16 value (1 sign, 5 exponent, 10 fraction bits, bias 15)
 * as a double, exactly: normal numbers are (1024 + fraction) * 2^(exponent - 25),
 * subnormals fraction * 2^-24, exponent 31 is infinity (fraction 0) or NaN. */
static double half_bits_to_double(uint16_t h)
{
    const int sign = h >> 15, expo = (h >> 10) & 0x1f, frac = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24);
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), expo - 25);
    return sign ? -v : v;
}

/* One stored element widened to double.  A bf16 value is the upper half of
 * an IEEE fp32 value, so shifting its 16 bits up gives that fp32 exactly. */
static double load_elem(const void *base, size_t idx, int dtype)
{
    if (dtype == ORACLE_F32) {
        return (double)((const float *)base)[idx];
    }
    if (dtype == ORACLE_F16) {
        return half_bits_to_double(((const uint16_t *)base)[idx]);
    }
    if (dtype == ORACLE_E4M3) {
        return e4m3_bits_to_double(((const uint8_t *)base)[idx]);
    }
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* bytes = 2 (K and V) x layers x KV heads x head dim x tokens x batch x bytes/elem */
unsigned long long oracle_cache_bytes(long long L, long long B, long long H_kv,
                                      long long D, long long T, long long bytes_per_elem)
{
    return (unsigned long long)(2LL * L * H_kv * D * T * B * bytes_per_elem);
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Append: for every sequence b, KV head h and new token i < N,
 *   cache[b, h, past_len[b] + i, :] = new[b, h, i, :]   (bit copy, K and V).
 * Slots outside [past_len[b], past_len[b] + N) are not touched.
 */
int oracle_append(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                  const int32_t *past_len, int B, int H_kv, int T_max, int D, int N,
                  int dtype)
{
    const int s = elem_bytes(dtype);
    if (!k_cache || !v_cache || !k_new || !v_new || !past_len || s == 0 ||
        B < 0 || H_kv <= 0 || T_max <= 0 || D <= 0 || N <= 0)
        return 1;
    int status = 0;
    const size_t row = (size_t)D * (size_t)s;
    for (int b = 0; b < B; ++b) {
        const long long P = past_len[b];
        if (P < 0 || P + N > T_max) {
            status = 2;
            continue;
        }
        for (int h = 0; h < H_kv; ++h) {
            for (int i = 0; i < N; ++i) {
                const size_t dst = (((size_t)b * H_kv + h) * (size_t)T_max + (size_t)(P + i)) * row;
                const size_t src = (((size_t)b * H_kv + h) * (size_t)N + (size_t)i) * row;
                memcpy((char *)k_cache + dst, (const char *)k_new + src, row);
                memcpy((char *)v_cache + dst, (const char *)v_new + src, row);
            }
        }
    }
    return status;
}

/*
 * Decode attention over an already-appended cache.  For sequence b, query
 * head hq, new-token row i (0 <= i < N), with g = H_q / H_kv and h = hq / g:
 *
 *   visible keys  j = 0 .. past_len[b] + i          (past_len[b] + i + 1 keys)
 *   s_j  = scale * sum_d q[b,hq,i,d] * K[b,h,j,d]
 *   m    = max_j s_j
 *   w_j  = exp(s_j - m)
 *   out[b,hq,i,d] = sum_j w_j * V[b,h,j,d] / sum_j w_j
 *
 * out is double [B, H_q, N, D].  Rows of a sequence with an invalid
 * past_len (P < 0 or P + N > T_max) are set to NaN and status 2 is returned.
 */
static int decode_attention_impl(const void *q, const void *k_cache, const void *v_cache,
                                 double *out, const int32_t *past_len, int B, int H_q,
                                 int H_kv, int T_max, int D, int N, double scale, int dtype,
                                 int kv_dtype, double k_scale, double v_scale)
{
    if (!q || !k_cache || !v_cache || !out || !past_len || elem_bytes(dtype) == 0 ||
        elem_bytes(kv_dtype) == 0 ||
        B < 0 || H_q <= 0 || H_kv <= 0 || H_q % H_kv != 0 || T_max <= 0 || D <= 0 || N <= 0)
        return 1;
    const int g = H_q / H_kv;
    int status = 0;
    for (int b = 0; b < B; ++b) {
        const long long P = past_len[b];
        if (P < 0 || P + N > T_max) status = 2;
    }

#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        for (int hq = 0; hq < H_q; ++hq) {
            const long long P = past_len[b];
            const int h = hq / g;
            double *scores = (double *)malloc(sizeof(double) * (size_t)T_max);
            for (int i = 0; i < N; ++i) {
                double *o = out + (((size_t)b * H_q + hq) * (size_t)N + (size_t)i) * (size_t)D;
                if (P < 0 || P + N > T_max || scores == NULL) {
                    for (int d = 0; d < D; ++d) o[d] = NAN;
                    continue;
                }
                const size_t q_row = (((size_t)b * H_q + hq) * (size_t)N + (size_t)i) * (size_t)D;
                const size_t kv_head = ((size_t)b * H_kv + h) * (size_t)T_max;
                const long long n_keys = P + i + 1; /* keys 0..P+i */

                double m = -INFINITY;
                for (long long j = 0; j < n_keys; ++j) {
                    const size_t k_row = (kv_head + (size_t)j) * (size_t)D;
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d)
                        dot += load_elem(q, q_row + d, dtype) * (k_scale * load_elem(k_cache, k_row + d, kv_dtype));
                    scores[j] = scale * dot;
                    if (scores[j] > m) m = scores[j];
                }

                double wsum = 0.0;
                for (int d = 0; d < D; ++d) o[d] = 0.0;
                for (long long j = 0; j < n_keys; ++j) {
                    const double w = exp(scores[j] - m);
                    const size_t v_row = (kv_head + (size_t)j) * (size_t)D;
                    wsum += w;
                    for (int d = 0; d < D; ++d) o[d] += w * (v_scale * load_elem(v_cache, v_row + d, kv_dtype));
                }
                for (int d = 0; d < D; ++d) o[d] /= wsum;
            }
            free(scores);
        }
    }
    return status;
}

int oracle_decode_attention(const void *q, const void *k_cache, const void *v_cache,
                            double *out, const int32_t *past_len, int B, int H_q,
                            int H_kv, int T_max, int D, int N, double scale, int dtype)
{
    return decode_attention_impl(q, k_cache, v_cache, out, past_len, B, H_q, H_kv, T_max, D, N,
                                 scale, dtype, dtype, 1.0, 1.0);
}

/*
 * The uncached route for one head: ordinary causal self-attention of T rows.
 * qf, kf, vf, out are double [T, D] row-major; row t sees keys 0..t:
 *   out[t, :] = sum_{j<=t} exp(s_tj - m_t) v_j / sum_{j<=t} exp(s_tj - m_t),
 *   s_tj = scale * q_t . k_j.
 */
int oracle_full_causal_attention(const double *qf, const double *kf, const double *vf,
                                 double *out, int T, int D, double scale)
{
    if (!qf || !kf || !vf || !out || T <= 0 || D <= 0) return 1;
    double *scores = (double *)malloc(sizeof(double) * (size_t)T);
    if (!scores) return 1;
    for (int t = 0; t < T; ++t) {
        double m = -INFINITY;
        for (int j = 0; j <= t; ++j) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += qf[(size_t)t * D + d] * kf[(size_t)j * D + d];
            scores[j] = scale * dot;
            if (scores[j] > m) m = scores[j];
        }
        double wsum = 0.0;
        for (int d = 0; d < D; ++d) out[(size_t)t * D + d] = 0.0;
        for (int j = 0; j <= t; ++j) {
            const double w = exp(scores[j] - m);
            wsum += w;
            for (int d = 0; d < D; ++d) out[(size_t)t * D + d] += w * vf[(size_t)j * D + d];
        }
        for (int d = 0; d < D; ++d) out[(size_t)t * D + d] /= wsum;
    }
    free(scores);
    return 0;
}

/* Physical page of token t of sequence b, or -1 when the entry is out of range. */
static long long paged_page(const int32_t *block_table, int b, long long t, int page_size,
                            int max_pages, int num_pages)
{
    const long long j = t / page_size;
    if (j < 0 || j >= max_pages) return -1;
    const long long page = block_table[(size_t)b * (size_t)max_pages + (size_t)j];
    if (page < 0 || page >= num_pages) return -1;
    return page;
}

/* Whether every page holding tokens 0 .. n_tok-1 of sequence b is valid. */
static int paged_pages_ok(const int32_t *block_table, int b, long long n_tok, int page_size,
                          int max_pages, int num_pages)
{
    for (long long t = 0; t < n_tok; t += page_size)
        if (paged_page(block_table, b, t, page_size, max_pages, num_pages) < 0) return 0;
    return 1;
}

/*
 * Paged append: for every sequence b, KV head h and new token i < N, with
 * t = past_len[b] + i,
 *   pages[page(b, t), h, t % page_size, :] = new[b, h, i, :]   (bit copy, K and V).
 * A sequence whose tokens do not fit (t >= max_pages * page_size) or whose
 * pages for tokens 0 .. past_len[b] + N - 1 are not all valid is left untouched.
 */
int oracle_paged_append(void *k_pages, void *v_pages, const void *k_new, const void *v_new,
                        const int32_t *block_table, const int32_t *past_len, int B, int H_kv,
                        int D, int N, int page_size, int max_pages, int num_pages, int dtype)
{
    const int s = elem_bytes(dtype);
    if (!k_pages || !v_pages || !k_new || !v_new || !block_table || !past_len || s == 0 ||
        B < 0 || H_kv <= 0 || D <= 0 || N <= 0 || page_size <= 0 || max_pages <= 0 || num_pages <= 0)
        return 1;
    int status = 0;
    const size_t row = (size_t)D * (size_t)s;
    const long long capacity = (long long)max_pages * page_size;
    for (int b = 0; b < B; ++b) {
        const long long P = past_len[b];
        if (P < 0 || P + N > capacity) {
            status = 2;
            continue;
        }
        if (!paged_pages_ok(block_table, b, P + N, page_size, max_pages, num_pages)) {
            if (status == 0) status = 3;
            continue;
        }
        for (int h = 0; h < H_kv; ++h) {
            for (int i = 0; i < N; ++i) {
                const long long t = P + i;
                const long long page = paged_page(block_table, b, t, page_size, max_pages, num_pages);
                const size_t dst = (((size_t)page * H_kv + h) * (size_t)page_size + (size_t)(t % page_size)) * row;
                const size_t src = (((size_t)b * H_kv + h) * (size_t)N + (size_t)i) * row;
                memcpy((char *)k_pages + dst, (const char *)k_new + src, row);
                memcpy((char *)v_pages + dst, (const char *)v_new + src, row);
            }
        }
    }
    return status;
}

/*
 * Paged decode attention: gather the keys and values of tokens
 * 0 .. past_len[b] + N - 1 of every (b, h) from their pages into a contiguous
 * [B, H_kv, max_pages * page_size, D] cache and apply oracle_decode_attention
 * to it.  Rows of a sequence with an invalid past_len are NaN (status 2); rows
 * of a sequence with an invalid page are NaN (status 3).
 */
int oracle_paged_decode_attention(const void *q, const void *k_pages, const void *v_pages,
                                  double *out, const int32_t *block_table, const int32_t *past_len,
                                  int B, int H_q, int H_kv, int D, int N, int page_size,
                                  int max_pages, int num_pages, double scale, int dtype)
{
    const int s = elem_bytes(dtype);
    if (!q || !k_pages || !v_pages || !out || !block_table || !past_len || s == 0 || B < 0 ||
        H_q <= 0 || H_kv <= 0 || H_q % H_kv != 0 || D <= 0 || N <= 0 || page_size <= 0 ||
        max_pages <= 0 || num_pages <= 0)
        return 1;
    const long long T = (long long)max_pages * page_size;
    const size_t row = (size_t)D * (size_t)s;
    const size_t head_bytes = (size_t)T * row;
    char *kc = (char *)calloc((size_t)B * H_kv, head_bytes);
    char *vc = (char *)calloc((size_t)B * H_kv, head_bytes);
    int32_t *pl = (int32_t *)malloc(sizeof(int32_t) * (size_t)(B > 0 ? B : 1));
    if (!kc || !vc || !pl) {
        free(kc);
        free(vc);
        free(pl);
        return 1;
    }
    int bad_pages = 0;
    pl[0] = 0;
    for (int b = 0; b < B; ++b) {
        const long long P = past_len[b];
        pl[b] = past_len[b];
        if (P < 0 || P + N > T) continue; /* reported as capacity below */
        if (!paged_pages_ok(block_table, b, P + N, page_size, max_pages, num_pages)) {
            pl[b] = -1; /* makes the contiguous oracle mark the rows NaN */
            bad_pages = 1;
            continue;
        }
        for (int h = 0; h < H_kv; ++h) {
            for (long long t = 0; t < P + N; ++t) {
                const long long page = paged_page(block_table, b, t, page_size, max_pages, num_pages);
                const size_t src = (((size_t)page * H_kv + h) * (size_t)page_size + (size_t)(t % page_size)) * row;
                const size_t dst = (((size_t)b * H_kv + h) * (size_t)T + (size_t)t) * row;
                memcpy(kc + dst, (const char *)k_pages + src, row);
                memcpy(vc + dst, (const char *)v_pages + src, row);
            }
        }
    }
    int status = oracle_decode_attention(q, kc, vc, out, pl, B, H_q, H_kv, (int)T, D, N, scale, dtype);
    if (status != 1) status = bad_pages ? 3 : 0;
    /* a capacity violation of some sequence takes precedence, as in the contiguous oracle */
    for (int b = 0; b < B && status != 1; ++b) {
        const long long P = past_len[b];
        if (P < 0 || P + N > T) status = 2;
    }
    free(kc);
    free(vc);
    free(pl);
    return status;
}

/* The dtype's stored values widened to double (test hook for the widening pins). */
int oracle_widen(const void *src, double *dst, long long n, int dtype)
{
    if (!src || !dst || n < 0 || elem_bytes(dtype) == 0) return 1;
    for (long long i = 0; i < n; ++i) dst[i] = load_elem(src, (size_t)i, dtype);
    return 0;
}

/*
 * E4M3 quantization of one fp32 value: the nearest finite E4M3 value, ties to
 * the even code (the one whose fraction ends in 0), magnitudes beyond 448
 * saturated to 448 (the conversion saturates instead of overflowing), NaN
 * kept NaN.  Written as a search over the 127 non-negative finite codes, in
 * increasing order of value.
 */
static uint8_t e4m3_from_float(float x)
{
    if (isnan(x)) return 0x7f;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double a = fabs((double)x);
    int best = 0;
    double best_err = a;  /* code 0 is +0 */
    for (int c = 1; c < 0x7f; ++c) {
        const double err = fabs(e4m3_bits_to_double((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(sign | best);
}

/*
 * Append with an E4M3 cache: as oracle_append, with the stored code of each
 * new element x (new_dtype: fp32, bf16 or fp16) being the quantization of the
 * fp32 quotient x / scale (k_scale for K, v_scale for V), divided in fp32.
 */
int oracle_append_e4m3(uint8_t *k_cache, uint8_t *v_cache, const void *k_new, const void *v_new,
                       const int32_t *past_len, int B, int H_kv, int T_max, int D, int N,
                       int new_dtype, float k_scale, float v_scale)
{
    if (!k_cache || !v_cache || !k_new || !v_new || !past_len || elem_bytes(new_dtype) == 0 ||
        new_dtype == ORACLE_E4M3 || B < 0 || H_kv <= 0 || T_max <= 0 || D <= 0 || N <= 0 ||
        !(k_scale > 0.0f) || !(v_scale > 0.0f))
        return 1;
    int status = 0;
    for (int b = 0; b < B; ++b) {
        const long long P = past_len[b];
        if (P < 0 || P + N > T_max) {
            status = 2;
            continue;
        }
        for (int h = 0; h < H_kv; ++h) {
            for (int i = 0; i < N; ++i) {
                const size_t dst = (((size_t)b * H_kv + h) * (size_t)T_max + (size_t)(P + i)) * (size_t)D;
                const size_t src = (((size_t)b * H_kv + h) * (size_t)N + (size_t)i) * (size_t)D;
                for (int d = 0; d < D; ++d) {
                    const float kx = (float)load_elem(k_new, src + d, new_dtype);
                    const float vx = (float)load_elem(v_new, src + d, new_dtype);
                    k_cache[dst + d] = e4m3_from_float(kx / k_scale);
                    v_cache[dst + d] = e4m3_from_float(vx / v_scale);
                }
            }
        }
    }
    return status;
}

/*
 * Decode attention over an E4M3 cache: as oracle_decode_attention with key j
 * = k_scale * K[b,h,j,:] and value j = v_scale * V[b,h,j,:] (the stored codes
 * decoded exactly); q in q_dtype (fp32, bf16 or fp16).
 */
int oracle_decode_attention_e4m3(const void *q, const uint8_t *k_cache, const uint8_t *v_cache,
                                 double *out, const int32_t *past_len, int B, int H_q, int H_kv,
                                 int T_max, int D, int N, double scale, int q_dtype, double k_scale,
                                 double v_scale)
{
    if (q_dtype == ORACLE_E4M3) return 1;
    return decode_attention_impl(q, k_cache, v_cache, out, past_len, B, H_q, H_kv, T_max, D, N, scale,
                                 q_dtype, ORACLE_E4M3, k_scale, v_scale);
}

/* E4M3 codes of n fp32 values (test hook for the quantization pins). */
int oracle_quantize_e4m3(const float *src, uint8_t *dst, long long n)
{
    if (!src || !dst || n < 0) return 1;
    for (long long i = 0; i < n; ++i) dst[i] = e4m3_from_float(src[i]);
    return 0;
}
