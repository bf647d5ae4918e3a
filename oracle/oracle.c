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
 *   - bf16 values are widened exactly (bf16 bits << 16 is the fp32 value).
 *
 * Status codes: 0 = ok, 1 = invalid argument, 2 = capacity (P + N > T_max or
 * P < 0 for some sequence; that sequence is left untouched).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

static int elem_bytes(int dtype)
{
    return dtype == ORACLE_F32 ? 4 : (dtype == ORACLE_BF16 ? 2 : 0);
}

/* One stored element widened to double.  A bf16 value is the upper half of
 * an IEEE fp32 value, so shifting its 16 bits up gives that fp32 exactly. */
static double load_elem(const void *base, size_t idx, int dtype)
{
    if (dtype == ORACLE_F32) {
        return (double)((const float *)base)[idx];
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
int oracle_decode_attention(const void *q, const void *k_cache, const void *v_cache,
                            double *out, const int32_t *past_len, int B, int H_q,
                            int H_kv, int T_max, int D, int N, double scale, int dtype)
{
    if (!q || !k_cache || !v_cache || !out || !past_len || elem_bytes(dtype) == 0 ||
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
                        dot += load_elem(q, q_row + d, dtype) * load_elem(k_cache, k_row + d, dtype);
                    scores[j] = scale * dot;
                    if (scores[j] > m) m = scores[j];
                }

                double wsum = 0.0;
                for (int d = 0; d < D; ++d) o[d] = 0.0;
                for (long long j = 0; j < n_keys; ++j) {
                    const double w = exp(scores[j] - m);
                    const size_t v_row = (kv_head + (size_t)j) * (size_t)D;
                    wsum += w;
                    for (int d = 0; d < D; ++d) o[d] += w * load_elem(v_cache, v_row + d, dtype);
                }
                for (int d = 0; d < D; ++d) o[d] /= wsum;
            }
            free(scores);
        }
    }
    return status;
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
