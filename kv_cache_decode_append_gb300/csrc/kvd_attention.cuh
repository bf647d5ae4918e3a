// kvd_attention.cuh -- split-T decode attention for sm_103a.
//
// Decode attention of the new query rows over the cached history
// ("7.1 自回归生成过程", code 1-2: scores = q.K^T / sqrt(D), softmax, .V),
// with the history-offset causal mask for chunked decode (new row i sees keys
// 0..P+i: "GPT-2缓存实测：千倍计算只快6倍", section "一个很容易漏掉的错误") and GQA
// grouping (many query heads share one KV head, so each K/V tile is read
// once per group: same page, section "GPT-2缓存要占多少显存").
//
// Decode is bound by reading K/V from HBM ("7.1", the bullets under code 1-2),
// so the kernel is a streaming reduction on the CUDA cores, not a GEMM:
//
//   * one CTA = one (sequence b, KV head h, block of RB query rows, T-split);
//   * one elected thread streams [TK, D] K and V tiles of the split, which are
//     contiguous in the [B, H_kv, T_max, D] cache, through a STAGES-deep ring
//     of shared-memory buffers with 1-D bulk (TMA) copies completing on
//     mbarriers, L2 evict-first;
//   * each warp splits into key groups of L lanes; a group owns whole keys,
//     each lane owns E = D / L head-dim elements of q (in registers,
//     pre-scaled by scale*log2 e) and of the output accumulators for all RB
//     rows; a dot product is E FMAs per lane plus a log2(L)-step xor-shuffle
//     reduction inside the group;
//   * every group keeps its own online softmax (running max m, sum l, output
//     o) in registers; the running max is only moved when a tile's max
//     exceeds it by more than 2^8, which keeps exp2 arguments <= 8 and makes
//     the rescale of o rare; o/l is unchanged by that choice;
//   * at the end the CTA merges its groups through shared memory by
//     log-sum-exp and writes either the final output (the sequence fits one
//     split) or a partial (o, m, l) for attn_merge_kernel.
//
// Masked slots (past P+i for row i, or past the split) never feed the
// arithmetic: their scores are forced to -inf and value rows past the end of
// the sequence are replaced by zeros before the weighted sum.
#pragma once

#include "kvd_device.cuh"

namespace kvd {

struct AttnArgs {
    const void *q;           // [B, H_q, N, D]
    const void *k_cache;     // [B, H_kv, T_max, D]
    const void *v_cache;     // [B, H_kv, T_max, D]
    void *out;               // [B, H_q, N, D]
    const int32_t *past_len; // [B]
    float *part_o;           // [B*H_kv][n_splits][rows_pad][D]   (unnormalised)
    float *part_ml;          // [B*H_kv][n_splits][rows_pad][2]   (max in log2 units, sum)
    uint32_t *err_word;
    int B, H_kv, T_max, N, max_past_len;
    int rows;        // query rows per (b, h): (H_q / H_kv) * N, contiguous in q and out
    int rows_pad;    // n_rowblocks * RB
    int n_rowblocks;
    int n_splits;    // T-splits per (b, h, row block)
    int split_keys;  // keys per split, a multiple of the tile
    float qscale;    // softmax scale * log2(e)
};

// Compile-time shape of one kernel variant.
template <typename T, int D, int RB> struct AttnShape {
    using Ty = Elem<T>;
    static constexpr int kRowBytes = D * Ty::kBytes;
    static constexpr int kRowChunks = kRowBytes / 16;
    // Lanes per key: 8 keeps each 8-lane shared-memory phase on one 128-byte
    // run of a row (no bank conflicts); 16 when 8 would need > 64 q registers.
    static constexpr int kL = ((kRowChunks / 8) * Ty::kPerChunk * RB <= 64) ? 8 : 16;
    static constexpr int kCpl = kRowChunks / kL;       // 16-byte chunks per lane per row
    static constexpr int kE = kCpl * Ty::kPerChunk;    // head-dim elements per lane
    static constexpr int kGpw = 32 / kL;               // key groups per warp
    static constexpr int kKpg = 4;                     // keys per group per tile
    static constexpr int kTK = (kRowBytes <= 256) ? 64 : 32;  // keys per tile
    static constexpr int kNW = kTK / (kGpw * kKpg);    // warps
    static constexpr int kThreads = kNW * 32;
    static constexpr int kKpw = kGpw * kKpg;           // keys per warp per tile
    static constexpr int kTileBytes = kTK * kRowBytes; // one of K or V
    static constexpr int kStages = (2 * kTileBytes <= 16384) ? 4 : 3;
    static constexpr int kPipeBytes = kStages * 2 * kTileBytes;
    static constexpr int kParts = kNW * kGpw;          // partial softmax states per CTA
    static constexpr int kEpiFloats = kParts * RB * (D + 3) + RB;
    static constexpr int kEpiBytes = kEpiFloats * 4;
    static constexpr int kBarOffset = ((kPipeBytes > kEpiBytes ? kPipeBytes : kEpiBytes) + 127) / 128 * 128;
    static constexpr int kSmemBytes = kBarOffset + kStages * 8;

    static_assert(kRowBytes % 16 == 0, "rows must be whole 16-byte chunks");
    static_assert(kCpl >= 1 && kRowChunks % kL == 0, "lane mapping");
    static_assert(kNW >= 1 && kTK % kKpw == 0, "tile mapping");
    static_assert(kParts * RB <= kThreads, "epilogue mapping");
};

template <typename T, int D, int RB, bool kMasked>
__device__ __forceinline__ void attn_tile(const unsigned char *Ks, const unsigned char *Vs,
                                          const float (&qv)[RB][AttnShape<T, D, RB>::kE],
                                          float (&o)[RB][AttnShape<T, D, RB>::kE], float (&m_run)[RB],
                                          float (&l_run)[RB], int warp, int grp, int j,
                                          int tile_k0, const int (&lim)[RB], int k_end)
{
    using S = AttnShape<T, D, RB>;
    using Ty = Elem<T>;
    const float kNegInf = __int_as_float(0xff800000);
    constexpr float kRescaleThreshold = 8.0f;

    float sc[S::kKpg][RB];
    uint4 raw[S::kKpg][S::kCpl];

#pragma unroll
    for (int u = 0; u < S::kKpg; ++u) {
        const int kk = warp * S::kKpw + u * S::kGpw + grp;
#pragma unroll
        for (int c = 0; c < S::kCpl; ++c)
            raw[u][c] = lds128(Ks + kk * S::kRowBytes + (c * S::kL + j) * 16);
    }
#pragma unroll
    for (int u = 0; u < S::kKpg; ++u) {
        float kf[S::kE];
#pragma unroll
        for (int c = 0; c < S::kCpl; ++c) Ty::widen(raw[u][c], kf + c * Ty::kPerChunk);
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < S::kE; ++e) acc = fmaf(qv[r][e], kf[e], acc);
            sc[u][r] = acc;
        }
    }
#pragma unroll
    for (int off = S::kL / 2; off >= 1; off /= 2) {
#pragma unroll
        for (int u = 0; u < S::kKpg; ++u)
#pragma unroll
            for (int r = 0; r < RB; ++r) sc[u][r] += __shfl_xor_sync(0xffffffffu, sc[u][r], off);
    }
    if constexpr (kMasked) {
#pragma unroll
        for (int u = 0; u < S::kKpg; ++u) {
            const int key = tile_k0 + warp * S::kKpw + u * S::kGpw + grp;
#pragma unroll
            for (int r = 0; r < RB; ++r)
                if (key >= lim[r]) sc[u][r] = kNegInf;
        }
    }

    // Online softmax, one state per key group.
    float p[S::kKpg][RB];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        float mt = sc[0][r];
#pragma unroll
        for (int u = 1; u < S::kKpg; ++u) mt = fmaxf(mt, sc[u][r]);
        if (mt > m_run[r] + kRescaleThreshold) {
            const float alpha = exp2f(m_run[r] - mt);
            l_run[r] *= alpha;
#pragma unroll
            for (int e = 0; e < S::kE; ++e) o[r][e] *= alpha;
            m_run[r] = mt;
        }
        const float mu = (m_run[r] == kNegInf) ? 0.f : m_run[r];
#pragma unroll
        for (int u = 0; u < S::kKpg; ++u) {
            p[u][r] = exp2f(sc[u][r] - mu);
            l_run[r] += p[u][r];
        }
    }

#pragma unroll
    for (int u = 0; u < S::kKpg; ++u) {
        const int kk = warp * S::kKpw + u * S::kGpw + grp;
#pragma unroll
        for (int c = 0; c < S::kCpl; ++c)
            raw[u][c] = lds128(Vs + kk * S::kRowBytes + (c * S::kL + j) * 16);
    }
#pragma unroll
    for (int u = 0; u < S::kKpg; ++u) {
        float vf[S::kE];
#pragma unroll
        for (int c = 0; c < S::kCpl; ++c) Ty::widen(raw[u][c], vf + c * Ty::kPerChunk);
        if constexpr (kMasked) {
            // Rows past the end of the split were not loaded: stale shared memory.
            if (tile_k0 + warp * S::kKpw + u * S::kGpw + grp >= k_end) {
#pragma unroll
                for (int e = 0; e < S::kE; ++e) vf[e] = 0.f;
            }
        }
#pragma unroll
        for (int r = 0; r < RB; ++r)
#pragma unroll
            for (int e = 0; e < S::kE; ++e) o[r][e] = fmaf(p[u][r], vf[e], o[r][e]);
    }
}

template <typename T, int D, int RB>
__global__ void __launch_bounds__(AttnShape<T, D, RB>::kThreads)
    attn_split_kernel(const AttnArgs a)
{
    using S = AttnShape<T, D, RB>;
    using Ty = Elem<T>;
    const float kNegInf = __int_as_float(0xff800000);
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::kBarOffset);

    const int split = blockIdx.x % a.n_splits;
    const int rest = blockIdx.x / a.n_splits;
    const int rb = rest % a.n_rowblocks;
    const int bh = rest / a.n_rowblocks;
    const int b = bh / a.H_kv;

    const int P = __ldg(a.past_len + b);
    if (!past_len_ok(P, a.N, a.T_max, a.max_past_len)) {
        if (split == 0 && rb == 0 && bh % a.H_kv == 0 && threadIdx.x == 0)
            raise_error(a.err_word, KVD_DEVERR_PAST_LEN);
        return;
    }
    const int T_b = P + a.N;
    const int k0 = split * a.split_keys;
    if (k0 >= T_b) return;  // this split lies past the end of a shorter sequence
    const int k1 = min(T_b, k0 + a.split_keys);
    const int n_valid_splits = (T_b + a.split_keys - 1) / a.split_keys;
    const int n_tiles = (k1 - k0 + S::kTK - 1) / S::kTK;

    const int tid = threadIdx.x;
    const int warp = tid / 32, lane = tid % 32;
    const int grp = lane / S::kL, j = lane % S::kL;

    const size_t row0 = (size_t)bh * a.T_max + k0;
    const unsigned char *kg = static_cast<const unsigned char *>(a.k_cache) + row0 * S::kRowBytes;
    const unsigned char *vg = static_cast<const unsigned char *>(a.v_cache) + row0 * S::kRowBytes;

    uint64_t policy = 0;
    auto issue = [&](int t) {
        const int s = t % S::kStages;
        const int nk = min(S::kTK, k1 - k0 - t * S::kTK);
        const uint32_t bytes = (uint32_t)nk * S::kRowBytes;
        unsigned char *dst = smem + s * 2 * S::kTileBytes;
        mbar_arrive_expect_tx(&bars[s], 2u * bytes);
        bulk_load_g2s(dst, kg + (size_t)t * S::kTileBytes, bytes, &bars[s], policy);
        bulk_load_g2s(dst + S::kTileBytes, vg + (size_t)t * S::kTileBytes, bytes, &bars[s], policy);
    };

    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < S::kStages; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
        policy = l2_evict_first_policy();
        for (int t = 0; t < min(n_tiles, S::kStages); ++t) issue(t);
    }
    int issued = min(n_tiles, S::kStages);  // meaningful in thread 0 only

    // q rows of this block, pre-scaled into log2 units; padding rows are 0.
    float qv[RB][S::kE];
    int lim[RB];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        const int rg = rb * RB + r;
        lim[r] = P + 1 + (rg % a.N);
        if (rg < a.rows) {
            const unsigned char *qrow =
                static_cast<const unsigned char *>(a.q) + ((size_t)bh * a.rows + rg) * S::kRowBytes;
#pragma unroll
            for (int c = 0; c < S::kCpl; ++c) {
                Ty::widen(ldg128_nc(qrow + (c * S::kL + j) * 16), &qv[r][c * Ty::kPerChunk]);
            }
#pragma unroll
            for (int e = 0; e < S::kE; ++e) qv[r][e] *= a.qscale;
        } else {
#pragma unroll
            for (int e = 0; e < S::kE; ++e) qv[r][e] = 0.f;
        }
    }

    float o[RB][S::kE];
    float m_run[RB], l_run[RB];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        m_run[r] = kNegInf;
        l_run[r] = 0.f;
#pragma unroll
        for (int e = 0; e < S::kE; ++e) o[r][e] = 0.f;
    }

    __syncthreads();  // barrier initialisation visible to every thread

    bool timed_out = false;
    int first_unwaited = n_tiles;  // first tile whose wait this thread gave up on
    for (int t = 0; t < n_tiles; ++t) {
        const int s = t % S::kStages;
        const uint32_t parity = (uint32_t)(t / S::kStages) & 1u;
        if (!timed_out && !mbar_wait_bounded(&bars[s], parity)) {
            timed_out = true;
            first_unwaited = t;
        }
        const unsigned char *Ks = smem + s * 2 * S::kTileBytes;
        const unsigned char *Vs = Ks + S::kTileBytes;
        const int tile_k0 = k0 + t * S::kTK;
        if (tile_k0 + S::kTK <= P + 1) {
            attn_tile<T, D, RB, false>(Ks, Vs, qv, o, m_run, l_run, warp, grp, j, tile_k0, lim, k1);
        } else {
            attn_tile<T, D, RB, true>(Ks, Vs, qv, o, m_run, l_run, warp, grp, j, tile_k0, lim, k1);
        }
        __syncthreads();  // every warp is done with stage s
        if (tid == 0 && !timed_out && t + S::kStages < n_tiles) {
            issue(t + S::kStages);
            issued = t + S::kStages + 1;
        }
    }
    if (__syncthreads_or(timed_out)) {  // uniform: every thread takes this branch or none
        if (timed_out) raise_error(a.err_word, KVD_DEVERR_TIMEOUT);
        // Copies still in flight must land before the CTA reuses or releases
        // its shared memory: wait for them under one overall deadline.  Only
        // thread 0 can have copies outstanding that it did not see complete.
        if (tid == 0 && timed_out) {
            const uint64_t t0 = global_timer_ns();
            for (int t = first_unwaited; t < issued; ++t) {
                const uint32_t parity = (uint32_t)(t / S::kStages) & 1u;
                while (!mbar_try_wait(&bars[t % S::kStages], parity) &&
                       global_timer_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
        __syncthreads();
    }

    // ---- merge the CTA's key groups (shared memory aliases the ring) ----
    // ep_o first: every (part, row) slice starts on a 16-byte boundary.
    float *ep_o = reinterpret_cast<float *>(smem);
    float *ep_m = ep_o + S::kParts * RB * D;
    float *ep_l = ep_m + S::kParts * RB;
    float *ep_w = ep_l + S::kParts * RB;
    float *ep_M = ep_w + S::kParts * RB;
    const int part = warp * S::kGpw + grp;
    if (j == 0) {
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            ep_m[part * RB + r] = m_run[r];
            ep_l[part * RB + r] = l_run[r];
        }
    }
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        float *dst = ep_o + (part * RB + r) * D;
#pragma unroll
        for (int c = 0; c < S::kCpl; ++c) {
            const int d0 = (c * S::kL + j) * Ty::kPerChunk;
#pragma unroll
            for (int e = 0; e < Ty::kPerChunk; e += 4)
                *reinterpret_cast<float4 *>(dst + d0 + e) =
                    make_float4(o[r][c * Ty::kPerChunk + e], o[r][c * Ty::kPerChunk + e + 1],
                                o[r][c * Ty::kPerChunk + e + 2], o[r][c * Ty::kPerChunk + e + 3]);
        }
    }
    __syncthreads();
    if (tid < S::kParts * RB) {
        const int r = tid % RB;
        float M = kNegInf;
#pragma unroll
        for (int pp = 0; pp < S::kParts; ++pp) M = fmaxf(M, ep_m[pp * RB + r]);
        const float mp = ep_m[tid];
        ep_w[tid] = (mp == kNegInf) ? 0.f : exp2f(mp - M);
        if (tid < RB) ep_M[r] = M;
    }
    __syncthreads();

    const bool single = (n_valid_splits == 1);
    for (int idx = tid; idx < RB * D; idx += S::kThreads) {
        const int r = idx / D, d = idx % D;
        const int rg = rb * RB + r;
        if (rg >= a.rows) continue;
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int pp = 0; pp < S::kParts; ++pp) {
            const float w = ep_w[pp * RB + r];
            num = fmaf(w, ep_o[(pp * RB + r) * D + d], num);
            den = fmaf(w, ep_l[pp * RB + r], den);
        }
        if (single) {
            T *out = static_cast<T *>(a.out) + ((size_t)bh * a.rows + rg) * D + d;
            Ty::store(out, num / den);
        } else {
            const size_t pidx = ((size_t)bh * a.n_splits + split) * a.rows_pad + rg;
            a.part_o[pidx * D + d] = num;
            if (d == 0) {
                a.part_ml[pidx * 2 + 0] = ep_M[r];
                a.part_ml[pidx * 2 + 1] = den;
            }
        }
    }
}

// Second pass: log-sum-exp merge of the T-splits of one query row per warp.
//   M = max_s m_s;  w_s = 2^(m_s - M);  out = sum_s w_s o_s / sum_s w_s l_s
template <typename T, int D>
__global__ void __launch_bounds__(128) attn_merge_kernel(const AttnArgs a)
{
    using Ty = Elem<T>;
    const float kNegInf = __int_as_float(0xff800000);
    constexpr int kDpl = D / 32;
    const int gw = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) / 32);
    const int lane = threadIdx.x % 32;
    if (gw >= a.B * a.H_kv * a.rows) return;
    const int bh = gw / a.rows, rg = gw % a.rows;
    const int b = bh / a.H_kv;
    const int P = __ldg(a.past_len + b);
    if (!past_len_ok(P, a.N, a.T_max, a.max_past_len)) return;  // reported by the split pass
    const int T_b = P + a.N;
    const int nv = (T_b + a.split_keys - 1) / a.split_keys;
    if (nv <= 1) return;  // the split pass wrote this row directly

    const size_t base = (size_t)bh * a.n_splits * a.rows_pad + rg;
    const size_t stride = a.rows_pad;
    float M = kNegInf;
    for (int s = lane; s < nv; s += 32) M = fmaxf(M, a.part_ml[(base + s * stride) * 2]);
#pragma unroll
    for (int off = 16; off >= 1; off /= 2) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

    float acc[kDpl];
#pragma unroll
    for (int k = 0; k < kDpl; ++k) acc[k] = 0.f;
    float den = 0.f;
    for (int s = 0; s < nv; ++s) {
        const size_t pidx = base + s * stride;
        const float ms = a.part_ml[pidx * 2];
        const float w = (ms == kNegInf) ? 0.f : exp2f(ms - M);
        den = fmaf(w, a.part_ml[pidx * 2 + 1], den);
        const float *po = a.part_o + pidx * D + lane * kDpl;
        if constexpr (kDpl == 4) {
            const float4 v = *reinterpret_cast<const float4 *>(po);
            acc[0] = fmaf(w, v.x, acc[0]);
            acc[1] = fmaf(w, v.y, acc[1]);
            acc[2] = fmaf(w, v.z, acc[2]);
            acc[3] = fmaf(w, v.w, acc[3]);
        } else {
#pragma unroll
            for (int k = 0; k < kDpl; ++k) acc[k] = fmaf(w, po[k], acc[k]);
        }
    }
    T *out = static_cast<T *>(a.out) + ((size_t)bh * a.rows + rg) * D + lane * kDpl;
#pragma unroll
    for (int k = 0; k < kDpl; ++k) Ty::store(out + k, acc[k] / den);
}

// Launch facts of one compiled variant, for the host planner.
struct AttnVariant {
    const void *split_fn;
    const void *merge_fn;
    int threads;
    int smem_bytes;
    int tile_keys;
    int rows_per_block;
};

template <typename T, int D, int RB> AttnVariant make_variant()
{
    using S = AttnShape<T, D, RB>;
    AttnVariant v;
    v.split_fn = reinterpret_cast<const void *>(&attn_split_kernel<T, D, RB>);
    v.merge_fn = reinterpret_cast<const void *>(&attn_merge_kernel<T, D>);
    v.threads = S::kThreads;
    v.smem_bytes = S::kSmemBytes;
    v.tile_keys = S::kTK;
    v.rows_per_block = RB;
    return v;
}

template <typename T, int D> bool pick_rb(int RB, AttnVariant *v)
{
    switch (RB) {
    case 1: *v = make_variant<T, D, 1>(); return true;
    case 2: *v = make_variant<T, D, 2>(); return true;
    case 4: *v = make_variant<T, D, 4>(); return true;
    case 8: *v = make_variant<T, D, 8>(); return true;
    default: return false;
    }
}

template <typename T> bool pick_variant(int D, int RB, AttnVariant *v)
{
    switch (D) {
    case 64: return pick_rb<T, 64>(RB, v);
    case 128: return pick_rb<T, 128>(RB, v);
    default: return false;
    }
}

// Defined in kvd_attn_f32.cu / kvd_attn_bf16.cu (one translation unit each).
bool attn_variant_f32(int D, int RB, AttnVariant *v);
bool attn_variant_bf16(int D, int RB, AttnVariant *v);

}  // namespace kvd
