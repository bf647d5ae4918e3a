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
// so the kernel is a streaming reduction on the CUDA cores, not a GEMM.
//
// Work decomposition (flash-decoding split over T, balanced statically):
//   * a "sequence-head" u is one (sequence b, KV head h, block of RB query
//     rows); its query rows are g*N rows (g query heads of the group x N new
//     tokens), contiguous in q and out; its keys 0..P_b+N-1 form
//     ceil((P_b+N)/TK) tiles of TK keys;
//   * every CTA reads past_len, forms the prefix sum over all sequence-heads
//     of their cost in units (tiles plus a fixed overhead per head for the
//     piece boundary), and takes an equal contiguous range of that flattened
//     list (the grid is SMs x resident CTAs; with fewer units than CTAs only
//     the first n_units CTAs work): every CTA gets the same work whatever the
//     mix of sequence lengths, with no atomics and a split that depends only
//     on the inputs;
//   * thread 0 walks the range and streams each tile's [TK, D] K and V rows
//     (contiguous in the [B, H_kv, T_max, D] cache), plus the q rows at the
//     start of each sequence-head, into a STAGES-deep shared-memory ring with
//     1-D bulk (TMA) copies completing on "full" mbarriers (L2 evict-first);
//     each warp releases a slot on its "empty" mbarrier when done with it, so
//     warps drift independently and the CTA only synchronises where a piece
//     ends;
//   * the warps split into key groups of L lanes; a group owns whole keys,
//     each lane owns E = D / L head-dim elements of q (registers, pre-scaled
//     by scale*log2 e) and of the output accumulators for all RB rows, as
//     fp32 pairs for the packed f32x2 FMA; a dot product is E/2 packed FMAs
//     per lane plus a log2(L)-step xor-shuffle reduction inside the group; every group keeps its own online softmax (running
//     max m, sum l, output o); the running max only moves when a tile's max
//     exceeds it by more than 2^8, which keeps exp2 arguments <= 8 and makes
//     the rescale of o rare (o/l is unchanged by that choice);
//   * where the range leaves a sequence-head the warps merge their groups by
//     log-sum-exp (shuffles) and then, between two CTA barriers, across warps
//     (shared memory): the output is written directly when the sequence-head
//     lies inside one CTA's range, else the piece goes to a partial slot (a
//     CTA holds at most two: the head it continues and the head it starts);
//   * the pieces of split heads are merged by log-sum-exp in one of two ways,
//     chosen per call by the host: (a) in the kernel: after its range, a CTA
//     counts its pieces on their heads' tickets (one acquire-release atomic
//     per piece, no waiting) and the CTA that completes a head's count merges
//     its pieces and resets the ticket to zero; or (b) by attn_merge_kernel, a
//     second launch that starts early (programmatic dependent launch) and
//     merges once this grid has finished.  (a) saves the second launch and
//     wins on short ranges; on long ranges (tens of tiles per CTA) the tail
//     merge of the last CTA to finish costs more than (b), measured on GB300.
//     Counting only once the range is done keeps memory fences out of the
//     streaming phase, where a fence stalled for microseconds behind the
//     CTA's in-flight bulk copies.
//
// Masked slots (past P+i for row i, or past the end of the sequence) never
// feed the arithmetic: their scores are forced to -inf and value rows past
// the end of the sequence are replaced by zeros before the weighted sum.
#pragma once

#include <type_traits>

#include "kvd_device.cuh"

namespace kvd {

// Kernel arguments, passed by value.  Kept at 128 bytes: on GB300 a larger
// parameter block (even one more int) measured about 1 us slower per launch
// of the long-context layer, so mode-specific fields share slots.
struct AttnArgs {
    const void *q;           // [B, H_q, N, D]
    const void *k_cache;     // contiguous [B, H_kv, T_max, D], or pages [num_pages, H_kv, page_size, D]
    const void *v_cache;     // same layout as k_cache
    void *out;               // [B, H_q, N, D]
    const int32_t *past_len; // [B]
    const void *k_new;       // [B, H_kv, N, D]: fused step only (append inside)
    const void *v_new;       // [B, H_kv, N, D]: fused step only
    float *part;             // [grid][2][RB][D + 4]: piece partials o (unnormalised), m (log2 units), l
    void *merge_state;       // merge pass: int2 [B*H_kv*n_rowblocks] (first CTA, CTAs) per
                             // sequence-head; in-kernel merge: int tickets, the same count (pieces
                             // counted so far; zero between calls: the merging CTA resets its ticket)
    uint32_t *err_word;
    union {
        const int32_t *block_table;  // paged: [B, T_max >> page_shift] physical page of each logical page
        float2 kv_scale;             // E4M3 cache: (k_scale, v_scale), stored code = value / scale
    };
    int B, H_kv, T_max, N, max_past_len;  // paged: T_max = pages per sequence x page_size
    int rows;         // query rows per (b, h): (H_q / H_kv) * N, contiguous in q and out
    int n_rowblocks;  // ceil(rows / RB)
    float qscale;     // softmax scale * log2(e)
    int num_pages;    // paged only: pages in the pool
    short page_shift; // paged only: log2(page_size); page_size is a multiple of the tile keys
    short flags;      // kArgEarly, kArgHistoryStable
};
// AttnArgs::flags: the CTAs let the next kernel on the stream launch as soon
// as they start (before their own griddepcontrol.wait), so that its CTAs take
// free SM slots early and, with a stable history, start their loads.  Chosen
// for small layers, where a launch's fixed latencies are a large part of it.
constexpr short kArgEarly = 1;
// AttnArgs::flags (with kArgEarly): the caller guarantees that no work
// queued before this call on the stream writes past_len or the cache rows
// below past_len.  The CTAs then read past_len and fill their ring with K/V
// tiles before griddepcontrol.wait; the q rows (second arrival on each full
// barrier), the new rows of a fused step and every write wait for it.
constexpr short kArgHistoryStable = 2;
#ifdef KVD_TIMEOUT_TEST
// Test builds only: the first tile fill of every CTA expects 16 bytes more
// than its copies bring, so that stage never completes and every wait for it
// runs out (kWaitLimitNs is 2 ms in those builds).  Nothing is left in flight.
constexpr short kArgTestStall = 4;
#endif

// How RangeWalk::fill arms a stage's full barrier.
enum FillMode {
    kFillOne = 0,     // one arrival: K/V (+ q) bytes
    kFillKvOnly = 1,  // first of two arrivals, K/V bytes only; the q rows are issued by issue_pending
    kFillTwo = 2,     // both arrivals at once: K/V (+ q) bytes, then a plain arrival
};
static_assert(sizeof(AttnArgs) == 128, "keep the kernel parameter block at 128 bytes");


// Compile-time shape of one kernel variant: q / out elements T, cache
// elements C (T, or E4M3 codes with bf16 q).
template <typename T, int D, int RB, typename C = T> struct AttnShape {
    using Ty = Elem<C>;   // cache rows (the K/V tiles)
    using Tq = Elem<T>;   // q, new K/V and out rows
    static constexpr bool kTma = false;  // tiles arrive by 1-D bulk copies
    static constexpr bool kQInRing = true;  // a piece's q rows ride with its first tile
    static constexpr int kRB = RB;
    static constexpr int kRowBytes = D * Ty::kBytes;   // one cache row
    static constexpr int kQRowBytes = D * Tq::kBytes;  // one q / new K/V / out row
    static constexpr int kQChunks = Ty::kPerChunk * Tq::kBytes / 16;  // q chunks per cache chunk
    static constexpr int kRowChunks = kRowBytes / 16;
    // Lanes per key: 8 keeps each 8-lane shared-memory phase on one 128-byte
    // run of a row (no bank conflicts); 16 when 8 would need > 64 q registers;
    // never more than a row's chunks (64-byte E4M3 rows: 4).
    static constexpr int kLw = ((kRowChunks / 8) * Ty::kPerChunk * RB <= 64) ? 8 : 16;
    static constexpr int kL = kLw < kRowChunks ? kLw : kRowChunks;
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
    static constexpr int kQSlotBytes = RB * kQRowBytes;
    // Cost of a piece boundary in tile units for the static split (a sweep
    // over 0..8 on GB300 put the best at 2 for both the 32 KB tiles of D=128
    // bf16 and the 16 KB tiles of D=64 bf16).
    static constexpr int kPieceUnits = 2;

    // shared memory layout (bytes); the per-sequence tables follow kFixedBytes
    static constexpr int kRingOff = 0;
    static constexpr int kQOff = kRingOff + kStages * 2 * kTileBytes;
    static constexpr int kEpiOff = kQOff + kStages * kQSlotBytes;
    static constexpr int kEpiFloats = ((kNW * RB * (D + 2) + 3) / 4) * 4;  // o, m, l per warp
    static constexpr int kEpiBytes = (kEpiFloats > kThreads ? kEpiFloats : kThreads) * 4;
    static constexpr int kMetaOff = kEpiOff + kEpiBytes;
    static constexpr int kBarOff = kMetaOff + kStages * 32;
    static constexpr int kJobOff = kBarOff + 2 * kStages * 8;     // after the full and empty barriers
    static constexpr int kPageOff = kJobOff + 32;                   // two pieces to count (4 ints each)
    static constexpr int kCtlOff = kPageOff + 16;                   // physical page of each stage (paged)
    static constexpr int kFixedBytes = kCtlOff + 16;                // AbortCtl words

    static_assert(kRowBytes % 16 == 0, "rows must be whole 16-byte chunks");
    static_assert(kQChunks >= 1, "q chunks per cache chunk");
    static_assert(kCpl >= 1 && kRowChunks % kL == 0, "lane mapping");
    static_assert(kNW >= 1 && kTK % kKpw == 0, "tile mapping");
    static_assert(kQOff % 128 == 0 && kEpiOff % 16 == 0 && kBarOff % 8 == 0, "alignment");
    // the merge of a split head borrows the epilogue area (see merge_pieces)
    static_assert((kThreads >= RB * D ? (kThreads / (RB * D) - 1) * (RB * D + 2 * RB) : 0) * 4 <= kEpiBytes,
                  "merge scratch");
};

// Shared-memory bytes of a launch with B sequences: fixed part + tile prefix
// sums (B + 1 ints) + history lengths (B ints).
template <typename S> constexpr size_t attn_smem_bytes(int B)
{
    return (size_t)S::kFixedBytes + (((size_t)(2 * B + 1) * 4 + 15) / 16) * 16;
}

// Per-stage description written by thread 0, read by every thread.
struct TileMeta {
    int bh, rb, tile_k0, nk;      // pair, row block, global key index of tile row 0, rows loaded
    int P, flags, n_chunks, c_first; // history, kMeta*, CTAs sharing the head, the first of them
};
constexpr int kMetaFirst = 1;  // first tile of a piece: the stage also carries the q rows
constexpr int kMetaLast = 2;   // last tile of a piece
constexpr int kMetaEnd = 4;    // no more work
constexpr int kMetaSkip = 8;   // a speculative tile that turned out not to be needed: release it

// One tile for one warp: keys warp*kKpw .. +kKpw of the tile, RB query rows.
// q, K, V and the accumulators are held as fp32 pairs (E/2 per row) and
// multiplied with packed f32x2 FMAs; a score is the sum of its even and odd
// partial dot products.
// In a fused step (kFused) the new keys P..P+N-1 are not in the cache yet: in
// the tiles that hold them (always on the masked path) their K/V rows are read
// from k_new / v_new (kn, vn: the rows of this (b, h)) and, when kc / vc are
// given, written to their cache slots by the lanes that read them: kc + key
// rows (contiguous cache: kc is the (b, h) row base), or kc + (key - tile_k0)
// rows when kTileRel (paged cache: kc is the slot of the tile's first key).
// With an E4M3 cache (C != T) the new rows are quantized on the way in
// (kv_scale: the K and V scales), exactly as the E4M3 append stores them.
template <typename T, int D, int RB, bool kMasked, bool kFused, bool kTileRel = false, typename C = T>
__device__ __forceinline__ void attn_tile(const unsigned char *Ks, const unsigned char *Vs,
                                          const f32x2 (&qv)[RB][AttnShape<T, D, RB, C>::kE / 2],
                                          f32x2 (&o)[RB][AttnShape<T, D, RB, C>::kE / 2], float (&m_run)[RB],
                                          float (&l_run)[RB], int warp, int grp, int j,
                                          int tile_k0, const int (&lim)[RB], int k_end, int P,
                                          const unsigned char *kn, const unsigned char *vn,
                                          unsigned char *kc, unsigned char *vc, float2 kv_scale = float2{})
{
    using S = AttnShape<T, D, RB, C>;
    using Ty = Elem<C>;
    constexpr bool kQuant = !std::is_same<T, C>::value;
    constexpr int E2 = S::kE / 2;
    constexpr int P2 = Ty::kPerChunk / 2;  // pairs per 16-byte chunk
    const float kNegInf = __int_as_float(0xff800000);
    constexpr float kRescaleThreshold = 8.0f;

    float sc[S::kKpg][RB];
    uint4 raw[S::kKpg][S::kCpl];

#pragma unroll
    for (int u = 0; u < S::kKpg; ++u) {
        const int kk = warp * S::kKpw + u * S::kGpw + grp;
        if constexpr (kMasked && kFused) {
            const int key = tile_k0 + kk;
            if (key >= P && key < k_end) {
                const unsigned char *src = kn + (size_t)(key - P) * S::kQRowBytes;
#pragma unroll
                for (int c = 0; c < S::kCpl; ++c) {
                    if constexpr (kQuant)
                        raw[u][c] = e4m3_chunk_from<T>(src + (c * S::kL + j) * S::kQChunks * 16, kv_scale.x);
                    else
                        raw[u][c] = ldg128_nc(src + (c * S::kL + j) * 16);
                }
                if (kc != nullptr) {
#pragma unroll
                    for (int c = 0; c < S::kCpl; ++c)
                        stg128(kc + (size_t)(kTileRel ? kk : key) * S::kRowBytes + (c * S::kL + j) * 16, raw[u][c]);
                }
                continue;
            }
        }
#pragma unroll
        for (int c = 0; c < S::kCpl; ++c)
            raw[u][c] = lds128(Ks + kk * S::kRowBytes + (c * S::kL + j) * 16);
    }
#pragma unroll
    for (int u = 0; u < S::kKpg; ++u) {
        f32x2 kf[E2];
#pragma unroll
        for (int c = 0; c < S::kCpl; ++c) Ty::widen2(raw[u][c], kf + c * P2);
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            f32x2 acc = fma2(qv[r][0], kf[0], 0ull);
#pragma unroll
            for (int e = 1; e < E2; ++e) acc = fma2(qv[r][e], kf[e], acc);
            float lo, hi;
            unpack2(acc, lo, hi);
            sc[u][r] = lo + hi;
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
    f32x2 p2[S::kKpg][RB];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        float mt = sc[0][r];
#pragma unroll
        for (int u = 1; u < S::kKpg; ++u) mt = fmaxf(mt, sc[u][r]);
        if (mt > m_run[r] + kRescaleThreshold) {
            const float alpha = fast_exp2(m_run[r] - mt);
            l_run[r] *= alpha;
            const f32x2 alpha2 = pack2(alpha, alpha);
#pragma unroll
            for (int e = 0; e < E2; ++e) o[r][e] = mul2(o[r][e], alpha2);
            m_run[r] = mt;
        }
        const float mu = (m_run[r] == kNegInf) ? 0.f : m_run[r];
#pragma unroll
        for (int u = 0; u < S::kKpg; ++u) {
            const float p = fast_exp2(sc[u][r] - mu);
            l_run[r] += p;
            p2[u][r] = pack2(p, p);
        }
    }

#pragma unroll
    for (int u = 0; u < S::kKpg; ++u) {
        const int kk = warp * S::kKpw + u * S::kGpw + grp;
        if constexpr (kMasked && kFused) {
            const int key = tile_k0 + kk;
            if (key >= P && key < k_end) {
                const unsigned char *src = vn + (size_t)(key - P) * S::kQRowBytes;
#pragma unroll
                for (int c = 0; c < S::kCpl; ++c) {
                    if constexpr (kQuant)
                        raw[u][c] = e4m3_chunk_from<T>(src + (c * S::kL + j) * S::kQChunks * 16, kv_scale.y);
                    else
                        raw[u][c] = ldg128_nc(src + (c * S::kL + j) * 16);
                }
                if (vc != nullptr) {
#pragma unroll
                    for (int c = 0; c < S::kCpl; ++c)
                        stg128(vc + (size_t)(kTileRel ? kk : key) * S::kRowBytes + (c * S::kL + j) * 16, raw[u][c]);
                }
                continue;
            }
        }
#pragma unroll
        for (int c = 0; c < S::kCpl; ++c)
            raw[u][c] = lds128(Vs + kk * S::kRowBytes + (c * S::kL + j) * 16);
    }
#pragma unroll
    for (int u = 0; u < S::kKpg; ++u) {
        f32x2 vf[E2];
#pragma unroll
        for (int c = 0; c < S::kCpl; ++c) Ty::widen2(raw[u][c], vf + c * P2);
        if constexpr (kMasked) {
            // Rows past the end of the chunk were not loaded: stale shared memory.
            if (tile_k0 + warp * S::kKpw + u * S::kGpw + grp >= k_end) {
#pragma unroll
                for (int e = 0; e < E2; ++e) vf[e] = 0ull;
            }
        }
#pragma unroll
        for (int r = 0; r < RB; ++r)
#pragma unroll
            for (int e = 0; e < E2; ++e) o[r][e] = fma2(p2[u][r], vf[e], o[r][e]);
    }
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ float safe_weight(float m, float M)
{
    return (m == __int_as_float(0xff800000)) ? 0.f : exp2f(m - M);
}

// Giving up on a wait (the CUDA-core and mma.sync kernels).  A wait that runs
// out of time -- which a healthy GPU never sees -- must not leave the CTA's
// threads on different paths: the piece epilogues contain CTA barriers, so
// every thread has to step through the same ring positions.  Thread 0
// publishes how many positions it has described (their TileMeta written)
// before it can block at a CTA barrier, and once its own warp gives up it
// describes no more and publishes that count as the last; a warp that has
// given up steps on through described positions without waiting for their
// data (its results are garbage, flagged by KVD_DEVERR_TIMEOUT) and stops
// where the walk stops.  A stage is refilled only after every warp released
// it, which a warp that gave up never does, so no barrier is ever armed while
// its previous phase is open; thread 0 waits (kDrainLimitNs) for its copies
// still in flight before the CTA exits.
struct AbortCtl {
    volatile int *w;  // [0] abort, [1] positions described, [2] final count + 1 (0: not yet)

    __device__ __forceinline__ void init() const
    {
        w[0] = 0;
        w[1] = 0;
        w[2] = 0;
    }
    __device__ __forceinline__ const volatile int *flag() const { return w; }
    __device__ __forceinline__ void set_abort() const { w[0] = 1; }
    __device__ __forceinline__ bool aborted() const { return w[0] != 0; }
    // thread 0, after writing the TileMeta of positions < n
    __device__ __forceinline__ void described(int n) const { st_release_cta(w + 1, n); }
    __device__ __forceinline__ void final_count(int n) const { st_release_cta(w + 2, n + 1); }
    // A thread that gave up, at position pos: whether pos is described (its
    // TileMeta may be read), else the walk stops before it.  Bounded.
    __device__ __forceinline__ bool describable(int pos) const
    {
        const uint64_t t0 = global_timer_ns();
        for (uint32_t it = 0;; ++it) {
            if (pos < ld_acquire_cta(w + 1)) return true;
            const int f = ld_acquire_cta(w + 2);
            if (f != 0) return pos < f - 1;
            if ((it & 63u) == 0u && global_timer_ns() - t0 > 2 * kDrainLimitNs) return false;
        }
    }
};

// CTA whose range [c*n/G, (c+1)*n/G) holds flattened unit t.  With G <= n
// every range is non-empty, so the CTAs holding a head's tiles are consecutive.
__device__ __forceinline__ int owner_cta(long long t, long long n, long long G)
{
    const unsigned long long num = (unsigned long long)(t + 1) * G + n - 1;
    if (num < (1ull << 32)) return (int)((unsigned)num / (unsigned)n) - 1;  // common case: 32-bit divide
    return (int)(num / (unsigned long long)n) - 1;
}

// Thread 0's walk over the CTA's range.  The range is counted in units: a
// sequence-head with tb tiles is kPieceUnits overhead units (what a piece
// boundary costs: merges, restarting the ring) followed by tb tile units, so
// CTAs whose range crosses more head starts receive fewer tiles.  Per-head
// values are computed once when the walk enters a head; a tile only costs a
// few stores and the bulk copies.
template <typename S, bool kWriteSeg, bool kPaged> struct RangeWalk {
    long long t, hi, n, G;  // unit of the next tile, end of range, units in total, working CTAs
    int b, hr, tin, tb;     // sequence, head x row block, tile within the head, its tiles
    int HR;                 // H_kv * n_rowblocks
    bool ended;
    bool piece_start;       // the next tile starts a piece (the head's first tile, or the range's)
    // per-head values
    int bh, rb, P, T_b, n_chunks, c_first, q_bytes;
    const unsigned char *kg, *vg, *qg;
    uint64_t policy;
    int page_next;          // paged: physical page of the next tile (loaded one tile ahead)
    const unsigned char *pend_q[S::kStages];  // kFillKvOnly: the q rows each stage still has to load
    uint32_t pend_qb[S::kStages];
#ifdef KVD_TIMEOUT_TEST
    bool stalled;  // kArgTestStall: the stall has been planted
    __device__ __forceinline__ uint32_t stall_bytes(const AttnArgs &a)
    {
        if (!(a.flags & kArgTestStall) || stalled) return 0u;
        stalled = true;
        return 16u;
    }
#else
    __device__ __forceinline__ uint32_t stall_bytes(const AttnArgs &) { return 0u; }
#endif
    const int32_t *bt_row;  // paged: block-table row of the current sequence
    const void *tm_k, *tm_v;  // tensor-map tiles (S::kTma): the K and V tensor maps

    // Paged: start the load of the next tile's page-table entry; it is used
    // one fill later, so its latency hides behind the current tile.
    __device__ __forceinline__ void prefetch_page(const AttnArgs &a)
    {
        if constexpr (kPaged) {
            if (t < hi)
                page_next = __ldg(bt_row + ((tin * S::kTK) >> a.page_shift));
        }
    }

    __device__ __forceinline__ void enter_head(const AttnArgs &a, const int *pl)
    {
        const long long ts = t - tin;  // unit of the head's first tile
        c_first = owner_cta(ts, n, G);
        n_chunks = owner_cta(ts + tb - 1, n, G) - c_first + 1;
        if constexpr (kWriteSeg) {  // the split's shape, for the merge pass
            if (tin == 0) static_cast<int2 *>(a.merge_state)[(size_t)b * HR + hr] = make_int2(c_first, n_chunks);
        }
        set_head(a, pl[b]);
    }

    // Per-head fields of (b, hr) with history P_: row block, addresses, q rows.
    __device__ __forceinline__ void set_head(const AttnArgs &a, int P_)
    {
        const int h = hr / a.n_rowblocks;
        rb = hr % a.n_rowblocks;
        bh = b * a.H_kv + h;
        P = P_;
        T_b = P + a.N;
        if constexpr (kPaged) {
            const size_t hoff = ((size_t)h << a.page_shift) * S::kRowBytes;
            kg = static_cast<const unsigned char *>(a.k_cache) + hoff;
            vg = static_cast<const unsigned char *>(a.v_cache) + hoff;
            bt_row = a.block_table + (size_t)b * (a.T_max >> a.page_shift);
        } else {
            const size_t row = (size_t)bh * a.T_max;
            kg = static_cast<const unsigned char *>(a.k_cache) + row * S::kRowBytes;
            vg = static_cast<const unsigned char *>(a.v_cache) + row * S::kRowBytes;
        }
        qg = static_cast<const unsigned char *>(a.q) + ((size_t)bh * a.rows + rb * S::kRB) * S::kQRowBytes;
        q_bytes = min(S::kRB, a.rows - rb * S::kRB) * S::kQRowBytes;
    }

    // Cluster mode: the walk covers tiles [tin0, tin1) of the one
    // sequence-head (b_, hr_) with history P_ and tb_ tiles; t counts the
    // piece's tiles and HR is set so that the walk never moves to a next head.
    __device__ __forceinline__ void start_piece(const AttnArgs &a, int b_, int hr_, int P_, int tb_, int tin0,
                                                int tin1, int n_chunks_)
    {
        policy = l2_evict_first_policy();
#ifdef KVD_TIMEOUT_TEST
        stalled = false;
#endif
        HR = 0x7fffffff;
        b = b_;
        hr = hr_;
        tb = tb_;
        tin = tin0;
        t = 0;
        hi = tin1 - tin0;
        n = hi;
        G = 1;
        ended = false;
        piece_start = true;
        c_first = 0;
        n_chunks = n_chunks_;
        if (t < hi) set_head(a, P_);
        prefetch_page(a);
    }

    // pre[b] = units of sequences 0..b-1 per head (a head of sequence b has
    // pre[b+1] - pre[b] units, kPieceUnits of them overhead, or 0 if empty).
    __device__ __forceinline__ void start(const AttnArgs &a, const int *pre, const int *pl, long long lo,
                                          long long hi_, long long n_, long long G_)
    {
        policy = l2_evict_first_policy();
#ifdef KVD_TIMEOUT_TEST
        stalled = false;
#endif
        HR = a.H_kv * a.n_rowblocks;
        hi = hi_;
        n = n_;
        G = G_;
        ended = false;
        piece_start = true;
        if (lo >= hi) {
            t = hi;
            return;
        }
        int lo_b = 0, hi_b = a.B - 1;  // last b with pre[b] * HR <= lo
        while (lo_b < hi_b) {
            const int mid = (lo_b + hi_b + 1) / 2;
            if ((long long)pre[mid] * HR <= lo) lo_b = mid; else hi_b = mid - 1;
        }
        b = lo_b;
        const int ub = pre[b + 1] - pre[b];
        tb = ub - S::kPieceUnits;
        const long long local = lo - (long long)pre[b] * HR;
        hr = (int)(local / ub);
        const int off = (int)(local % ub);
        tin = max(0, off - S::kPieceUnits);
        t = (long long)pre[b] * HR + (long long)hr * ub + S::kPieceUnits + tin;
        if (t < hi) enter_head(a, pl);
        prefetch_page(a);
    }

    // Describe and load the next tile into slot s, or mark the end of work.
    __device__ __forceinline__ void fill(const AttnArgs &a, const int *pre, const int *pl,
                                         unsigned char *smem, TileMeta *meta, uint64_t *full, int s,
                                         FillMode mode = kFillOne)
    {
        // (paged) page of the tile: a tile never straddles a page
        int page = 0;
        if (ended) return;
        if (t >= hi) {
            meta[s].flags = kMetaEnd;
            mbar_arrive(&full[s]);
            if (mode == kFillTwo) mbar_arrive(&full[s]);
            if (mode == kFillKvOnly) pend_qb[s] = 0u;
            ended = true;
            return;
        }
        TileMeta mt;
        mt.bh = bh;
        mt.rb = rb;
        mt.tile_k0 = tin * S::kTK;
        mt.nk = min(S::kTK, T_b - mt.tile_k0);
        mt.P = P;
        mt.flags = (piece_start ? kMetaFirst : 0) | ((tin == tb - 1 || t == hi - 1) ? kMetaLast : 0);
        mt.n_chunks = n_chunks;
        mt.c_first = c_first;
        meta[s] = mt;

        const uint32_t bytes = (uint32_t)mt.nk * S::kRowBytes;
        uint32_t qbytes = (S::kQInRing && piece_start) ? (uint32_t)q_bytes : 0u;
        if (mode == kFillKvOnly) {
            pend_q[s] = qg;
            pend_qb[s] = qbytes;
            qbytes = 0u;
        }
        size_t off;
        if constexpr (kPaged) {
            page = page_next;
            int *stage_page = reinterpret_cast<int *>(smem + S::kPageOff);
            if ((unsigned)page >= (unsigned)a.num_pages) {
                // Never read outside the pool: load page 0 instead, flag the
                // error, and tell the fused step not to write this tile.
                raise_error(a.err_word, KVD_DEVERR_PAGE);
                stage_page[s] = -1;
                page = 0;
            } else {
                stage_page[s] = page;
            }
            // (kg already points at head h's rows of page 0; few operations
            // here, as this runs on the producer's critical path every tile)
            off = (size_t)page * (((size_t)a.H_kv * S::kRowBytes) << a.page_shift) +
                  (size_t)(mt.tile_k0 & ((1 << a.page_shift) - 1)) * S::kRowBytes;
        } else {
            off = (size_t)mt.tile_k0 * S::kRowBytes;
        }
        unsigned char *dst = smem + S::kRingOff + s * 2 * S::kTileBytes;
        if constexpr (S::kTma) {
            // whole boxes of kTK rows (rows past the head are masked, or zero
            // past the tensor), 128-byte swizzled, kBoxes per K or V tile
            (void)off;
            mbar_arrive_expect_tx(&full[s], 2u * S::kTileBytes + qbytes + stall_bytes(a));
            int y;  // first row of the tile in the tensor map's [rows, D] view
            if constexpr (kPaged)
                y = ((page * a.H_kv + (bh - b * a.H_kv)) << a.page_shift) + (mt.tile_k0 & ((1 << a.page_shift) - 1));
            else
                y = bh * a.T_max + mt.tile_k0;
#pragma unroll
            for (int bx = 0; bx < S::kBoxes; ++bx) {
                tma_load_2d(dst + bx * S::kBoxBytes, tm_k, bx * S::kBoxCols, y, &full[s], policy);
                tma_load_2d(dst + S::kTileBytes + bx * S::kBoxBytes, tm_v, bx * S::kBoxCols, y, &full[s], policy);
            }
        } else {
            mbar_arrive_expect_tx(&full[s], 2u * bytes + qbytes + stall_bytes(a));
            bulk_load_g2s(dst, kg + off, bytes, &full[s], policy);
            bulk_load_g2s(dst + S::kTileBytes, vg + off, bytes, &full[s], policy);
        }
        if (qbytes) bulk_load_g2s(smem + S::kQOff + s * S::kQSlotBytes, qg, qbytes, &full[s], policy);
        if (mode == kFillTwo) mbar_arrive(&full[s]);

        // advance to the next tile of the flattened list (skipping the next
        // head's overhead units)
        ++t;
        piece_start = false;
        if (++tin == tb) {
            tin = 0;
            piece_start = true;
            if (++hr == HR) {
                hr = 0;
                do {
                    ++b;
                } while (b < a.B && pre[b + 1] == pre[b]);
                if (b < a.B) tb = pre[b + 1] - pre[b] - S::kPieceUnits;
            }
            t += S::kPieceUnits;
            if (t < hi) enter_head(a, pl);
        }
        prefetch_page(a);
    }

    // The history of the current head, once known (cluster mode fills with
    // the host's bound first).
    __device__ __forceinline__ void set_history(const AttnArgs &a, int P_)
    {
        P = P_;
        T_b = P + a.N;
    }

    // Stage s (filled, not yet consumed) becomes a tile to skip.
    __device__ __forceinline__ void skip_stage(TileMeta *meta, int s)
    {
        meta[s].flags = kMetaSkip;
        pend_qb[s] = 0u;
    }

    // The second arrival of stage s filled with kFillKvOnly: its q rows, if any.
    __device__ __forceinline__ void issue_pending(unsigned char *smem, uint64_t *full, int s)
    {
        if (pend_qb[s]) {
            mbar_arrive_expect_tx(&full[s], pend_qb[s]);
            bulk_load_g2s(smem + S::kQOff + s * S::kQSlotBytes, pend_q[s], pend_qb[s], &full[s], policy);
        } else {
            mbar_arrive(&full[s]);
        }
    }
};

// Rows per partial slot.  Row blocks of fewer than 16 rows (the CUDA-core
// kernels' RB 1, 2, 4, 8 and the 8-row E4M3 tensor-core form) keep all RB
// slots; the tensor-core kernels' 16- and 128-row blocks keep only the
// block's real rows, min(RB, rows), so few-row decodes do not carry padded
// partials.  The host sizes the workspace by the same rule.
template <int RB> __device__ __forceinline__ int part_rows(int rows)
{
    if constexpr (RB >= 16) return rows < RB ? rows : RB;
    else return RB;
}

// A piece of a split head this CTA computed, or a head it merges.
struct MergeJob {
    int bh, rb, c_first, n_chunks;
};

// Merge the n_chunks pieces of a split head by log-sum-exp and write its
// output rows, with every thread of the CTA.  Piece k is CTA c_first + k's
// partial (slot 1 for k = 0, the head's first CTA, else slot 0).  The pieces
// are split over kNG thread groups when the head has fewer output elements
// than the CTA has threads; the groups then combine through scr (shared
// memory, free on entry and again on return).
template <typename T, int D, int RB, int kThreads, bool kScaleV = false>
__device__ __forceinline__ void merge_pieces(const AttnArgs &a, const MergeJob &job, float *scr, int tid)
{
    using Ty = Elem<T>;
    constexpr int kNE = RB * D;                                  // output elements of the head's rows
    constexpr int kNG = kThreads >= kNE ? kThreads / kNE : 1;    // groups sharing out the pieces
    constexpr int kPer = kThreads >= kNE ? 1 : kNE / kThreads;   // elements per thread
    static_assert(kNG * kNE == kThreads || kPer * kThreads == kNE, "merge mapping");
    const float kNegInf = __int_as_float(0xff800000);
    const int g = kNG > 1 ? tid / kNE : 0;
    const int e0 = kNG > 1 ? tid % kNE : tid;
    float M[kPer], num[kPer], den[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        M[i] = kNegInf;
        num[i] = 0.f;
        den[i] = 0.f;
    }
    // The loads of a piece do not depend on the running values: each pass
    // issues all of them before the updates.
#pragma unroll 2
    for (int k = g; k < job.n_chunks; k += kNG) {
        const size_t pb = ((size_t)(job.c_first + k) * 2 + (k == 0)) * part_rows<RB>(a.rows);
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int e = e0 + i * kThreads, r = e / D, d = e % D;
            const float *pr = a.part + (pb + r) * (D + 4);
            const float2 ml = __ldcg(reinterpret_cast<const float2 *>(pr + D));
            const float o_k = __ldcg(pr + d);
            const float Mn = fmaxf(M[i], ml.x);
            const float wa = safe_weight(M[i], Mn), wb = safe_weight(ml.x, Mn);
            num[i] = num[i] * wa + o_k * wb;
            den[i] = den[i] * wa + ml.y * wb;
            M[i] = Mn;
        }
    }
    if constexpr (kNG > 1) {
        // groups 1.. hand their running values to group 0
        const int r = e0 / D, d = e0 % D;
        float *s_num = scr, *s_ml = scr + (kNG - 1) * kNE;
        if (g > 0) {
            s_num[(g - 1) * kNE + e0] = num[0];
            if (d == 0) {
                s_ml[((g - 1) * RB + r) * 2 + 0] = M[0];
                s_ml[((g - 1) * RB + r) * 2 + 1] = den[0];
            }
        }
        __syncthreads();
        if (g == 0) {
#pragma unroll
            for (int gg = 0; gg < kNG - 1; ++gg) {
                const float m_g = s_ml[(gg * RB + r) * 2 + 0];
                const float Mn = fmaxf(M[0], m_g);
                const float wa = safe_weight(M[0], Mn), wb = safe_weight(m_g, Mn);
                num[0] = num[0] * wa + s_num[gg * kNE + e0] * wb;
                den[0] = den[0] * wa + s_ml[(gg * RB + r) * 2 + 1] * wb;
                M[0] = Mn;
            }
        }
        __syncthreads();
    }
    if (g == 0) {
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int e = e0 + i * kThreads, r = e / D, d = e % D;
            const int rg = job.rb * RB + r;
            if (rg < a.rows) {
                if constexpr (kScaleV)  // E4M3 cache: values are stored / v_scale
                    Ty::store(static_cast<T *>(a.out) + ((size_t)job.bh * a.rows + rg) * D + d,
                              num[i] / den[i] * a.kv_scale.y);
                else
                    Ty::store(static_cast<T *>(a.out) + ((size_t)job.bh * a.rows + rg) * D + d, num[i] / den[i]);
            }
        }
    }
}

// Units per sequence-head, prefix-summed over sequences by warp 0's scan:
// pre[b] = units of sequences 0..b-1 per head, pl[b] = P_b.  A sequence with
// an invalid P_b gets no units; CTA 0 reports it, or (defer_error) returns
// true for the caller to report later.
template <typename S>
__device__ __forceinline__ bool unit_prefix(const AttnArgs &a, int *pre, int *pl, int lane, bool defer_error = false)
{
    bool bad = false;
    int carry = 0;
    if (lane == 0) pre[0] = 0;
    for (int b0 = 0; b0 < a.B; b0 += 32) {
        const int b = b0 + lane;
        int units = 0;
        if (b < a.B) {
            const int P = __ldg(a.past_len + b);
            const bool ok = past_len_ok(P, a.N, a.T_max, a.max_past_len);
            if (!ok && blockIdx.x == 0) {
                if (defer_error) bad = true;
                else raise_error(a.err_word, KVD_DEVERR_PAST_LEN);
            }
            units = ok ? (P + a.N + S::kTK - 1) / S::kTK + S::kPieceUnits : 0;
            pl[b] = P;
        }
        int v = units;  // inclusive scan over the warp
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += n;
        }
        if (b < a.B) pre[b + 1] = carry + v;
        carry += __shfl_sync(0xffffffffu, v, 31);
    }
    __syncwarp();
    return __any_sync(0xffffffffu, bad);
}

// This CTA's range [lo, hi) of the flattened unit list (see RangeWalk).
__device__ __forceinline__ void cta_range(const AttnArgs &a, const int *pre, long long *n_total, long long *G,
                                          long long *lo, long long *hi)
{
    const int HR = a.H_kv * a.n_rowblocks;
    *n_total = (long long)pre[a.B] * HR;
    *G = min((long long)gridDim.x, *n_total);  // CTAs that get work
    *lo = blockIdx.x < *G ? *n_total * blockIdx.x / *G : 0;
    *hi = blockIdx.x < *G ? *n_total * (blockIdx.x + 1) / *G : 0;
}

// Cluster mode, thread 0: the CTA's piece of its cluster's sequence-head (an
// equal share of the head's tiles by cluster rank) and its first ring fills.
// For a contiguous cache the share is first taken with the history at
// max_past_len (the host's bound) while past_len is being read; if the real tile count is the same the
// filled stages only get their history and row count corrected, else they are
// marked to be skipped and the walk starts again.  Returns whether past_len
// of the head's sequence is valid (else the range is empty and the sequence
// is skipped).
template <typename S, bool kPaged, typename Walk>
__device__ __forceinline__ bool cluster_start(const AttnArgs &a, Walk &walk, unsigned char *smem, TileMeta *meta,
                                              uint64_t *full, int &issued, FillMode mode)
{
    const int csize = (int)cluster_nctarank(), crank = (int)cluster_ctarank();
    const int HR = a.H_kv * a.n_rowblocks;
    const int u = (int)blockIdx.x / csize;  // the cluster's sequence-head (b, hr)
    const int b = u / HR, hr = u % HR;
    const int P = __ldg(a.past_len + b);  // (in flight during the fills below)
    if constexpr (kPaged) {
        // (no speculation: block-table entries past a sequence's end need not
        // name valid pages)
        const bool ok = past_len_ok(P, a.N, a.T_max, a.max_past_len);
        const int tb = ok ? (P + a.N + S::kTK - 1) / S::kTK : 0;
        walk.start_piece(a, b, hr, P, tb, tb * crank / csize, tb * (crank + 1) / csize, csize);
        for (; issued < S::kStages && !walk.ended; ++issued)
            walk.fill(a, nullptr, nullptr, smem, meta, full, issued, mode);
        return ok;
    }
    const int tb_bound = (a.max_past_len + a.N + S::kTK - 1) / S::kTK;
    walk.start_piece(a, b, hr, a.max_past_len, tb_bound, tb_bound * crank / csize, tb_bound * (crank + 1) / csize,
                     csize);
    for (; issued < S::kStages && !walk.ended; ++issued) walk.fill(a, nullptr, nullptr, smem, meta, full, issued, mode);
    const bool ok = past_len_ok(P, a.N, a.T_max, a.max_past_len);
    const int tb = ok ? (P + a.N + S::kTK - 1) / S::kTK : 0;
    if (tb == tb_bound) {  // the same tiles: correct the history and the rows of each filled tile
        walk.set_history(a, P);
        for (int s = 0; s < issued; ++s)
            if (!(meta[s].flags & kMetaEnd)) {
                meta[s].P = P;
                meta[s].nk = min(S::kTK, P + a.N - meta[s].tile_k0);
            }
    } else {
        for (int s = 0; s < issued; ++s) walk.skip_stage(meta, s);
        walk.start_piece(a, b, hr, P, tb, tb * crank / csize, tb * (crank + 1) / csize, csize);
    }
    return ok;
}

// kFused: append inside (kvd_decode_step).  kTicketMerge: split heads are
// merged at the end of this kernel (else by attn_merge_kernel).  kPaged: the
// cache is paged (block table), else contiguous [B, H_kv, T_max, D].
// kCluster (small layers): the grid is one thread-block
// cluster per sequence-head; the cluster's CTAs split the head's tiles in equal
// shares by rank, each loads its whole share into its ring and stores its
// piece into rank 0's shared memory, and rank 0 merges them (no workspace, no
// atomics, one cluster barrier).  The pieces live after the fixed layout, in
// place of the per-sequence tables: cluster size x RB rows of (o[D], m, l).
template <typename T, int D, int RB, bool kFused, bool kTicketMerge, bool kPaged, typename C = T,
          bool kCluster = false>
__global__ void __launch_bounds__(AttnShape<T, D, RB, C>::kThreads)
    attn_balanced_kernel(const AttnArgs a)
{
    using S = AttnShape<T, D, RB, C>;
    using Ty = Elem<C>;                                // cache rows
    using Tq = Elem<T>;                                // q / out rows
    constexpr bool kQuant = !std::is_same<T, C>::value;  // E4M3 cache: scales apply
    static_assert(!(kQuant && kPaged), "the E4M3 cache is contiguous only");
    const float kNegInf = __int_as_float(0xff800000);
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::kBarOff);
    uint64_t *empty = full + S::kStages;
    TileMeta *meta = reinterpret_cast<TileMeta *>(smem + S::kMetaOff);
    MergeJob *jobs = reinterpret_cast<MergeJob *>(smem + S::kJobOff);  // this CTA's split pieces (two at most)
    int *pre = reinterpret_cast<int *>(smem + S::kFixedBytes);  // [B + 1] unit prefix per head
    int *pl = pre + a.B + 1;                                     // [B] history lengths
    const AbortCtl ctl{reinterpret_cast<volatile int *>(smem + S::kCtlOff)};

    const int tid = threadIdx.x;
    const int warp = tid / 32, lane = tid % 32;
    const int grp = lane / S::kL, j = lane % S::kL;

    const bool early = (a.flags & kArgEarly) != 0;
    const bool stable = early && (a.flags & kArgHistoryStable) != 0;
    const FillMode refill = stable ? kFillTwo : kFillOne;
    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < S::kStages; ++s) {
            mbar_init(&full[s], stable ? 2 : 1);  // (stable: K/V before the wait, q after)
            mbar_init(&empty[s], S::kNW);
        }
        ctl.init();
        fence_mbar_init();
    }
    // Warp 0 forms the unit prefix over sequences and thread 0 starts the ring
    // (slot s of ring position p is free again once every warp has released
    // position p - STAGES on empty[s]); the other warps go straight to
    // waiting for the first tile.
    RangeWalk<S, !kTicketMerge, kPaged> walk;  // used by thread 0 only
    int issued = 0;     // ring positions filled so far (thread 0)
    bool bad_past = false;
    int *cl_ok = reinterpret_cast<int *>(jobs);  // cluster mode: the head's sequence is valid
    if constexpr (kCluster) {
        // (planned for small layers only: the next kernel may launch now)
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        if (stable && tid == 0) bad_past = !cluster_start<S, kPaged>(a, walk, smem, meta, full, issued, kFillKvOnly);
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (tid == 0) {
            if (stable) {
                for (int p = 0; p < issued; ++p) walk.issue_pending(smem, full, p);  // the q rows
            } else {
                bad_past = !cluster_start<S, kPaged>(a, walk, smem, meta, full, issued, kFillOne);
            }
            *cl_ok = bad_past ? 0 : 1;
            ctl.described(issued);
            // (one report per sequence: the first rank of its first head's cluster)
            if (bad_past && cluster_ctarank() == 0 && ((int)blockIdx.x / (int)cluster_nctarank()) % (a.H_kv * a.n_rowblocks) == 0)
                raise_error(a.err_word, KVD_DEVERR_PAST_LEN);
        }
        __syncthreads();
    } else {
    if (early) {
        // Small layers: the next kernel may launch now (its CTAs take the SM
        // slots that are free and wait in their turn).  With a stable
        // history, the split and the first K/V tiles need nothing from the
        // previous kernel: start them before waiting.
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        if (stable && warp == 0) {
            bad_past = unit_prefix<S>(a, pre, pl, lane, true);
            if (lane == 0) {
                long long n_total, G, lo, hi;
                cta_range(a, pre, &n_total, &G, &lo, &hi);
                walk.start(a, pre, pl, lo, hi, n_total, G);
                for (; issued < S::kStages && !walk.ended; ++issued)
                    walk.fill(a, pre, pl, smem, meta, full, issued, kFillKvOnly);
            }
        }
    }
    // Every input may come from the previous kernel on the stream.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // The next kernel on the stream may launch now: its CTAs take the SM
    // slots this grid frees and run up to their own griddepcontrol.wait,
    // which still waits for this whole grid to finish and flush.
    if (!early) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (stable && warp == 0 && lane == 0) {
        if (bad_past) raise_error(a.err_word, KVD_DEVERR_PAST_LEN);
        for (int p = 0; p < issued; ++p) walk.issue_pending(smem, full, p);  // the q rows
        ctl.described(issued);
    }
    __syncthreads();  // barrier initialisation visible to every thread

    if (warp == 0 && !stable) {
        unit_prefix<S>(a, pre, pl, lane);
        if (lane == 0) {
            long long n_total, G, lo, hi;
            cta_range(a, pre, &n_total, &G, &lo, &hi);
            walk.start(a, pre, pl, lo, hi, n_total, G);
            for (; issued < S::kStages && !walk.ended; ++issued) walk.fill(a, pre, pl, smem, meta, full, issued);
            ctl.described(issued);
        }
    }
    }  // (not kCluster)

    f32x2 qv[RB][S::kE / 2];
    f32x2 o[RB][S::kE / 2];
    float m_run[RB], l_run[RB];
    int lim[RB];
    bool gave_up = false;     // this warp no longer waits for data (see AbortCtl)
    int first_unwaited = -1;  // thread 0: first ring position whose copies it did not see land
    int n_pieces = 0;         // split pieces computed so far (two at most)

    for (int pos = 0;; ++pos) {  // until the end marker
        const int s = pos % S::kStages;
        const uint32_t ph = (uint32_t)(pos / S::kStages) & 1u;
        if (!gave_up) {
            if (tid == 0) {
                // Position pos must have been issued before anyone waits for it; its
                // slot frees as soon as the slower warps release pos - STAGES.
                while (issued <= pos && !walk.ended) {
                    const int fs = issued % S::kStages;
                    const uint32_t fph = ((uint32_t)(issued / S::kStages) & 1u) ^ 1u;
                    const int r = mbar_wait_or_abort(&empty[fs], fph, ctl.flag());
                    if (r != 0) {
                        if (r == 1) {
                            ctl.set_abort();
                            raise_error(a.err_word, KVD_DEVERR_TIMEOUT);
                        }
                        break;
                    }
                    walk.fill(a, pre, pl, smem, meta, full, fs, refill);
                    ++issued;
                }
            }
            const int r = mbar_wait_or_abort(&full[s], ph, ctl.flag());
            if (r == 1) {
                ctl.set_abort();
                raise_error(a.err_word, KVD_DEVERR_TIMEOUT);
            }
            gave_up = __any_sync(0xffffffffu, r != 0);  // (warp-uniform: the tile code shuffles)
            if (gave_up && tid == 0) first_unwaited = pos;
        }
        if (gave_up) {
            if (tid == 0) ctl.final_count(issued);
            if (!ctl.describable(pos)) break;
        }
        const TileMeta mt = meta[s];
        if (mt.flags & kMetaEnd) break;
        if (mt.flags & kMetaSkip) {  // (cluster mode: a speculative tile, not needed)
            __syncwarp();
            if (lane == 0 && !gave_up) mbar_arrive(&empty[s]);
            continue;
        }
        const unsigned char *Ks = smem + S::kRingOff + s * 2 * S::kTileBytes;
        const unsigned char *Vs = Ks + S::kTileBytes;

        if (mt.flags & kMetaFirst) {
            const unsigned char *qs = smem + S::kQOff + s * S::kQSlotBytes;
            const int q_rows = min(RB, a.rows - mt.rb * RB);
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                const int rg = mt.rb * RB + r;
                lim[r] = mt.P + 1 + (rg % a.N);
                m_run[r] = kNegInf;
                l_run[r] = 0.f;
#pragma unroll
                for (int e = 0; e < S::kE / 2; ++e) o[r][e] = 0ull;
                if (r < q_rows) {
                    const f32x2 qs2 = pack2(a.qscale, a.qscale);
#pragma unroll
                    for (int c = 0; c < S::kCpl; ++c)
#pragma unroll
                        for (int qc = 0; qc < S::kQChunks; ++qc)  // the q elements of cache chunk c*L + j
                            Tq::widen2(lds128(qs + r * S::kQRowBytes + ((c * S::kL + j) * S::kQChunks + qc) * 16),
                                       &qv[r][c * (Ty::kPerChunk / 2) + qc * (Tq::kPerChunk / 2)]);
#pragma unroll
                    for (int e = 0; e < S::kE / 2; ++e) qv[r][e] = mul2(qv[r][e], qs2);
                } else {
#pragma unroll
                    for (int e = 0; e < S::kE / 2; ++e) qv[r][e] = 0ull;
                }
            }
        }

        const int k_end = mt.tile_k0 + mt.nk;
        // Tiles below every row's limit (and, in a fused step, below the new
        // keys) take the unmasked path; the rest the masked one.  (A warp that
        // gave up computes nothing and writes nothing.)
        if (gave_up) {
        } else if (mt.tile_k0 + S::kTK <= mt.P + (kFused ? 0 : 1)) {
            attn_tile<T, D, RB, false, kFused, false, C>(Ks, Vs, qv, o, m_run, l_run, warp, grp, j, mt.tile_k0,
                                                         lim, k_end, mt.P, nullptr, nullptr, nullptr, nullptr);
        } else {
            const unsigned char *kn = nullptr, *vn = nullptr;
            unsigned char *kc = nullptr, *vc = nullptr;
            if constexpr (kFused) {
                const size_t nrow = (size_t)mt.bh * a.N * S::kQRowBytes;
                kn = static_cast<const unsigned char *>(a.k_new) + nrow;
                vn = static_cast<const unsigned char *>(a.v_new) + nrow;
                if constexpr (kPaged) {
                    // the slot of the tile's first key in its page (none if the page is invalid)
                    const int page = reinterpret_cast<const int *>(smem + S::kPageOff)[s];
                    if (mt.rb == 0 && page >= 0) {
                        const size_t crow = (((size_t)page * a.H_kv + mt.bh % a.H_kv) << a.page_shift) +
                                            (mt.tile_k0 & ((1 << a.page_shift) - 1));
                        kc = static_cast<unsigned char *>(const_cast<void *>(a.k_cache)) + crow * S::kRowBytes;
                        vc = static_cast<unsigned char *>(const_cast<void *>(a.v_cache)) + crow * S::kRowBytes;
                    }
                } else if (mt.rb == 0) {  // one row block writes the new rows into the cache
                    const size_t crow = (size_t)mt.bh * a.T_max * S::kRowBytes;
                    kc = static_cast<unsigned char *>(const_cast<void *>(a.k_cache)) + crow;
                    vc = static_cast<unsigned char *>(const_cast<void *>(a.v_cache)) + crow;
                }
            }
            float2 kvs = float2{};
            if constexpr (kQuant) kvs = a.kv_scale;
            attn_tile<T, D, RB, true, kFused, kPaged, C>(Ks, Vs, qv, o, m_run, l_run, warp, grp, j, mt.tile_k0,
                                                         lim, k_end, mt.P, kn, vn, kc, vc, kvs);
        }
        __syncwarp();
        if (lane == 0 && !gave_up) mbar_arrive(&empty[s]);  // this warp is done with slot s

        // Opportunistic refill: if every warp has released the slot, issue now.
        if (tid == 0 && !gave_up && !walk.ended && issued < pos + 1 + S::kStages) {
            const int fs = issued % S::kStages;
            const uint32_t fph = ((uint32_t)(issued / S::kStages) & 1u) ^ 1u;
            if (mbar_test_wait(&empty[fs], fph)) {
                walk.fill(a, pre, pl, smem, meta, full, fs, refill);
                ++issued;
            }
        }

        if (!(mt.flags & kMetaLast)) continue;

        // ---- end of a piece: merge the key groups of each warp (xor shuffles),
        //      then the warps through shared memory ----
        float *ep_o = reinterpret_cast<float *>(smem + S::kEpiOff);
        float *ep_m = ep_o + S::kNW * RB * D;
        float *ep_l = ep_m + S::kNW * RB;
#pragma unroll
        for (int off = S::kL; off < 32; off *= 2) {
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                const float m_o = __shfl_xor_sync(0xffffffffu, m_run[r], off);
                const float l_o = __shfl_xor_sync(0xffffffffu, l_run[r], off);
                const float M = fmaxf(m_run[r], m_o);
                const float wa = safe_weight(m_run[r], M), wb = safe_weight(m_o, M);
                l_run[r] = l_run[r] * wa + l_o * wb;
#pragma unroll
                for (int e = 0; e < S::kE / 2; ++e) {
                    float lo, hi;
                    unpack2(o[r][e], lo, hi);
                    lo = lo * wa + __shfl_xor_sync(0xffffffffu, lo, off) * wb;
                    hi = hi * wa + __shfl_xor_sync(0xffffffffu, hi, off) * wb;
                    o[r][e] = pack2(lo, hi);
                }
                m_run[r] = M;
            }
        }
        // (thread 0 may now block at a CTA barrier: what it has described must
        // be known to warps that gave up, so that they can reach it too)
        if (tid == 0) ctl.described(issued);
        __syncthreads();  // the previous piece's readers are done with the shared area
        if (grp == 0) {
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                float *dst = ep_o + (warp * RB + r) * D;
#pragma unroll
                for (int c = 0; c < S::kCpl; ++c) {
                    const int d0 = (c * S::kL + j) * Ty::kPerChunk;
#pragma unroll
                    for (int e = 0; e < Ty::kPerChunk; e += 4) {
                        float4 v;
                        unpack2(o[r][(c * Ty::kPerChunk + e) / 2], v.x, v.y);
                        unpack2(o[r][(c * Ty::kPerChunk + e) / 2 + 1], v.z, v.w);
                        *reinterpret_cast<float4 *>(dst + d0 + e) = v;
                    }
                }
                if (j == 0) {
                    ep_m[warp * RB + r] = m_run[r];
                    ep_l[warp * RB + r] = l_run[r];
                }
            }
        }
        __syncthreads();
        const bool single = !kCluster && (mt.n_chunks == 1);
        // Cluster mode: the CTA's one piece goes to its slot in rank 0's
        // shared memory, for rank 0 to merge after the cluster barrier.
        float *cl_part = reinterpret_cast<float *>(smem + S::kFixedBytes) +
                         (kCluster ? cluster_ctarank() * RB * (D + 2) : 0);
        // A CTA holds at most two partial pieces: slot 1 for the head it starts
        // (it is that head's first CTA), slot 0 for the head it continues.
        const size_t pbase = ((size_t)blockIdx.x * 2 + ((int)blockIdx.x == mt.c_first ? 1 : 0)) * RB;
        for (int idx = tid; idx < RB * D; idx += S::kThreads) {
            const int r = idx / D, d = idx % D;
            const int rg = mt.rb * RB + r;
            if (rg >= a.rows) continue;
            float M = kNegInf;
#pragma unroll
            for (int w = 0; w < S::kNW; ++w) M = fmaxf(M, ep_m[w * RB + r]);
            float num = 0.f, den = 0.f;
#pragma unroll
            for (int w = 0; w < S::kNW; ++w) {
                const float wt = safe_weight(ep_m[w * RB + r], M);
                num = fmaf(wt, ep_o[(w * RB + r) * D + d], num);
                den = fmaf(wt, ep_l[w * RB + r], den);
            }
            if (single) {
                if constexpr (kQuant)  // values are stored / v_scale
                    Tq::store(static_cast<T *>(a.out) + ((size_t)mt.bh * a.rows + rg) * D + d,
                              num / den * a.kv_scale.y);
                else
                    Tq::store(static_cast<T *>(a.out) + ((size_t)mt.bh * a.rows + rg) * D + d, num / den);
            } else if constexpr (kCluster) {
                float *pr = cl_part + r * (D + 2);
                st_cluster_f32(pr + d, 0u, num);
                if (d == 0) {
                    st_cluster_f32(pr + D, 0u, M);
                    st_cluster_f32(pr + D + 1, 0u, den);
                }
            } else {
                float *pr = a.part + (pbase + r) * (D + 4);
                pr[d] = num;
                if (d == 0) {
                    pr[D] = M;
                    pr[D + 1] = den;
                }
            }
        }
        if constexpr (kCluster) ++n_pieces;
        if constexpr (kTicketMerge && !kCluster) {
            if (!single) {  // (a range holds at most two split pieces: the head it continues, the head it starts)
                if (tid == 0 && n_pieces < 2) jobs[n_pieces] = MergeJob{mt.bh, mt.rb, mt.c_first, mt.n_chunks};
                ++n_pieces;
            }
        }
    }

    if (tid == 0) {  // (as above: the barriers below need every thread)
        ctl.described(issued);
        ctl.final_count(issued);
    }
    if constexpr (kCluster) {
        // ---- merge the cluster's pieces in rank 0 ----
        const uint32_t crank = cluster_ctarank();
        float *cl_base = reinterpret_cast<float *>(smem + S::kFixedBytes);
        if (n_pieces == 0) {  // an empty share: a piece of weight zero
            float *pr = cl_base + crank * RB * (D + 2);
            for (int idx = tid; idx < RB * (D + 2); idx += S::kThreads)
                st_cluster_f32(pr + idx, 0u, (idx % (D + 2) == D) ? kNegInf : 0.f);
        }
        cluster_arrive_release();  // this CTA's piece is in rank 0
        if (crank == 0) {
            cluster_wait_acquire();  // every piece is in
            if (*cl_ok) {
                const int csize = (int)cluster_nctarank();
                const int HR = a.H_kv * a.n_rowblocks;
                const int u = (int)blockIdx.x / csize;
                const int bh = (u / HR) * a.H_kv + (u % HR) / a.n_rowblocks, rb = (u % HR) % a.n_rowblocks;
                for (int idx = tid; idx < RB * D; idx += S::kThreads) {
                    const int r = idx / D, d = idx % D;
                    const int rg = rb * RB + r;
                    if (rg >= a.rows) continue;
                    float M = kNegInf;
                    for (int k = 0; k < csize; ++k) M = fmaxf(M, cl_base[(k * RB + r) * (D + 2) + D]);
                    float num = 0.f, den = 0.f;
                    for (int k = 0; k < csize; ++k) {
                        const float *pr = cl_base + (k * RB + r) * (D + 2);
                        const float wt = safe_weight(pr[D], M);
                        num = fmaf(wt, pr[d], num);
                        den = fmaf(wt, pr[D + 1], den);
                    }
                    if constexpr (kQuant)  // values are stored / v_scale
                        Tq::store(static_cast<T *>(a.out) + ((size_t)bh * a.rows + rg) * D + d,
                                  num / den * a.kv_scale.y);
                    else
                        Tq::store(static_cast<T *>(a.out) + ((size_t)bh * a.rows + rg) * D + d, num / den);
                }
            }
        }
        // (the other CTAs may exit now: no one reads their shared memory)
    } else if constexpr (kTicketMerge) {
        // ---- count this CTA's split pieces; merge the heads they complete ----
        n_pieces = min(n_pieces, 2);
        __syncthreads();  // every thread's share of the partials is written
        if (tid == 0 && n_pieces > 0) {
            int *tickets = static_cast<int *>(a.merge_state);
            // Each count releases this CTA's partials and, for the count that
            // completes a head, acquires the other CTAs' (acquire-release atomics).
            int seen[2];
#pragma unroll
            for (int i = 0; i < 2; ++i)
                if (i < n_pieces) seen[i] = atomic_add_acq_rel_gpu(tickets + (size_t)jobs[i].bh * a.n_rowblocks + jobs[i].rb, 1);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                if (i < n_pieces && seen[i] == jobs[i].n_chunks - 1)
                    tickets[(size_t)jobs[i].bh * a.n_rowblocks + jobs[i].rb] = 0;  // the next call starts from zero
                else
                    jobs[i].n_chunks = 0;  // another CTA completes this head (or no piece)
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const MergeJob job = jobs[i];
            if (i < n_pieces && job.n_chunks)
                merge_pieces<T, D, RB, S::kThreads, kQuant>(a, job, reinterpret_cast<float *>(smem + S::kEpiOff),
                                                            tid);
        }
    }

    if (tid == 0 && gave_up && first_unwaited >= 0) {
        // Copies that may still be in flight must land before the CTA exits:
        // wait for every issued position from the first abandoned one, one deadline.
        const uint64_t t0 = global_timer_ns();
        for (int p = first_unwaited; p < issued; ++p) {
            const uint32_t ph = (uint32_t)(p / S::kStages) & 1u;
            while (!mbar_try_wait(&full[p % S::kStages], ph) && global_timer_ns() - t0 < kDrainLimitNs) {
            }
        }
    }
}

// Second pass: log-sum-exp merge of the pieces of a query row.
//   M = max_c m_c;  w_c = 2^(m_c - M);  out = sum_c w_c o_c / sum_c w_c l_c
// (times v_scale with an E4M3 cache: kScaleV).  The warps stride over the
// heads' real rows (B * H_kv * rows; a row block's padding rows have none),
// so the host may launch fewer warps than rows.  A warp takes one row at a
// time when the grid has a warp per row, else kMergeRows consecutive rows of
// one head with the loads of all of them in flight together (a row alone is
// two dependent memory round trips).  Measured on GB300 (long-context layer):
// one row per warp is best at 1024 rows, two at 8192 and 32768 rows.
constexpr int kMergeRows = 2;

template <typename T, int D, int RB, bool kScaleV = false>
__global__ void __launch_bounds__(128) attn_merge_kernel(const AttnArgs a)
{
    using Ty = Elem<T>;
    const float kNegInf = __int_as_float(0xff800000);
    constexpr int kDpl = D / 32;
    constexpr int kR = kMergeRows;
    // The next kernel may launch at once: like every kernel here it waits for
    // this grid's completion before it touches anything this grid writes,
    // and launching early lets its CTAs take the SMs as these warps finish.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x % 32;
    const int HR = a.H_kv * a.n_rowblocks;
    const long long stride = (long long)gridDim.x * (blockDim.x / 32);
    const int kr = (long long)a.B * a.H_kv * a.rows > stride ? kR : 1;  // rows per warp at a time
    const int gph = (a.rows + kr - 1) / kr;  // row groups per head
    const long long n_groups = (long long)a.B * a.H_kv * gph;
    const int prow = part_rows<RB>(a.rows);
    for (long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / 32; gw < n_groups; gw += stride) {
        const int bh = (int)(gw / gph);
        const int rg0 = (int)(gw % gph) * kr;
        const int b = bh / a.H_kv, h = bh % a.H_kv;
        // (all loads issued before any is used)
        const int P = __ldg(a.past_len + b);
        int2 seg[kR];
#pragma unroll
        for (int i = 0; i < kR; ++i)
            seg[i] = i < kr && rg0 + i < a.rows
                         ? static_cast<const int2 *>(a.merge_state)[(size_t)b * HR + h * a.n_rowblocks + (rg0 + i) / RB]
                         : make_int2(0, 0);
        if (!past_len_ok(P, a.N, a.T_max, a.max_past_len)) continue;  // reported by the split pass
        // pieces to merge per row (0: the split pass wrote the row directly)
        int cnt[kR], kmax = 0;
#pragma unroll
        for (int i = 0; i < kR; ++i) {
            cnt[i] = seg[i].y > 1 ? seg[i].y : 0;
            kmax = max(kmax, cnt[i]);
        }
        if (kmax == 0) continue;

        // One pass over the pieces, merged online (running max M, weighted
        // sums); two pieces of every row loaded before their updates.
        float M[kR], den[kR], acc[kR][kDpl];
#pragma unroll
        for (int i = 0; i < kR; ++i) {
            M[i] = kNegInf;
            den[i] = 0.f;
#pragma unroll
            for (int k = 0; k < kDpl; ++k) acc[i][k] = 0.f;
        }
        for (int k0 = 0; k0 < kmax; k0 += 2) {
            float2 ml[kR][2];
            float ov[kR][2][kDpl];
#pragma unroll
            for (int i = 0; i < kR; ++i) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int k = k0 + j;
                    if (k < cnt[i]) {
                        const size_t pidx = ((size_t)(seg[i].x + k) * 2 + (k == 0)) * prow + (rg0 + i) % RB;
                        const float *pr = a.part + pidx * (D + 4);
                        ml[i][j] = *reinterpret_cast<const float2 *>(pr + D);
                        const float *po = pr + lane * kDpl;
                        if constexpr (kDpl == 4) {
                            const float4 v = *reinterpret_cast<const float4 *>(po);
                            ov[i][j][0] = v.x;
                            ov[i][j][1] = v.y;
                            ov[i][j][2] = v.z;
                            ov[i][j][3] = v.w;
                        } else {
#pragma unroll
                            for (int k2 = 0; k2 < kDpl; ++k2) ov[i][j][k2] = po[k2];
                        }
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < kR; ++i) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    if (k0 + j < cnt[i]) {
                        const float Mn = fmaxf(M[i], ml[i][j].x);
                        const float wa = safe_weight(M[i], Mn), wb = safe_weight(ml[i][j].x, Mn);
                        den[i] = den[i] * wa + ml[i][j].y * wb;
#pragma unroll
                        for (int k2 = 0; k2 < kDpl; ++k2) acc[i][k2] = acc[i][k2] * wa + ov[i][j][k2] * wb;
                        M[i] = Mn;
                    }
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kR; ++i) {
            if (cnt[i] == 0) continue;
            T *out = static_cast<T *>(a.out) + ((size_t)bh * a.rows + rg0 + i) * D + lane * kDpl;
#pragma unroll
            for (int k = 0; k < kDpl; ++k) {
                if constexpr (kScaleV)
                    Ty::store(out + k, acc[i][k] / den[i] * a.kv_scale.y);
                else
                    Ty::store(out + k, acc[i][k] / den[i]);
            }
        }
    }
}

// Launch facts of one compiled variant, for the host planner.
struct AttnVariant {
    const void *fn;        // attention over an appended cache
    const void *fused_fn;  // append + attention (kvd_decode_step)
    const void *merge_fn;  // the separate merge pass
    int threads;
    int fixed_smem_bytes;  // plus (2B + 1) ints, rounded to 16 bytes
    int tile_keys;
    int rows_per_block;
    int piece_units;       // cost of a piece boundary in tile units
    bool tma = false;      // tensor-core kernel: takes the K and V tensor maps
    bool q_map = false;    // tcgen05 kernel: also a Q tensor map (128-row boxes)
    int stages = 0;        // ring stages
    const void *cluster_fn = nullptr;        // cluster mode (contiguous, small layers), attention
    const void *cluster_fused_fn = nullptr;  // cluster mode, fused step
};

template <typename T, int D, int RB, bool kTicketMerge, bool kPaged, typename C = T> AttnVariant make_variant()
{
    using S = AttnShape<T, D, RB, C>;
    constexpr bool kQuant = !std::is_same<T, C>::value;
    AttnVariant v;
    v.fn = reinterpret_cast<const void *>(&attn_balanced_kernel<T, D, RB, false, kTicketMerge, kPaged, C>);
    v.fused_fn = reinterpret_cast<const void *>(&attn_balanced_kernel<T, D, RB, true, kTicketMerge, kPaged, C>);
    if constexpr (kTicketMerge) v.merge_fn = nullptr;
    else v.merge_fn = reinterpret_cast<const void *>(&attn_merge_kernel<T, D, RB, kQuant>);
    if constexpr (kTicketMerge) {  // (built with the in-kernel-merge variants)
        v.cluster_fn = reinterpret_cast<const void *>(&attn_balanced_kernel<T, D, RB, false, true, kPaged, C, true>);
        v.cluster_fused_fn = reinterpret_cast<const void *>(&attn_balanced_kernel<T, D, RB, true, true, kPaged, C, true>);
    }
    v.threads = S::kThreads;
    v.fixed_smem_bytes = S::kFixedBytes;
    v.tile_keys = S::kTK;
    v.rows_per_block = RB;
    v.piece_units = S::kPieceUnits;
    v.stages = S::kStages;
    return v;
}

template <typename T, int D, bool kTicketMerge, bool kPaged, typename C = T> bool pick_rb(int RB, AttnVariant *v)
{
    switch (RB) {
    case 1: *v = make_variant<T, D, 1, kTicketMerge, kPaged, C>(); return true;
    case 2: *v = make_variant<T, D, 2, kTicketMerge, kPaged, C>(); return true;
    case 4: *v = make_variant<T, D, 4, kTicketMerge, kPaged, C>(); return true;
    case 8:  // (an E4M3 cache keeps row blocks of at most 4: 8 would need twice the q registers)
        if constexpr (std::is_same<T, C>::value) {
            *v = make_variant<T, D, 8, kTicketMerge, kPaged>();
            return true;
        } else {
            return false;
        }
    default: return false;
    }
}

template <typename T, bool kTicketMerge, bool kPaged, typename C = T> bool pick_variant(int D, int RB, AttnVariant *v)
{
    switch (D) {
    case 64: return pick_rb<T, 64, kTicketMerge, kPaged, C>(RB, v);
    case 128: return pick_rb<T, 128, kTicketMerge, kPaged, C>(RB, v);
    default: return false;
    }
}

// One translation unit each: kvd_attn_{f32,bf16,f16}[_tk][_paged].cu -- merge
// pass or in-kernel merge (_tk), contiguous or paged cache (_paged).
bool attn_variant_f32(int D, int RB, AttnVariant *v);
bool attn_variant_bf16(int D, int RB, AttnVariant *v);
bool attn_variant_f32_tk(int D, int RB, AttnVariant *v);
bool attn_variant_bf16_tk(int D, int RB, AttnVariant *v);
bool attn_variant_f32_paged(int D, int RB, AttnVariant *v);
bool attn_variant_bf16_paged(int D, int RB, AttnVariant *v);
bool attn_variant_f32_tk_paged(int D, int RB, AttnVariant *v);
bool attn_variant_bf16_tk_paged(int D, int RB, AttnVariant *v);
bool attn_variant_f16(int D, int RB, AttnVariant *v);
bool attn_variant_f16_tk(int D, int RB, AttnVariant *v);
bool attn_variant_f16_paged(int D, int RB, AttnVariant *v);
bool attn_variant_f16_tk_paged(int D, int RB, AttnVariant *v);
bool attn_variant_e4m3(int D, int RB, AttnVariant *v);      // bf16 q / out, E4M3 cache
bool attn_variant_e4m3_tk(int D, int RB, AttnVariant *v);
// tensor-core kernels (kvd_attention_mma.cuh): 16-row blocks, contiguous or paged caches
bool attn_variant_mma_bf16(int D, bool paged, AttnVariant *v);
bool attn_variant_mma_bf16_tk(int D, bool paged, AttnVariant *v);
bool attn_variant_mma_f16(int D, bool paged, AttnVariant *v);
bool attn_variant_mma_f16_tk(int D, bool paged, AttnVariant *v);
bool attn_variant_mma_e4m3(int D, int rows, AttnVariant *v);  // bf16 q / out, E4M3 cache, D = 128
bool attn_variant_mma_e4m3_tk(int D, int rows, AttnVariant *v);
// tcgen05 kernels (kvd_attention_tc5.cuh): 128-row blocks, contiguous or paged caches
bool attn_variant_tc5_bf16(int D, bool paged, AttnVariant *v);
bool attn_variant_tc5_bf16_tk(int D, bool paged, AttnVariant *v);
bool attn_variant_tc5_f16(int D, bool paged, AttnVariant *v);
bool attn_variant_tc5_f16_tk(int D, bool paged, AttnVariant *v);

}  // namespace kvd
