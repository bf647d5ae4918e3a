// kvd_attention_tc5.cuh -- split-T decode attention for many query rows per
// KV head on the fifth-generation tensor cores (tcgen05, accumulators in
// tensor memory).
//
// The same computation as attn_balanced_kernel and attn_mma_kernel
// (offset-causal GQA decode attention, "7.1 自回归生成过程", code 1-2;
// "GPT-2缓存实测：千倍计算只快6倍", section "一个很容易漏掉的错误"), with
// their split, tile ring, partial layout and merges, for blocks of up to 128
// query rows.  It serves chunked decode and chunked prefill with g * N > 16
// rows per KV head, where the 16-row mma.sync blocks would read every K/V
// tile once per block.  One CTA per SM, seven warps:
//   * warp 4, the producer: the unit prefix over past_len and the range walk
//     (RangeWalk); K/V tiles by 2-D TMA into a ring of kStages stages, and the
//     Q block of each piece (128 rows x D, through a third tensor map) into
//     one Q buffer;
//   * warp 5, the S warp: allocates the tensor memory; writes the new rows of
//     a fused step into the tile (and the cache) and zeroes value rows past
//     the sequence end; one thread issues S_j = Q . K_j^T (M = 128 rows,
//     N = 64 keys) into score buffer j % 2 as soon as the tile and the buffer
//     are free;
//   * warp 6, the P . V warp: one thread issues O += P_j . V_j (M = 128,
//     N = D, O in tensor memory) as soon as P_j is written, which also
//     releases the ring slot; both issuers signal completion by
//     tcgen05.commit on mbarriers;
//   * warps 0-3, the softmax warps: thread r owns query row r (tensor-memory
//     lane r).  It loads the row's 64 scores, masks them, keeps the running
//     max and sum in registers (a row is one thread: no shuffles), writes the
//     weights P (bf16 / fp16) into its tensor-memory lane as the A operand of
//     P . V (no shared-memory round trip), rescales its O row in tensor
//     memory when the max grows by more than 2^8, and at the end of a piece
//     reads O back and writes the output row or the piece's partial (o, m, l).
// Shared-memory operands are 128-byte swizzled: Q and K K-major (the head
// dimension contiguous), V MN-major (D contiguous), each described to the
// tensor core by a shared-memory matrix descriptor.
//
// Every mbarrier is waited for phase by phase in order, so a parity never
// stands for two phases; every wait is bounded and also ends when another
// warp of the CTA has given up (abort flag), and a CTA that gave up still
// drains its copies and MMAs before it frees the tensor memory.
#pragma once

#include <type_traits>

#include "kvd_attention.cuh"

namespace kvd {

// ---- tcgen05 primitives ----

// Allocate ncols tensor-memory columns (whole warp); the address is written
// to shared memory at dst.
__device__ __forceinline__ void tc5_alloc(uint32_t *dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc5_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc5_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Order tensor-core operations of this thread before / after a thread
// synchronisation (an mbarrier arrive or wait, a CTA barrier).
__device__ __forceinline__ void tc5_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc5_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive once on bar when every tcgen05.mma this thread issued so far is complete.
__device__ __forceinline__ void tc5_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

// D (tensor memory) = A . B (+ D when accumulate), 16-bit operands from
// shared memory, fp32 accumulators.
__device__ __forceinline__ void tc5_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate)
{
    asm volatile(
        "{\n"
        "  .reg .pred p;\n"
        "  setp.ne.b32 p, %4, 0;\n"
        "  tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same with A (M rows x K) in tensor memory at a_tmem: row i in lane i,
// two 16-bit elements per 32-bit column, K / 2 consecutive columns.
__device__ __forceinline__ void tc5_mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate)
{
    asm volatile(
        "{\n"
        "  .reg .pred p;\n"
        "  setp.ne.b32 p, %4, 0;\n"
        "  tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Instruction descriptor of a kind::f16 MMA with fp32 accumulators: A and B
// bf16 (else fp16), M x N, each operand K-major or MN-major.
template <bool kBf16> __host__ __device__ constexpr uint32_t tc5_idesc(int M, int N, bool a_mn, bool b_mn)
{
    return (1u << 4)                                // D format: fp32
           | ((kBf16 ? 1u : 0u) << 7)               // A format
           | ((kBf16 ? 1u : 0u) << 10)              // B format
           | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16)
           | ((uint32_t)(N >> 3) << 17)             // N / 8
           | ((uint32_t)(M >> 4) << 24);            // M / 16
}

// Shared-memory matrix descriptor of a 128-byte-swizzled operand at shared
// address saddr: lbo / sbo the byte strides between 128-byte-swizzle atoms
// along the leading (MN-major: MN) and strided (8-row groups) dimensions.
__device__ __forceinline__ uint64_t tc5_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((saddr & 0x3ffffu) >> 4)              // start address / 16
           | ((uint64_t)((lbo >> 4) & 0x3fffu) << 16)        // leading byte offset / 16
           | ((uint64_t)((sbo >> 4) & 0x3fffu) << 32)        // stride byte offset / 16
           | (1ull << 46)                                    // descriptor version
           | (2ull << 61);                                   // 128-byte swizzle
}

// tcgen05.ld of 64 consecutive 32-bit TMEM columns of this thread's lane
// (32x32b shape: thread i of the warp reads lane (warp % 4) * 32 + i), waited
// for in the same statement so no use of the registers can move above the wait.
__device__ __forceinline__ void tc5_ld64(uint32_t taddr, uint32_t (&r)[64])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr)
        : "memory");
}

// tcgen05.ld of 32 consecutive 32-bit TMEM columns of this thread's lane
// (32x32b shape: thread i of the warp reads lane (warp % 4) * 32 + i), waited
// for in the same statement so no use of the registers can move above the wait.
__device__ __forceinline__ void tc5_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// tcgen05.st of 32 consecutive 32-bit TMEM columns of this thread's lane,
// waited for in the same statement.
__device__ __forceinline__ void tc5_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n"
        "tcgen05.wait::st.sync.aligned;\n"
        :
        : "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// ---- shape and shared-memory layout ----

// 128-row blocks, 64-key tiles, 16-bit caches, D = 64 or 128.  Member names
// match AttnShape where RangeWalk uses them.
template <typename T, int D> struct Tc5Shape {
    static constexpr bool kTma = true;
    static constexpr bool kQInRing = false;        // Q has its own buffer and tensor map
    static constexpr int kRB = 128;
    static constexpr int kRowBytes = D * 2;
    static constexpr int kQRowBytes = D * 2;
    static constexpr int kTK = 64;
    static constexpr int kBoxCols = 64;            // elements per 128-byte box row
    static constexpr int kBoxes = D / 64;
    static constexpr int kBoxBytes = kTK * 128;    // K / V box: 64 keys x 128 bytes
    static constexpr int kTileBytes = kBoxes * kBoxBytes;
    // (a ring slot is released by its tile's P . V: the stages beyond the
    // two being computed are the copies in flight)
    static constexpr int kStages = D == 128 ? 5 : 8;
    // Cost of a piece boundary in tile units for the static split: a piece
    // ends with its 128-row epilogue and starts with a Q load (measured on
    // GB300 at 128 rows per KV head: 2 units 191.8 us, 4 183.8, 6 181.5).
    static constexpr int kPieceUnits = 6;
    static constexpr int kQBoxBytes = kRB * 128;   // Q box: 128 rows x 128 bytes
    static constexpr int kQBytes = kBoxes * kQBoxBytes;
    static constexpr int kThreads = 224;
    static constexpr int kTmemCols = 512;
    static constexpr int kTmemS = 0;               // two score buffers of 64 columns
    static constexpr int kTmemO = 128;             // O: D columns
    static constexpr int kTmemP = 256;             // two P buffers of 32 columns (64 keys, 16-bit pairs)

    static constexpr int kRingOff = 0;
    static constexpr int kQOff = kRingOff + kStages * 2 * kTileBytes;  // the Q buffer
    static constexpr int kQSlotBytes = 0;          // (no q in the ring stages)
    static constexpr int kMetaOff = kQOff + kQBytes;
    static constexpr int kBarOff = kMetaOff + kStages * (int)sizeof(TileMeta);
    // full[kStages], empty[kStages], q_full, q_empty, s_full[2], s_free[2],
    // p_full[2], p_empty[2], mma_done[2] (the S and the P . V issuer)
    static constexpr int kNumBars = 2 * kStages + 12;
    static constexpr int kJobOff = kBarOff + kNumBars * 8;
    static constexpr int kPageOff = kJobOff + 2 * (int)sizeof(MergeJob);
    static constexpr int kMiscOff = kPageOff + 4 * kStages;  // tensor-memory base, abort flag
    static constexpr int kFixedBytes = kMiscOff + 16;

    static_assert(D == 64 || D == 128, "head dim");
    static_assert(kQOff % 1024 == 0 && kTileBytes % 1024 == 0, "swizzle atoms");
    static_assert(kTmemO + D <= kTmemP && kTmemP + 2 * (kTK / 2) <= kTmemCols, "tensor memory columns");
    static_assert(kFixedBytes + 4096 <= 227 * 1024, "shared memory");
};

// Shared address of the 16-byte chunk c (0 .. D/8-1) of row r of a tile of
// 128-byte-swizzled boxes (64 rows x 128 bytes) at shared address tile.
template <typename S> __device__ __forceinline__ uint32_t tc5_chunk_addr(uint32_t tile, int r, int c)
{
    const uint32_t lin = tile + (c >> 3) * S::kBoxBytes + r * 128 + ((c & 7) << 4);
    return lin ^ ((lin >> 3) & 0x70u);
}

// Bounded wait for phase `parity` of bar; also gives up once *abort is set.
__device__ __forceinline__ bool tc5_wait(uint64_t *bar, uint32_t parity, volatile uint32_t *abort)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0u && (*abort != 0u || global_timer_ns() - t0 > kWaitLimitNs)) return false;
    }
}

__device__ __forceinline__ void named_barrier_sync(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// The MMA warp's repairs of a tile before S = Q . K^T reads it: in a fused
// step the new keys P .. P+N-1 it holds are copied from k_new / v_new into
// the tile (and, by row block 0, into the cache: kc / vc address the cache row
// of the tile's first key); value rows at or past the sequence end are zeroed
// (a zero weight times a stale NaN is NaN inside the MMA).
template <typename T, int D, bool kFused>
__device__ __forceinline__ void tc5_fix_tile(const AttnArgs &a, uint32_t Ks, uint32_t Vs, const TileMeta &mt,
                                             unsigned char *kc, unsigned char *vc, int lane)
{
    using S = Tc5Shape<T, D>;
    constexpr int kChunks = S::kRowBytes / 16;
    const int k_end = mt.tile_k0 + mt.nk;
    if constexpr (kFused) {
        const int lo = max(0, mt.P - mt.tile_k0), hi = k_end - mt.tile_k0;
        if (lo < hi) {
            const unsigned char *kn = static_cast<const unsigned char *>(a.k_new) + (size_t)mt.bh * a.N * S::kRowBytes;
            const unsigned char *vn = static_cast<const unsigned char *>(a.v_new) + (size_t)mt.bh * a.N * S::kRowBytes;
            const int n = (hi - lo) * kChunks;
            // batches of 8 chunks per lane: all loads of a batch in flight
            // before its stores (a chunk at a time would wait a full load
            // latency per chunk)
            for (int base = 0; base < n; base += 8 * 32) {
                uint4 kv[8], vv[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int idx = base + u * 32 + lane;
                    if (idx < n) {
                        const int r = lo + idx / kChunks, c = idx % kChunks;
                        const size_t nrow = (size_t)(mt.tile_k0 + r - mt.P) * S::kRowBytes + c * 16;
                        kv[u] = ldg128_nc(kn + nrow);
                        vv[u] = ldg128_nc(vn + nrow);
                    }
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int idx = base + u * 32 + lane;
                    if (idx < n) {
                        const int r = lo + idx / kChunks, c = idx % kChunks;
                        sts128(tc5_chunk_addr<S>(Ks, r, c), kv[u]);
                        sts128(tc5_chunk_addr<S>(Vs, r, c), vv[u]);
                        if (kc != nullptr) {
                            stg128(kc + (size_t)r * S::kRowBytes + c * 16, kv[u]);
                            stg128(vc + (size_t)r * S::kRowBytes + c * 16, vv[u]);
                        }
                    }
                }
            }
        }
    }
    for (int idx = lane; idx < (S::kTK - mt.nk) * kChunks; idx += 32) {
        const int r = mt.nk + idx / kChunks, c = idx % kChunks;
        sts128(tc5_chunk_addr<S>(Vs, r, c), make_uint4(0u, 0u, 0u, 0u));
    }
}

// Log-sum-exp merge of a split head's pieces, one warp per query row (the
// four softmax warps share the rows): the pieces' partials were written by the
// CTAs c_first .. c_first + n_chunks - 1 (slot 1 of the first, else slot 0).
template <typename T, int D>
__device__ __forceinline__ void tc5_merge_rows(const AttnArgs &a, const MergeJob &job, int warp, int lane)
{
    using Tq = Elem<T>;
    constexpr int kRB = Tc5Shape<T, D>::kRB;
    constexpr int kDpl = D / 32;
    const float kNegInf = __int_as_float(0xff800000);
    const int prow = part_rows<kRB>(a.rows);
    const int n_rows = min(kRB, a.rows - job.rb * kRB);
    for (int r = warp; r < n_rows; r += 4) {
        float M = kNegInf;
        for (int k = lane; k < job.n_chunks; k += 32)
            M = fmaxf(M, __ldcg(a.part + (((size_t)(job.c_first + k) * 2 + (k == 0)) * prow + r) * (D + 4) + D));
#pragma unroll
        for (int off = 16; off >= 1; off /= 2) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        float acc[kDpl];
#pragma unroll
        for (int i = 0; i < kDpl; ++i) acc[i] = 0.f;
        float den = 0.f;
        for (int k = 0; k < job.n_chunks; ++k) {
            const float *pr = a.part + (((size_t)(job.c_first + k) * 2 + (k == 0)) * prow + r) * (D + 4);
            const float2 ml = __ldcg(reinterpret_cast<const float2 *>(pr + D));
            const float w = safe_weight(ml.x, M);
            den = fmaf(w, ml.y, den);
#pragma unroll
            for (int i = 0; i < kDpl; ++i) acc[i] = fmaf(w, __ldcg(pr + lane * kDpl + i), acc[i]);
        }
        T *dst = static_cast<T *>(a.out) + ((size_t)job.bh * a.rows + job.rb * kRB + r) * D + lane * kDpl;
#pragma unroll
        for (int i = 0; i < kDpl; ++i) Tq::store(dst + i, acc[i] / den);
    }
}

// The kernel.  kFused: append + attention (kvd_decode_step); kTicketMerge:
// split heads merged at the end of the kernel by the CTA that completes them,
// else by the separate merge pass; kPaged: tiles from a page pool.
template <typename T, int D, bool kFused, bool kTicketMerge, bool kPaged>
__global__ void __launch_bounds__(224, 1)
    attn_tc5_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_q)
{
    using S = Tc5Shape<T, D>;
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr float kRescaleThreshold = 8.0f;
    const float kNegInf = __int_as_float(0xff800000);
    extern __shared__ __align__(1024) unsigned char smem_tc5[];
    unsigned char *smem = smem_tc5;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::kBarOff);
    uint64_t *empty = full + S::kStages;
    uint64_t *q_full = empty + S::kStages, *q_empty = q_full + 1;
    uint64_t *s_full = q_full + 2, *s_free = s_full + 2, *p_full = s_free + 2, *p_empty = p_full + 2;
    uint64_t *mma_done = p_empty + 2;
    TileMeta *meta = reinterpret_cast<TileMeta *>(smem + S::kMetaOff);
    MergeJob *jobs = reinterpret_cast<MergeJob *>(smem + S::kJobOff);
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + S::kMiscOff);  // [0] tensor memory, [1] abort
    volatile uint32_t *abort = misc + 1;
    int *pre = reinterpret_cast<int *>(smem + S::kFixedBytes);
    int *pl = pre + a.B + 1;

    const int tid = threadIdx.x;
    const int warp = tid / 32, lane = tid % 32;

    // The swizzled boxes need 1024-byte-aligned shared memory (checked; every
    // thread takes the same branch, before any barrier or allocation).
    if ((smem_addr(smem) & 1023u) != 0) {
        if (tid == 0) raise_error(a.err_word, KVD_DEVERR_INTERNAL);
        return;
    }
    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < S::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_free[i], 128);
            mbar_init(&p_full[i], 128);
            mbar_init(&p_empty[i], 1);
        }
        mbar_init(&mma_done[0], 1);
        mbar_init(&mma_done[1], 1);
        misc[1] = 0u;
        fence_mbar_init();
    }
    if (warp == 5) {
        tc5_alloc(&misc[0], S::kTmemCols);
        tc5_relinquish();
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // (as attn_balanced_kernel)
    tc5_fence_before();
    __syncthreads();
    tc5_fence_after();
    const uint32_t tmem = misc[0];
    const uint32_t ring = smem_addr(smem + S::kRingOff);
    const uint32_t qbuf = smem_addr(smem + S::kQOff);

    if (warp == 4) {
        // ---- producer: unit prefix over sequences (warp scan), then the walk ----
        int carry = 0;
        if (lane == 0) pre[0] = 0;
        for (int b0 = 0; b0 < a.B; b0 += 32) {
            const int b = b0 + lane;
            int units = 0;
            if (b < a.B) {
                const int P = __ldg(a.past_len + b);
                const bool ok = past_len_ok(P, a.N, a.T_max, a.max_past_len);
                if (!ok && blockIdx.x == 0) raise_error(a.err_word, KVD_DEVERR_PAST_LEN);
                units = ok ? (P + a.N + S::kTK - 1) / S::kTK + S::kPieceUnits : 0;
                pl[b] = P;
            }
            int v = units;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, v, off);
                if (lane >= off) v += n;
            }
            if (b < a.B) pre[b + 1] = carry + v;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
        __syncwarp();
        if (lane == 0) {
            RangeWalk<S, !kTicketMerge, kPaged> walk;
            const int HR = a.H_kv * a.n_rowblocks;
            const long long n_total = (long long)pre[a.B] * HR;
            const long long G = min((long long)gridDim.x, n_total);
            const long long lo = blockIdx.x < G ? n_total * blockIdx.x / G : 0;
            const long long hi = blockIdx.x < G ? n_total * (blockIdx.x + 1) / G : 0;
            walk.tm_k = &tm_k;
            walk.tm_v = &tm_v;
            walk.start(a, pre, pl, lo, hi, n_total, G);
            int issued = 0, q_loads = 0;
            bool dead = false;
            while (!walk.ended) {
                const int s = issued % S::kStages;
                // the slot's previous tile (issued - kStages) is released by its P . V
                if (issued >= S::kStages && !tc5_wait(&empty[s], (uint32_t)((issued / S::kStages) - 1) & 1u, abort)) {
                    dead = true;
                    break;
                }
                const bool q_load = walk.t < walk.hi && walk.piece_start;
                const int qy = walk.bh * a.rows + walk.rb * S::kRB;  // first q row of the piece's block
                walk.fill(a, pre, pl, smem, meta, full, s);
                ++issued;
                if (q_load) {
                    // the Q buffer is free once the previous piece's last S was computed
                    if (q_loads > 0 && !tc5_wait(q_empty, (uint32_t)(q_loads - 1) & 1u, abort)) {
                        dead = true;
                        break;
                    }
                    mbar_arrive_expect_tx(q_full, (uint32_t)S::kQBytes);
#pragma unroll
                    for (int bx = 0; bx < S::kBoxes; ++bx)
                        tma_load_2d(smem + S::kQOff + bx * S::kQBoxBytes, &tm_q, bx * S::kBoxCols, qy, q_full,
                                    walk.policy);
                    ++q_loads;
                }
            }
            if (dead) {
                *abort = 1u;
                raise_error(a.err_word, KVD_DEVERR_TIMEOUT);
                // copies still in flight land before the CTA exits: the last
                // position of each stage, and the last Q block (one deadline)
                const uint64_t t0 = global_timer_ns();
                for (int p = max(0, issued - S::kStages); p < issued; ++p)
                    while (!mbar_try_wait(&full[p % S::kStages], (uint32_t)(p / S::kStages) & 1u) &&
                           global_timer_ns() - t0 < kDrainLimitNs) {
                    }
                if (q_loads > 0)
                    while (!mbar_try_wait(q_full, (uint32_t)(q_loads - 1) & 1u) && global_timer_ns() - t0 < kDrainLimitNs) {
                    }
            }
        }
    } else if (warp == 5) {
        // ---- S warp: repairs the tiles, one thread issues S_j = Q . K_j^T ----
        constexpr uint32_t kIdescS = tc5_idesc<kBf16>(128, S::kTK, false, false);
        bool dead = false;
        int n_pieces = 0;
        for (int pos = 0;; ++pos) {
            const int st = pos % S::kStages;
            int ok = 1;
            if (lane == 0) ok = tc5_wait(&full[st], (uint32_t)(pos / S::kStages) & 1u, abort) ? 1 : 0;
            __syncwarp();
            if (!__shfl_sync(0xffffffffu, ok, 0)) {
                dead = true;
                break;
            }
            const TileMeta mt = meta[st];
            if (mt.flags & kMetaEnd) break;
            const bool first = (mt.flags & kMetaFirst) != 0;
            if (first) ++n_pieces;
            const uint32_t kt = ring + st * 2 * S::kTileBytes;
            if ((kFused && mt.tile_k0 + S::kTK > mt.P) || mt.nk < S::kTK) {
                unsigned char *kc = nullptr, *vc = nullptr;
                if constexpr (kFused) {
                    size_t crow = 0;  // cache row of the tile's first key
                    bool write = mt.rb == 0;  // one row block writes the new rows into the cache
                    if constexpr (kPaged) {
                        const int page = reinterpret_cast<const int *>(smem + S::kPageOff)[st];
                        write = write && page >= 0;  // (none into an invalid page)
                        crow = (((size_t)page * a.H_kv + mt.bh % a.H_kv) << a.page_shift) +
                               (mt.tile_k0 & ((1 << a.page_shift) - 1));
                    } else {
                        crow = (size_t)mt.bh * a.T_max + mt.tile_k0;
                    }
                    if (write) {
                        kc = static_cast<unsigned char *>(const_cast<void *>(a.k_cache)) + crow * S::kRowBytes;
                        vc = static_cast<unsigned char *>(const_cast<void *>(a.v_cache)) + crow * S::kRowBytes;
                    }
                }
                tc5_fix_tile<T, D, kFused>(a, kt, kt + S::kTileBytes, mt, kc, vc, lane);
                fence_proxy_async_shared();  // generic writes before the tensor core reads the tile
                __syncwarp();
            }
            if (lane == 0) {
                if (first && !tc5_wait(q_full, (uint32_t)(n_pieces - 1) & 1u, abort)) ok = 0;
                // the score buffer was last read by the softmax of tile pos - 2
                if (ok && pos >= 2 && !tc5_wait(&s_free[pos & 1], (uint32_t)((pos >> 1) - 1) & 1u, abort)) ok = 0;
                if (ok) {
                    tc5_fence_after();
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        tc5_mma_f16(tmem + S::kTmemS + (pos & 1) * S::kTK,
                                    tc5_desc(qbuf + (ks >> 2) * S::kQBoxBytes + (ks & 3) * 32, 0u, 1024u),
                                    tc5_desc(kt + (ks >> 2) * S::kBoxBytes + (ks & 3) * 32, 0u, 1024u), kIdescS,
                                    ks > 0 ? 1u : 0u);
                    tc5_commit(&s_full[pos & 1]);
                    if (mt.flags & kMetaLast) tc5_commit(q_empty);
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) {
                dead = true;
                break;
            }
        }
        if (lane == 0) {
            if (dead) {
                *abort = 1u;
                raise_error(a.err_word, KVD_DEVERR_TIMEOUT);
            }
            tc5_commit(&mma_done[0]);  // this thread's MMAs complete before the tensor memory is freed
            mbar_wait_drain(&mma_done[0], 0u);
        }
        __syncwarp();
    } else if (warp == 6) {
        // ---- P . V warp: one thread issues O += P_j . V_j once P_j is written ----
        if (lane == 0) {
            constexpr uint32_t kIdescO = tc5_idesc<kBf16>(128, D, false, true);
            bool dead = false;
            for (int j = 0;; ++j) {
                const int st = j % S::kStages;
                // the tile's meta (the slot is released by this thread, so its
                // phase cannot run ahead)
                if (!tc5_wait(&full[st], (uint32_t)(j / S::kStages) & 1u, abort)) {
                    dead = true;
                    break;
                }
                const TileMeta mt = meta[st];
                if (mt.flags & kMetaEnd) break;
                if (!tc5_wait(&p_full[j & 1], (uint32_t)(j >> 1) & 1u, abort)) {
                    dead = true;
                    break;
                }
                tc5_fence_after();
                const uint32_t vt = ring + st * 2 * S::kTileBytes + S::kTileBytes;
                const uint32_t pt = tmem + S::kTmemP + (j & 1) * (S::kTK / 2);  // P_j in tensor memory
                const bool first = (mt.flags & kMetaFirst) != 0;
#pragma unroll
                for (int ks = 0; ks < S::kTK / 16; ++ks)
                    tc5_mma_f16_ts(tmem + S::kTmemO, pt + ks * 8,
                                   tc5_desc(vt + ks * 16 * 128, (uint32_t)S::kBoxBytes, 1024u), kIdescO,
                                   (ks > 0 || !first) ? 1u : 0u);
                tc5_commit(&p_empty[j & 1]);  // P buffer j & 1 and O are free / final
                tc5_commit(&empty[st]);       // the ring slot is free
            }
            if (dead) {
                *abort = 1u;
                raise_error(a.err_word, KVD_DEVERR_TIMEOUT);
            }
            tc5_commit(&mma_done[1]);
            mbar_wait_drain(&mma_done[1], 0u);
        }
        __syncwarp();
    } else {
        // ---- softmax warps 0-3: thread tid owns row tid of the block ----
        const int r = tid;
        const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
        float m_run = kNegInf, l_run = 0.f;
        int lim = 0;
        int pe_cnt[2] = {0, 0};   // completions of p_empty[b] waited for
        int n_split = 0;          // split pieces computed (ticket merge)
        bool dead = false;
        // Waits are decided per warp (the tensor-memory loads and stores
        // below are warp-collective): a wait fails for all lanes if it
        // failed for one.
        auto warp_wait = [&](uint64_t *bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, tc5_wait(bar, parity, abort));
        };
        // wait until the P . V of tile `target` (buffer b = target & 1) is complete
        auto pe_wait = [&](int b, int target) -> bool {
            while (pe_cnt[b] * 2 + b <= target) {
                if (!warp_wait(&p_empty[b], (uint32_t)pe_cnt[b] & 1u)) return false;
                ++pe_cnt[b];
            }
            return true;
        };
        for (int pos = 0;; ++pos) {
            const int st = pos % S::kStages;
            if (!warp_wait(&full[st], (uint32_t)(pos / S::kStages) & 1u)) {
                dead = true;
                break;
            }
            const TileMeta mt = meta[st];
            if (mt.flags & kMetaEnd) break;
            const bool first = (mt.flags & kMetaFirst) != 0;
            if (first) {
                lim = mt.P + 1 + ((mt.rb * S::kRB + r) % a.N);
                m_run = kNegInf;
                l_run = 0.f;
            }
            const int sb = pos & 1;
            if (!warp_wait(&s_full[sb], (uint32_t)(pos >> 1) & 1u)) {
                dead = true;
                break;
            }
            tc5_fence_after();
            uint32_t sr[S::kTK];
            tc5_ld64(lane_addr + S::kTmemS + sb * S::kTK, sr);
            tc5_fence_before();
            mbar_arrive(&s_free[sb]);

            // Raw scores; keys at or past the row's limit masked by selection
            // (their rows may hold stale NaN).  The row max is taken on the raw
            // scores (qscale > 0) and the scale folded into the exponent; max
            // and sum run as 8 independent chains (a row is one thread).
            const bool masked = mt.tile_k0 + S::kTK > mt.P + 1;
            if (masked) {
#pragma unroll
                for (int c = 0; c < S::kTK; ++c)
                    if (mt.tile_k0 + c >= lim) sr[c] = 0xff800000u;  // -inf
            }
            float mx8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mx8[i] = __uint_as_float(sr[i]);
#pragma unroll
            for (int c = 8; c < S::kTK; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], __uint_as_float(sr[c]));
            const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                   fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * a.qscale;
            float alpha = 1.f;
            bool rescale = false;
            if (mx > m_run + kRescaleThreshold) {
                if (!first) {
                    alpha = fast_exp2(m_run - mx);
                    rescale = true;
                }
                m_run = mx;
            }
            const float nmu = (m_run == kNegInf) ? 0.f : -m_run;
            float l8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) l8[i] = 0.f;
            uint32_t pk[S::kTK / 2];
#pragma unroll
            for (int c = 0; c < S::kTK / 2; ++c) {
                const float p0 = fast_exp2(fmaf(__uint_as_float(sr[2 * c]), a.qscale, nmu));
                const float p1 = fast_exp2(fmaf(__uint_as_float(sr[2 * c + 1]), a.qscale, nmu));
                l8[c & 7] += p0 + p1;
                pk[c] = pack_pair<T>(p0, p1);
            }
            const float lt = ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
            l_run = l_run * alpha + lt;

            const int pb = pos & 1;
            if (!pe_wait(pb, pos - 2)) {  // the P buffer's previous P . V
                dead = true;
                break;
            }
            if (__any_sync(0xffffffffu, rescale)) {  // O holds the piece's P . V up to tile pos - 1
                // (the whole warp: rows that keep their max scale by 1)
                if (!pe_wait((pos - 1) & 1, pos - 1)) {
                    dead = true;
                    break;
                }
                tc5_fence_after();
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    tc5_ld32(lane_addr + S::kTmemO + c0, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tc5_st32(lane_addr + S::kTmemO + c0, o);
                }
            }
            // row r of P into its tensor-memory lane (P buffer pb)
            tc5_st32(lane_addr + S::kTmemP + pb * (S::kTK / 2), pk);
            tc5_fence_before();
            mbar_arrive(&p_full[pb]);

            if (!(mt.flags & kMetaLast)) continue;
            // ---- end of a piece: O after this tile's P . V ----
            if (!pe_wait(pb, pos)) {
                dead = true;
                break;
            }
            tc5_fence_after();
            const bool single = (mt.n_chunks == 1);
            const int rg = mt.rb * S::kRB + r;
            const bool real = rg < a.rows;  // (every lane loads: the loads are warp-collective)
            {
                const float inv = 1.f / l_run;
                float *pr = nullptr;
                T *orow = static_cast<T *>(a.out) + ((size_t)mt.bh * a.rows + rg) * D;
                if (!single) {
                    const size_t pbase =
                        ((size_t)blockIdx.x * 2 + ((int)blockIdx.x == mt.c_first ? 1 : 0)) * part_rows<S::kRB>(a.rows);
                    pr = a.part + (pbase + r) * (D + 4);
                }
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    tc5_ld32(lane_addr + S::kTmemO + c0, o);
                    if (!real) continue;
                    if (single) {
#pragma unroll
                        for (int i = 0; i < 32; i += 8)
                            stg128(orow + c0 + i,
                                   make_uint4(pack_pair<T>(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv),
                                              pack_pair<T>(__uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv),
                                              pack_pair<T>(__uint_as_float(o[i + 4]) * inv, __uint_as_float(o[i + 5]) * inv),
                                              pack_pair<T>(__uint_as_float(o[i + 6]) * inv, __uint_as_float(o[i + 7]) * inv)));
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            *reinterpret_cast<uint4 *>(pr + c0 + i) = make_uint4(o[i], o[i + 1], o[i + 2], o[i + 3]);
                    }
                }
                if (real && !single) *reinterpret_cast<float2 *>(pr + D) = make_float2(m_run, l_run);
            }
            tc5_fence_before();  // (the next arrive on p_full orders these reads before O is overwritten)
            if constexpr (kTicketMerge) {
                if (!single) {
                    if (r == 0 && n_split < 2) jobs[n_split] = MergeJob{mt.bh, mt.rb, mt.c_first, mt.n_chunks};
                    ++n_split;
                }
            }
        }
        if (dead) {
            *abort = 1u;
            raise_error(a.err_word, KVD_DEVERR_TIMEOUT);
        }
        if constexpr (kTicketMerge) {
            // ---- count this CTA's split pieces; merge the heads they complete ----
            // (every softmax thread takes part, also after a timeout: a named
            // barrier cannot be left early)
            n_split = min(n_split, 2);
            named_barrier_sync(1, 128);  // every row's partial is written
            if (tid == 0 && n_split > 0) {
                int *tickets = static_cast<int *>(a.merge_state);
                int seen[2];
#pragma unroll
                for (int i = 0; i < 2; ++i)
                    if (i < n_split)
                        seen[i] = atomic_add_acq_rel_gpu(tickets + (size_t)jobs[i].bh * a.n_rowblocks + jobs[i].rb, 1);
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    if (i < n_split && seen[i] == jobs[i].n_chunks - 1)
                        tickets[(size_t)jobs[i].bh * a.n_rowblocks + jobs[i].rb] = 0;  // the next call starts from zero
                    else
                        jobs[i].n_chunks = 0;
                }
            }
            named_barrier_sync(1, 128);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const MergeJob job = jobs[i];
                if (i < n_split && job.n_chunks) tc5_merge_rows<T, D>(a, job, warp, lane);
            }
        }
    }

    tc5_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc5_fence_after();
        tc5_dealloc(tmem, S::kTmemCols);
    }
}

template <typename T, int D, bool kTicketMerge, bool kPaged> AttnVariant make_tc5_variant()
{
    using S = Tc5Shape<T, D>;
    AttnVariant v;
    v.fn = reinterpret_cast<const void *>(&attn_tc5_kernel<T, D, false, kTicketMerge, kPaged>);
    v.fused_fn = reinterpret_cast<const void *>(&attn_tc5_kernel<T, D, true, kTicketMerge, kPaged>);
    if constexpr (kTicketMerge) v.merge_fn = nullptr;
    else v.merge_fn = reinterpret_cast<const void *>(&attn_merge_kernel<T, D, S::kRB, false>);
    v.threads = S::kThreads;
    v.fixed_smem_bytes = S::kFixedBytes;
    v.tile_keys = S::kTK;
    v.rows_per_block = S::kRB;
    v.piece_units = S::kPieceUnits;
    v.tma = true;
    v.q_map = true;
    return v;
}

// The tcgen05 builds for one element type and merge mode: D = 64 or 128,
// contiguous or paged.
template <typename T, bool kTicketMerge> bool pick_tc5_variant(int D, bool paged, AttnVariant *v)
{
    switch (D) {
    case 64: *v = paged ? make_tc5_variant<T, 64, kTicketMerge, true>() : make_tc5_variant<T, 64, kTicketMerge, false>();
        return true;
    case 128:
        *v = paged ? make_tc5_variant<T, 128, kTicketMerge, true>() : make_tc5_variant<T, 128, kTicketMerge, false>();
        return true;
    default: return false;
    }
}

}  // namespace kvd
