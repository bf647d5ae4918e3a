// kvd_attention_mma.cuh -- split-T decode attention on the tensor cores.
//
// The same computation as attn_balanced_kernel (offset-causal GQA decode
// attention with a statically balanced split over T and a log-sum-exp merge;
// "7.1 自回归生成过程", code 1-2; "GPT-2缓存实测：千倍计算只快6倍", section
// "一个很容易漏掉的错误"), for blocks of 16 query rows: S = Q.K^T and O += P.V
// are dense contractions per tile, run as mma.sync m16n8k16 (bf16 or fp16
// operands, fp32 accumulators) instead of packed FMAs.  This serves chunked
// decode with many rows per KV head (g * N >= 16, where the CUDA-core kernel
// would need several row blocks and re-read K/V for each), and moves the
// per-element work of every decode off the CUDA cores.
//
// Differences from attn_balanced_kernel:
//   * tiles arrive by 2-D TMA through tensor maps over the cache viewed as
//     [B*H_kv*T_max, D] (or a page pool as [num_pages*H_kv*page_size, D]),
//     in boxes of 64 keys x 128 bytes with the 128-byte
//     swizzle, so that ldmatrix reads 8 keys at one column chunk without bank
//     conflicts (a plain row-major tile would serialize those reads 8 ways);
//   * a warp owns 16 keys of each 64-key tile and all 16 rows; its Q
//     fragments stay in registers for the piece, S lives in the MMA
//     accumulators, and the softmax weights P are repacked from the S
//     accumulators straight into the A fragments of the P.V MMA;
//   * scores are scaled after the MMA (Q stays exact in its 16-bit type); P
//     enters the MMA rounded to the operand type while the normaliser l sums
//     the fp32 weights;
//   * value rows past the end of a sequence are zeroed in shared memory
//     before they reach the MMA (a zero weight times a stale NaN would still
//     be NaN); in a fused step the new rows are written into the tile (and
//     the cache) before the tile is read;
//   * E4M3 caches widen their codes to fp16 fragments between ldmatrix and
//     the MMA; a KV head with at most 8 query rows runs in an 8-row form with
//     the operands swapped (mma_tile_e4m3_t), so that the MMA's 16-wide
//     dimension covers keys instead of mostly padding rows.
#pragma once

#include "kvd_attention.cuh"

namespace kvd {

// Compile-time shape of a tensor-core variant: 16 query rows, 64-key tiles,
// 4 warps of 16 keys.  Member names match AttnShape where RangeWalk and the
// epilogue use them.  RB = 8 (E4M3 caches only) is the swapped form of
// mma_tile_e4m3_t: blocks of at most 8 query rows, the rows as the MMA's
// 8-wide N dimension and keys / output columns as its 16-wide M dimension.
template <typename T, int D, typename C = T, int RB = 16> struct MmaShape {
    using Tq = Elem<T>;
    static constexpr bool k8 = sizeof(C) == 1;         // E4M3 cache (8-bit codes)
    static constexpr bool kT8 = RB == 8;               // swapped operands (mma_tile_e4m3_t)
    static constexpr bool kTma = true;
    static constexpr bool kQInRing = true;
    static constexpr int kRB = RB;
    static constexpr int kRowBytes = D * (int)sizeof(C);
    static constexpr int kQRowBytes = D * 2;
    static constexpr int kTK = 64;
    static constexpr int kNW = 4;
    static constexpr int kThreads = kNW * 32;
    static constexpr int kKpw = kTK / kNW;             // keys per warp per tile (16)
    static constexpr int kBoxCols = 128 / (int)sizeof(C);  // elements per 128-byte box row
    static constexpr int kBoxes = D / kBoxCols;
    static constexpr int kBoxBytes = kTK * 128;        // one box: 64 rows x 128 bytes
    static constexpr int kTileBytes = kBoxes * kBoxBytes;
    // E4M3: 3 stages, so that three CTAs (12 warps) share an SM; the
    // widening makes its tiles latency-bound with fewer warps.  The 8-row
    // form's 2 KB q slots leave room for a fourth stage at three CTAs per SM
    // (62.7 against 63.4 us per long-context layer).
    static constexpr int kStages = (D == 128 && !kT8) ? 3 : 4;
    // (the swapped form, at four CTAs per SM under 128 registers, spilled in
    // the fused step and was no faster than the 16-row form: three)
    static constexpr int kMinBlocks = k8 ? 3 : 1;     // CTAs per SM the registers must allow
    static constexpr int kQSlotBytes = kRB * kQRowBytes;
    static constexpr int kPieceUnits = 2;
    static constexpr int kKSteps = D / 16;             // k-steps of S = Q.K^T
    static constexpr int kNTiles = D / 8;              // 8-wide output column tiles of O
    static constexpr int kQRegs = kT8 ? 2 : 4;         // Q fragment registers per k-step (B or A operand)
    static constexpr int kOTiles = kT8 ? D / 16 : kNTiles;  // accumulator tiles of O (O^T when kT8)

    static constexpr int kRingOff = 0;                 // 1024-aligned boxes (swizzle pattern)
    static constexpr int kQOff = kRingOff + kStages * 2 * kTileBytes;
    // No separate epilogue area: a piece's last tile keeps its ring slot
    // until the warps are merged, and the merge uses that slot (o of 4 warps
    // x 16 rows x D fp32 = the K and V tile bytes of a 16-bit cache; m and l
    // in its q slot).  8-bit tiles hold half of that: the warps are merged in
    // two phases (warps 2, 3 folded into warps 0, 1 first).
    static constexpr int kMergePhases = (kNW * kRB * D * 4 <= 2 * kTileBytes) ? 1 : 2;
    static constexpr int kMergeWarps = kNW / kMergePhases;  // warps whose o is in the slot at once
    static constexpr int kMetaOff = kQOff + kStages * kQSlotBytes;
    static constexpr int kBarOff = kMetaOff + kStages * 32;
    static constexpr int kJobOff = kBarOff + 2 * kStages * 8;
    static constexpr int kPageOff = kJobOff + 32;
    static constexpr int kCtlOff = kPageOff + 16;    // AbortCtl words
    static constexpr int kFixedBytes = kCtlOff + 16;

    static_assert(D == 64 || D == 128, "head dim");
    static_assert(kBoxBytes % 1024 == 0 && kQOff % 1024 == 0, "swizzle atoms stay 1024-byte aligned");
    static_assert(2 * kNW * kRB * 4 <= kQSlotBytes, "m and l in the q slot");
    static_assert(kMergeWarps * kRB * D * 4 <= 2 * kTileBytes, "merge in the slot");
    static_assert(!k8 || D == 128, "E4M3 tiles: one 128-byte box per row");
    static_assert(RB == 16 || (kT8 && k8), "8-row blocks: the swapped E4M3 form only");
    static_assert(!kT8 || kMergePhases == 1, "8-row blocks merge in one phase");
};

// Shared-memory address of the 16-byte chunk c (0 .. D/8-1) of tile row r in
// a K or V tile of 128-byte-swizzled boxes starting at shared address tile.
// The 128-byte swizzle moves the 16-byte chunk of address bits [6:4] by
// bits [9:7] (XOR); applied to the actual address it holds for any
// 128-byte-aligned box.
template <typename S> __device__ __forceinline__ uint32_t mma_chunk_addr(uint32_t tile, int r, int c)
{
    const uint32_t lin = tile + (c >> 3) * S::kBoxBytes + r * 128 + ((c & 7) << 4);
    return lin ^ ((lin >> 3) & 0x70u);
}

// One tile for one warp: its 16 keys kb .. kb+15 of the tile, 16 rows.
//   qa     Q A-fragments per k-step (rows g, g+8; columns 16s + 2t, +8)
//   oacc   O accumulators per 8-column tile (C layout: rows g, g+8)
//   m, l   running max (log2 units) and this lane's share of the weight sum,
//          for rows g and g+8
// kMasked: per-key limits apply (lim: first key each row may not see), and
// value rows at or past k_end are zeroed first.
template <typename T, int D, bool kMasked>
__device__ __forceinline__ void mma_tile(unsigned char *Ks, unsigned char *Vs,
                                         const uint32_t (&qa)[MmaShape<T, D>::kKSteps][4],
                                         float (&oacc)[MmaShape<T, D>::kNTiles][4], float (&m)[2],
                                         float (&l)[2], int warp, int lane, int tile_k0,
                                         const int (&lim)[2], int k_end, float qscale)
{
    using S = MmaShape<T, D>;
    const float kNegInf = __int_as_float(0xff800000);
    constexpr float kRescaleThreshold = 8.0f;
    const int t = lane & 3;
    const int kb = warp * S::kKpw;
    const uint32_t k_base = smem_addr(Ks), v_base = smem_addr(Vs);

    // ---- S = Q . K^T for the warp's 16 keys (two 8-key column tiles) ----
    float sacc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
    {
        // ldmatrix.x4: matrices (keys kb.., chunk 2s), (kb.., 2s+1), (kb+8.., 2s), (kb+8.., 2s+1)
        // (all fragment loads first: the loads keep their order, the MMAs
        // then only wait for the first of them)
        const int key = kb + ((lane >> 4) << 3) + (lane & 7);
        const int csel = (lane >> 3) & 1;
        uint32_t b[S::kKSteps][4];
#pragma unroll
        for (int ks = 0; ks < S::kKSteps; ++ks) ldmatrix_x4_addr(b[ks], mma_chunk_addr<S>(k_base, key, 2 * ks + csel));
        // odd k-steps into a second set of accumulators: two dependency chains
        // of kKSteps / 2 MMAs instead of one of kKSteps
        float sodd[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) sodd[nt][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < S::kKSteps; ks += 2) {
            mma_16816<T>(sacc[0], qa[ks], b[ks][0], b[ks][1]);
            mma_16816<T>(sacc[1], qa[ks], b[ks][2], b[ks][3]);
            mma_16816<T>(sodd[0], qa[ks + 1], b[ks + 1][0], b[ks + 1][1]);
            mma_16816<T>(sodd[1], qa[ks + 1], b[ks + 1][2], b[ks + 1][3]);
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) sacc[nt][e] += sodd[nt][e];
    }

    // ---- scale, mask, online softmax (rows g: e = 0,1; g+8: e = 2,3) ----
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            sacc[nt][e] *= qscale;
            if constexpr (kMasked) {
                const int key = tile_k0 + kb + nt * 8 + 2 * t + (e & 1);
                if (key >= lim[e >> 1]) sacc[nt][e] = kNegInf;
            }
        }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        float mt = fmaxf(fmaxf(sacc[0][2 * r], sacc[0][2 * r + 1]), fmaxf(sacc[1][2 * r], sacc[1][2 * r + 1]));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
        if (mt > m[r] + kRescaleThreshold) {
            const float alpha = fast_exp2(m[r] - mt);
            l[r] *= alpha;
#pragma unroll
            for (int nt = 0; nt < S::kNTiles; ++nt) {
                oacc[nt][2 * r] *= alpha;
                oacc[nt][2 * r + 1] *= alpha;
            }
            m[r] = mt;
        }
        const float mu = (m[r] == kNegInf) ? 0.f : m[r];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 2 * r; e < 2 * r + 2; ++e) {
                const float p = fast_exp2(sacc[nt][e] - mu);
                l[r] += p;
                sacc[nt][e] = p;
            }
    }
    // P as the A fragments of P . V (the S accumulator layout is the A layout)
    const uint32_t pa[4] = {pack_pair<T>(sacc[0][0], sacc[0][1]), pack_pair<T>(sacc[0][2], sacc[0][3]),
                            pack_pair<T>(sacc[1][0], sacc[1][1]), pack_pair<T>(sacc[1][2], sacc[1][3])};

    // ---- value rows past the end of the sequence: zero (a NaN times 0 is NaN) ----
    if constexpr (kMasked) {
        if (tile_k0 + kb + S::kKpw > k_end) {
            for (int idx = lane; idx < S::kKpw * (D / 8); idx += 32) {
                const int r = kb + idx / (D / 8), c = idx % (D / 8);
                if (tile_k0 + r >= k_end) sts128(mma_chunk_addr<S>(v_base, r, c), make_uint4(0u, 0u, 0u, 0u));
            }
            fence_proxy_async_shared();  // before the slot is refilled by a bulk copy
            __syncwarp();
        }
    }

    // ---- O += P . V: ldmatrix.trans matrices (keys kb.., chunk c), (kb+8.., c), (kb.., c+1), (kb+8.., c+1) ----
    {
        const int key = kb + (((lane >> 3) & 1) << 3) + (lane & 7);
        const int csel = lane >> 4;
        uint32_t b[S::kNTiles / 2][4];
#pragma unroll
        for (int c = 0; c < S::kNTiles; c += 2) ldmatrix_x4_trans_addr(b[c / 2], mma_chunk_addr<S>(v_base, key, c + csel));
#pragma unroll
        for (int c = 0; c < S::kNTiles; c += 2) {
            mma_16816<T>(oacc[c], pa, b[c / 2][0], b[c / 2][1]);
            mma_16816<T>(oacc[c + 1], pa, b[c / 2][2], b[c / 2][3]);
        }
    }
}

// One tile for one warp over an E4M3 cache (D = 128, one 128-byte box per
// row).  The codes are widened to fp16 on the way into the fragments:
//   * K: ldmatrix.x4 of the 16-bit view gives lane (g, t) key g's codes
//     16c + 4t .. 4t+3 of chunk c; one cvt per code pair makes the two B
//     registers of k-step c.  That is a fixed permutation of the contraction
//     index within each 16-column step, applied to Q as well (qa holds, in
//     the slots of columns 2t, 2t+1, 2t+8, 2t+9, the q values of columns 4t,
//     4t+1, 4t+2, 4t+3), so S is unchanged.
//   * V: ldmatrix.x4.trans of the 16-bit view gives lane (g, t) the codes of
//     keys 2t, 2t+1 at columns 2g, 2g+1 of chunk c; byte permutes split them
//     into an even-column and an odd-column 8-wide tile (oacc[2c], oacc[2c+1])
//     whose column g is 16c + 2g and 16c + 2g + 1.
//   * sfac: per row, the score factor (scale * log2 e * k_scale, times the
//     power of two by which the row's q was brought into fp16 range).
// Value rows at or past k_end are zeroed first when kMasked.
template <int D, bool kMasked>
__device__ __forceinline__ void mma_tile_e4m3(unsigned char *Ks, unsigned char *Vs, const uint32_t (&qa)[D / 16][4],
                                              float (&oacc)[D / 8][4], float (&m)[2], float (&l)[2], int warp,
                                              int lane, int tile_k0, const int (&lim)[2], int k_end,
                                              const float (&sfac)[2])
{
    using S = MmaShape<__nv_bfloat16, D, __nv_fp8_e4m3>;
    const float kNegInf = __int_as_float(0xff800000);
    constexpr float kRescaleThreshold = 8.0f;
    const int t = lane & 3;
    const int kb = warp * S::kKpw;
    const uint32_t k_base = smem_addr(Ks), v_base = smem_addr(Vs);

    // ---- S = Q . K^T: matrices (keys kb.., chunk c), (kb+8.., c), (kb.., c+1), (kb+8.., c+1) ----
    float sacc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
    {
        const int key = kb + (((lane >> 3) & 1) << 3) + (lane & 7);
        const int csel = lane >> 4;
        uint32_t r[D / 32][4];
#pragma unroll
        for (int c = 0; c < D / 16; c += 2) ldmatrix_x4_addr(r[c / 2], mma_chunk_addr<S>(k_base, key, c + csel));
        float sodd[2][4];  // odd chunks: a second dependency chain (as in mma_tile)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) sodd[nt][e] = 0.f;
#pragma unroll
        for (int c = 0; c < D / 16; c += 2)
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // chunk c + h: registers 2h (keys kb..) and 2h+1 (kb+8..)
                const uint32_t k0 = r[c / 2][2 * h], k1 = r[c / 2][2 * h + 1];
                float (&acc)[2][4] = h ? sodd : sacc;
                mma_16816<__half>(acc[0], qa[c + h], e4m3x2_to_f16x2(k0 & 0xffffu), e4m3x2_to_f16x2(k0 >> 16));
                mma_16816<__half>(acc[1], qa[c + h], e4m3x2_to_f16x2(k1 & 0xffffu), e4m3x2_to_f16x2(k1 >> 16));
            }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) sacc[nt][e] += sodd[nt][e];
    }

    // ---- mask, online softmax (as mma_tile), the row's score factor folded
    //      into the exponent: the max is taken on the raw scores (sfac > 0, so
    //      the order is kept and max(s) sfac rounds as max(s sfac) does) and
    //      each weight is exp2(fma(s, sfac, -m)) -- one instruction less per
    //      score on this ALU-bound path ----
    if constexpr (kMasked) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = tile_k0 + kb + nt * 8 + 2 * t + (e & 1);
                if (key >= lim[e >> 1]) sacc[nt][e] = kNegInf;
            }
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        float mt = fmaxf(fmaxf(sacc[0][2 * rr], sacc[0][2 * rr + 1]), fmaxf(sacc[1][2 * rr], sacc[1][2 * rr + 1]));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
        mt *= sfac[rr];
        if (mt > m[rr] + kRescaleThreshold) {
            const float alpha = fast_exp2(m[rr] - mt);
            l[rr] *= alpha;
#pragma unroll
            for (int nt = 0; nt < D / 8; ++nt) {
                oacc[nt][2 * rr] *= alpha;
                oacc[nt][2 * rr + 1] *= alpha;
            }
            m[rr] = mt;
        }
        const float mu = (m[rr] == kNegInf) ? 0.f : m[rr];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 2 * rr; e < 2 * rr + 2; ++e) {
                const float p = fast_exp2(fmaf(sacc[nt][e], sfac[rr], -mu));
                l[rr] += p;
                sacc[nt][e] = p;
            }
    }
    const uint32_t pa[4] = {pack_pair<__half>(sacc[0][0], sacc[0][1]), pack_pair<__half>(sacc[0][2], sacc[0][3]),
                            pack_pair<__half>(sacc[1][0], sacc[1][1]), pack_pair<__half>(sacc[1][2], sacc[1][3])};

    if constexpr (kMasked) {
        if (tile_k0 + kb + S::kKpw > k_end) {
            for (int idx = lane; idx < S::kKpw * (D / 16); idx += 32) {
                const int rr = kb + idx / (D / 16), c = idx % (D / 16);
                if (tile_k0 + rr >= k_end) sts128(mma_chunk_addr<S>(v_base, rr, c), make_uint4(0u, 0u, 0u, 0u));
            }
            fence_proxy_async_shared();
            __syncwarp();
        }
    }

    // ---- O += P . V ----
    {
        const int key = kb + (((lane >> 3) & 1) << 3) + (lane & 7);
        const int csel = lane >> 4;
        uint32_t r[D / 32][4];
#pragma unroll
        for (int c = 0; c < D / 16; c += 2) ldmatrix_x4_trans_addr(r[c / 2], mma_chunk_addr<S>(v_base, key, c + csel));
#pragma unroll
        for (int c = 0; c < D / 16; c += 2)
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // chunk c + h
                const uint32_t v0 = r[c / 2][2 * h], v1 = r[c / 2][2 * h + 1];  // keys kb+2t.., kb+8+2t..
                // one permute per column parity: the low half holds keys kb+2t, +1,
                // the high half keys kb+8+2t, +1 (the two B registers)
                const uint32_t ev = __byte_perm(v0, v1, 0x6420), od = __byte_perm(v0, v1, 0x7531);
                mma_16816<__half>(oacc[2 * (c + h)], pa, e4m3x2_to_f16x2(ev & 0xffffu), e4m3x2_to_f16x2(ev >> 16));
                mma_16816<__half>(oacc[2 * (c + h) + 1], pa, e4m3x2_to_f16x2(od & 0xffffu), e4m3x2_to_f16x2(od >> 16));
            }
    }
}

// The same tile with at most 8 query rows per block (RB = 8), operands
// swapped: S^T = K . Q^T and O^T = V^T . P^T, so that the MMA's 16-wide M
// dimension runs over the warp's 16 keys (then over 16 output columns) and
// its 8-wide N dimension over the query rows.  The 16-row form computes 16
// rows of which 8 .. 15 would be padding; this one issues half the MMAs and
// holds half the scores, Q fragments and accumulators.  The widening is the
// same per code.
//   * K: ldmatrix.x4 of the 16-bit view gives lane (g, t) the codes
//     16c + 4t .. 4t+3 of keys kb+g and kb+8+g; the low pair widened is A's
//     columns 2t, 2t+1, the high pair its columns 2t+8, 2t+9 (rows g, g+8):
//     the contraction order of mma_tile_e4m3, which qb follows
//     (qb[c] = query row g's columns 16c + 4t, +1 | 4t+2, 4t+3).
//   * S^T's accumulators hold keys kb+g (e = 0, 1) and kb+8+g (e = 2, 3) of
//     query rows 2t + (e & 1); m, l, lim and sfac are per row 2t + j.
//   * P^T: each 8x8 half of S^T packed to fp16 is in ldmatrix's fragment
//     layout (row = key); movmatrix transposes it into B's layout (keys 2t,
//     2t+1 | 2t+8, 2t+9 at query row g).
//   * V: ldmatrix.x4.trans as in mma_tile_e4m3; the even-column permute
//     gives A's rows 0 .. 7 (output column 16c + 2g), the odd one its rows
//     8 .. 15 (column 16c + 2g + 1), so oacc[c][e] is query row 2t + (e & 1)
//     at output column 16c + 2g + (e >> 1).
template <int D, bool kMasked>
__device__ __forceinline__ void mma_tile_e4m3_t(unsigned char *Ks, unsigned char *Vs, const uint32_t (&qb)[D / 16][2],
                                                float (&oacc)[D / 16][4], float (&m)[2], float (&l)[2], int warp,
                                                int lane, int tile_k0, const int (&lim)[2], int k_end,
                                                const float (&sfac)[2])
{
    using S = MmaShape<__nv_bfloat16, D, __nv_fp8_e4m3, 8>;
    const float kNegInf = __int_as_float(0xff800000);
    constexpr float kRescaleThreshold = 8.0f;
    const int g = lane >> 2;
    const int kb = warp * S::kKpw;
    const uint32_t k_base = smem_addr(Ks), v_base = smem_addr(Vs);
    // ldmatrix.x4 matrices: (keys kb.., chunk c), (kb+8.., c), (kb.., c+1), (kb+8.., c+1)
    const int key = kb + (((lane >> 3) & 1) << 3) + (lane & 7);
    const int csel = lane >> 4;

    // ---- S^T = K . Q^T: even and odd chunks in two dependency chains ----
    float sacc[4] = {0.f, 0.f, 0.f, 0.f}, sodd[4] = {0.f, 0.f, 0.f, 0.f};
    {
        uint32_t r[D / 32][4];
#pragma unroll
        for (int c = 0; c < D / 16; c += 2) ldmatrix_x4_addr(r[c / 2], mma_chunk_addr<S>(k_base, key, c + csel));
#pragma unroll
        for (int c = 0; c < D / 16; c += 2)
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // chunk c + h: keys kb+g (register 2h), kb+8+g (2h+1)
                const uint32_t k0 = r[c / 2][2 * h], k1 = r[c / 2][2 * h + 1];
                const uint32_t ka[4] = {e4m3x2_to_f16x2(k0 & 0xffffu), e4m3x2_to_f16x2(k1 & 0xffffu),
                                        e4m3x2_to_f16x2(k0 >> 16), e4m3x2_to_f16x2(k1 >> 16)};
                mma_16816<__half>(h ? sodd : sacc, ka, qb[c + h][0], qb[c + h][1]);
            }
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[e] += sodd[e];
    }

    // ---- mask, online softmax per query row 2t + j (max over the keys of
    //      the 8 lanes g sharing t), the row's score factor in the exponent
    //      as in mma_tile_e4m3 ----
    if constexpr (kMasked) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (tile_k0 + kb + g + ((e >> 1) << 3) >= lim[e & 1]) sacc[e] = kNegInf;
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        float mt = fmaxf(sacc[j], sacc[j + 2]);
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 4));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 8));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
        mt *= sfac[j];
        if (mt > m[j] + kRescaleThreshold) {
            const float alpha = fast_exp2(m[j] - mt);
            l[j] *= alpha;
#pragma unroll
            for (int c = 0; c < D / 16; ++c) {
                oacc[c][j] *= alpha;
                oacc[c][j + 2] *= alpha;
            }
            m[j] = mt;
        }
        const float mu = (m[j] == kNegInf) ? 0.f : m[j];
#pragma unroll
        for (int e = j; e < 4; e += 2) {
            const float p = fast_exp2(fmaf(sacc[e], sfac[j], -mu));
            l[j] += p;
            sacc[e] = p;
        }
    }
    // P^T as the B fragments of O^T += V^T . P^T
    const uint32_t pb0 = movmatrix_trans(pack_pair<__half>(sacc[0], sacc[1]));
    const uint32_t pb1 = movmatrix_trans(pack_pair<__half>(sacc[2], sacc[3]));

    if constexpr (kMasked) {
        if (tile_k0 + kb + S::kKpw > k_end) {
            for (int idx = lane; idx < S::kKpw * (D / 16); idx += 32) {
                const int rr = kb + idx / (D / 16), c = idx % (D / 16);
                if (tile_k0 + rr >= k_end) sts128(mma_chunk_addr<S>(v_base, rr, c), make_uint4(0u, 0u, 0u, 0u));
            }
            fence_proxy_async_shared();
            __syncwarp();
        }
    }

    // ---- O^T += V^T . P^T ----
    {
        uint32_t r[D / 32][4];
#pragma unroll
        for (int c = 0; c < D / 16; c += 2) ldmatrix_x4_trans_addr(r[c / 2], mma_chunk_addr<S>(v_base, key, c + csel));
#pragma unroll
        for (int c = 0; c < D / 16; c += 2)
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // chunk c + h
                const uint32_t v0 = r[c / 2][2 * h], v1 = r[c / 2][2 * h + 1];  // keys kb+2t.., kb+8+2t..
                const uint32_t ev = __byte_perm(v0, v1, 0x6420), od = __byte_perm(v0, v1, 0x7531);
                const uint32_t va[4] = {e4m3x2_to_f16x2(ev & 0xffffu), e4m3x2_to_f16x2(od & 0xffffu),
                                        e4m3x2_to_f16x2(ev >> 16), e4m3x2_to_f16x2(od >> 16)};
                mma_16816<__half>(oacc[c + h], va, pb0, pb1);
            }
    }
}

// In a fused step the tile holding new keys P .. P+N-1 has stale cache rows:
// the warp copies its new rows from k_new / v_new into the tile (and, when
// kc / vc are given, into the cache: kc, vc address the cache row of the
// tile's first key) before the tile is read.
// With an E4M3 cache (C != T) the new rows are quantized as kvd_append_e4m3
// stores them (kv_scale: K and V scales).
template <typename T, int D, typename C = T>
__device__ __forceinline__ void mma_insert_new_rows(unsigned char *Ks, unsigned char *Vs, int warp, int lane,
                                                    int tile_k0, int P, int k_end, const unsigned char *kn,
                                                    const unsigned char *vn, unsigned char *kc, unsigned char *vc,
                                                    float2 kv_scale = float2{})
{
    using S = MmaShape<T, D, C>;
    const int kb = warp * S::kKpw;
    const int lo = max(kb, P - tile_k0), hi = min(kb + S::kKpw, k_end - tile_k0);
    if (lo >= hi) return;
    constexpr int kChunks = S::kRowBytes / 16;  // 16-byte chunks per cache row
    for (int idx = lane; idx < (hi - lo) * kChunks; idx += 32) {
        const int r = lo + idx / kChunks, c = idx % kChunks;
        const int key = tile_k0 + r;
        uint4 kv, vv;
        if constexpr (S::k8) {  // 16 new elements per chunk of codes
            const size_t nrow = (size_t)(key - P) * S::kQRowBytes + c * 32;
            kv = e4m3_chunk_from<T>(kn + nrow, kv_scale.x);
            vv = e4m3_chunk_from<T>(vn + nrow, kv_scale.y);
        } else {
            const size_t nrow = (size_t)(key - P) * S::kRowBytes + c * 16;
            kv = ldg128_nc(kn + nrow);
            vv = ldg128_nc(vn + nrow);
        }
        sts128(mma_chunk_addr<S>(smem_addr(Ks), r, c), kv);
        sts128(mma_chunk_addr<S>(smem_addr(Vs), r, c), vv);
        if (kc != nullptr) {
            stg128(kc + (size_t)r * S::kRowBytes + c * 16, kv);
            stg128(vc + (size_t)r * S::kRowBytes + c * 16, vv);
        }
    }
    fence_proxy_async_shared();  // before the slot is refilled by a bulk copy
    __syncwarp();
}

// The tensor-core kernel.  Same split, ring, epilogue and merges as
// attn_balanced_kernel; tiles by TMA through the K and V tensor maps (over
// the contiguous cache viewed as [B*H_kv*T_max, D], or over the page pool
// viewed as [num_pages*H_kv*page_size, D] when kPaged).
// C: the cache element type (T, or E4M3 codes with bf16 T: contiguous only).
// kRows: rows per block, 16, or 8 for the swapped E4M3 form (mma_tile_e4m3_t).
template <typename T, int D, bool kFused, bool kTicketMerge, bool kPaged, typename C = T, int kRows = 16>
__global__ void __launch_bounds__(MmaShape<T, D, C, kRows>::kThreads, MmaShape<T, D, C, kRows>::kMinBlocks)
    attn_mma_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v)
{
    using S = MmaShape<T, D, C, kRows>;
    using Tq = Elem<T>;
    constexpr bool k8 = S::k8;
    constexpr bool kT8 = S::kT8;
    static_assert(!(k8 && kPaged), "the E4M3 cache is contiguous only");
    constexpr int RB = S::kRB;
    const float kNegInf = __int_as_float(0xff800000);
    extern __shared__ __align__(1024) unsigned char smem_mma[];
    unsigned char *smem = smem_mma;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::kBarOff);
    uint64_t *empty = full + S::kStages;
    TileMeta *meta = reinterpret_cast<TileMeta *>(smem + S::kMetaOff);
    MergeJob *jobs = reinterpret_cast<MergeJob *>(smem + S::kJobOff);
    int *pre = reinterpret_cast<int *>(smem + S::kFixedBytes);
    int *pl = pre + a.B + 1;

    const int tid = threadIdx.x;
    const int warp = tid / 32, lane = tid % 32;
    const int g = lane >> 2, t = lane & 3;

    // The swizzled boxes need 1024-byte-aligned shared memory; the dynamic
    // shared memory of a CTA starts so aligned, which is checked rather than
    // assumed (every thread takes the same branch).
    if ((smem_addr(smem) & 1023u) != 0) {
        if (tid == 0) raise_error(a.err_word, KVD_DEVERR_INTERNAL);
        return;
    }

    const AbortCtl ctl{reinterpret_cast<volatile int *>(smem + S::kCtlOff)};
    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < S::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], S::kNW);
        }
        ctl.init();
        fence_mbar_init();
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __syncthreads();

    RangeWalk<S, !kTicketMerge, kPaged> walk;
    int issued = 0;
    if (warp == 0) {
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
            const int HR = a.H_kv * a.n_rowblocks;
            const long long n_total = (long long)pre[a.B] * HR;
            const long long G = min((long long)gridDim.x, n_total);
            const long long lo = blockIdx.x < G ? n_total * blockIdx.x / G : 0;
            const long long hi = blockIdx.x < G ? n_total * (blockIdx.x + 1) / G : 0;
            walk.tm_k = &tm_k;
            walk.tm_v = &tm_v;
            walk.start(a, pre, pl, lo, hi, n_total, G);
            for (; issued < S::kStages && !walk.ended; ++issued) walk.fill(a, pre, pl, smem, meta, full, issued);
            ctl.described(issued);
        }
    }

    uint32_t qa[S::kKSteps][S::kQRegs];
    float oacc[S::kOTiles][4];
    // per row: g, g+8 (16-row blocks) or 2t, 2t+1 (8-row blocks)
    float m_run[2], l_run[2];
    float sfac[2];  // E4M3: per-row score factor (see mma_tile_e4m3)
    int lim[2];
    bool gave_up = false;  // this warp no longer waits for data (AbortCtl)
    int first_unwaited = -1;
    int n_pieces = 0;

    for (int pos = 0;; ++pos) {
        const int s = pos % S::kStages;
        const uint32_t ph = (uint32_t)(pos / S::kStages) & 1u;
        if (!gave_up) {
            if (tid == 0) {
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
                    walk.fill(a, pre, pl, smem, meta, full, fs);
                    ++issued;
                }
            }
            const int r = mbar_wait_or_abort(&full[s], ph, ctl.flag());
            if (r == 1) {
                ctl.set_abort();
                raise_error(a.err_word, KVD_DEVERR_TIMEOUT);
            }
            gave_up = __any_sync(0xffffffffu, r != 0);  // (warp-uniform: the MMAs are warp-wide)
            if (gave_up && tid == 0) first_unwaited = pos;
        }
        if (gave_up) {
            if (tid == 0) ctl.final_count(issued);
            if (!ctl.describable(pos)) break;
        }
        const TileMeta mt = meta[s];
        if (mt.flags & kMetaEnd) break;
        unsigned char *Ks = smem + S::kRingOff + s * 2 * S::kTileBytes;
        unsigned char *Vs = Ks + S::kTileBytes;

        if (mt.flags & kMetaFirst) {
            // Q fragments of the 16 rows (rows past the block's rows are zero)
            const unsigned char *qs = smem + S::kQOff + s * S::kQSlotBytes;
            const int q_rows = min(RB, a.rows - mt.rb * RB);
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int rg = mt.rb * RB + (kT8 ? 2 * t + r : g + 8 * r);
                lim[r] = mt.P + 1 + (rg % a.N);
                m_run[r] = kNegInf;
                l_run[r] = 0.f;
            }
#pragma unroll
            for (int nt = 0; nt < S::kOTiles; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) oacc[nt][e] = 0.f;
            if constexpr (kT8) {
                // B fragments of Q^T: row g, columns 16c + 4t .. 4t+3 (the
                // permuted order of mma_tile_e4m3_t); the row's power-of-two
                // range factor as in the 16-row form, its score factor then
                // fetched by the lanes that hold the row's scores (t = row / 2)
                const int row = g;
                float qf[S::kKSteps][4];
                float amax = 0.f;
#pragma unroll
                for (int c = 0; c < S::kKSteps; ++c) {
                    uint2 raw = make_uint2(0u, 0u);
                    if (row < q_rows) raw = *reinterpret_cast<const uint2 *>(qs + row * S::kQRowBytes + (16 * c + 4 * t) * 2);
                    qf[c][0] = __uint_as_float(raw.x << 16);
                    qf[c][1] = __uint_as_float(raw.x & 0xffff0000u);
                    qf[c][2] = __uint_as_float(raw.y << 16);
                    qf[c][3] = __uint_as_float(raw.y & 0xffff0000u);
#pragma unroll
                    for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fabsf(qf[c][e]));
                }
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                const int ex = (int)((__float_as_uint(amax) >> 23) & 0xffu) - 127;
                const int shift = ex >= 15 ? ex - 14 : 0;
                const float down = __uint_as_float((uint32_t)(127 - shift) << 23);  // 2^-shift
                const float f = a.qscale * __uint_as_float((uint32_t)(127 + shift) << 23);
#pragma unroll
                for (int c = 0; c < S::kKSteps; ++c) {
                    qa[c][0] = pack_pair<__half>(qf[c][0] * down, qf[c][1] * down);
                    qa[c][1] = pack_pair<__half>(qf[c][2] * down, qf[c][3] * down);
                }
#pragma unroll
                for (int j = 0; j < 2; ++j) sfac[j] = __shfl_sync(0xffffffffu, f, (2 * t + j) * 4);
            } else if constexpr (k8) {
                // fp16 fragments with the permuted column order of mma_tile_e4m3
                // (slots 2t, 2t+1 | 2t+8, 2t+9 hold columns 4t, 4t+1 | 4t+2, 4t+3);
                // a row whose largest |q| reaches 2^15 is scaled by an exact power
                // of two into fp16 range, and the factor goes into its scores.
                float qf[2][S::kKSteps][4];
                float amax[2] = {0.f, 0.f};
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int row = g + 8 * r;
#pragma unroll
                    for (int ks = 0; ks < S::kKSteps; ++ks) {
                        uint2 raw = make_uint2(0u, 0u);
                        if (row < q_rows) raw = *reinterpret_cast<const uint2 *>(qs + row * S::kQRowBytes + (16 * ks + 4 * t) * 2);
                        qf[r][ks][0] = __uint_as_float(raw.x << 16);
                        qf[r][ks][1] = __uint_as_float(raw.x & 0xffff0000u);
                        qf[r][ks][2] = __uint_as_float(raw.y << 16);
                        qf[r][ks][3] = __uint_as_float(raw.y & 0xffff0000u);
#pragma unroll
                        for (int e = 0; e < 4; ++e) amax[r] = fmaxf(amax[r], fabsf(qf[r][ks][e]));
                    }
                    amax[r] = fmaxf(amax[r], __shfl_xor_sync(0xffffffffu, amax[r], 1));
                    amax[r] = fmaxf(amax[r], __shfl_xor_sync(0xffffffffu, amax[r], 2));
                    // exponent of amax minus 14, at least 0: amax / 2^shift < 2^15
                    const int ex = (int)((__float_as_uint(amax[r]) >> 23) & 0xffu) - 127;
                    const int shift = ex >= 15 ? ex - 14 : 0;
                    const float down = __uint_as_float((uint32_t)(127 - shift) << 23);  // 2^-shift
                    sfac[r] = a.qscale * __uint_as_float((uint32_t)(127 + shift) << 23);
#pragma unroll
                    for (int ks = 0; ks < S::kKSteps; ++ks)
#pragma unroll
                        for (int e = 0; e < 4; ++e) qf[r][ks][e] *= down;
                }
#pragma unroll
                for (int ks = 0; ks < S::kKSteps; ++ks) {
                    qa[ks][0] = pack_pair<__half>(qf[0][ks][0], qf[0][ks][1]);
                    qa[ks][1] = pack_pair<__half>(qf[1][ks][0], qf[1][ks][1]);
                    qa[ks][2] = pack_pair<__half>(qf[0][ks][2], qf[0][ks][3]);
                    qa[ks][3] = pack_pair<__half>(qf[1][ks][2], qf[1][ks][3]);
                }
            } else {
#pragma unroll
                for (int ks = 0; ks < S::kKSteps; ++ks)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int row = g + ((e & 1) << 3);
                        const int col = 16 * ks + 2 * t + ((e >> 1) << 3);
                        qa[ks][e] = row < q_rows ? *reinterpret_cast<const uint32_t *>(qs + row * S::kQRowBytes + col * 2)
                                                 : 0u;
                    }
            }
        }

        const int k_end = mt.tile_k0 + mt.nk;
        if (gave_up) {  // (computes nothing, writes nothing)
        } else if (mt.tile_k0 + S::kTK <= mt.P + (kFused ? 0 : 1)) {
            if constexpr (kT8)
                mma_tile_e4m3_t<D, false>(Ks, Vs, qa, oacc, m_run, l_run, warp, lane, mt.tile_k0, lim, k_end, sfac);
            else if constexpr (k8)
                mma_tile_e4m3<D, false>(Ks, Vs, qa, oacc, m_run, l_run, warp, lane, mt.tile_k0, lim, k_end, sfac);
            else
                mma_tile<T, D, false>(Ks, Vs, qa, oacc, m_run, l_run, warp, lane, mt.tile_k0, lim, k_end, a.qscale);
        } else {
            if constexpr (kFused) {
                const size_t nrow = (size_t)mt.bh * a.N * S::kQRowBytes;
                unsigned char *kc = nullptr, *vc = nullptr;
                size_t crow = 0;  // cache row of the tile's first key
                bool write = mt.rb == 0;  // one row block writes the new rows into the cache
                if constexpr (kPaged) {
                    const int page = reinterpret_cast<const int *>(smem + S::kPageOff)[s];
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
                float2 kvs = float2{};
                if constexpr (k8) kvs = a.kv_scale;
                mma_insert_new_rows<T, D, C>(Ks, Vs, warp, lane, mt.tile_k0, mt.P, k_end,
                                             static_cast<const unsigned char *>(a.k_new) + nrow,
                                             static_cast<const unsigned char *>(a.v_new) + nrow, kc, vc, kvs);
            }
            if constexpr (kT8)
                mma_tile_e4m3_t<D, true>(Ks, Vs, qa, oacc, m_run, l_run, warp, lane, mt.tile_k0, lim, k_end, sfac);
            else if constexpr (k8)
                mma_tile_e4m3<D, true>(Ks, Vs, qa, oacc, m_run, l_run, warp, lane, mt.tile_k0, lim, k_end, sfac);
            else
                mma_tile<T, D, true>(Ks, Vs, qa, oacc, m_run, l_run, warp, lane, mt.tile_k0, lim, k_end, a.qscale);
        }
        // (a piece's last tile keeps its slot for the merge below)
        if (!(mt.flags & kMetaLast)) {
            __syncwarp();
            if (lane == 0 && !gave_up) mbar_arrive(&empty[s]);
        }

        if (tid == 0 && !gave_up && !walk.ended && issued < pos + 1 + S::kStages) {
            const int fs = issued % S::kStages;
            const uint32_t fph = ((uint32_t)(issued / S::kStages) & 1u) ^ 1u;
            if (mbar_test_wait(&empty[fs], fph)) {
                walk.fill(a, pre, pl, smem, meta, full, fs);
                ++issued;
            }
        }

        if (!(mt.flags & kMetaLast)) continue;

        // ---- end of a piece: each warp's (o, m, l) to shared memory, then
        //      the warps merged by log-sum-exp (in the slot's K and V tile
        //      bytes; m and l in its q slot) ----
        float *ep_o = reinterpret_cast<float *>(Ks);
        float *ep_m = reinterpret_cast<float *>(smem + S::kQOff + s * S::kQSlotBytes);
        float *ep_l = ep_m + S::kNW * RB;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            if constexpr (kT8) {  // (a row's keys are spread over the 8 lanes g)
                l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 4);
                l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 8);
                l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 16);
            } else {
                l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
                l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
            }
        }
        // this warp's (o, m, l) as merge entry w; with fold, entry w is
        // instead read back and merged into the registers
        auto exchange = [&](int w, bool fold) {
            float wa[2], wb[2];
            if (fold) {
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int row = kT8 ? 2 * t + r : g + 8 * r;
                    const float mo = ep_m[w * RB + row];
                    const float M = fmaxf(m_run[r], mo);
                    wa[r] = safe_weight(m_run[r], M);
                    wb[r] = safe_weight(mo, M);
                    l_run[r] = l_run[r] * wa[r] + ep_l[w * RB + row] * wb[r];
                    m_run[r] = M;
                }
            }
            if constexpr (kT8) {
                // O^T tile c: lane (g, t) holds columns 16c + 2g, +1 of rows 2t, 2t+1
#pragma unroll
                for (int c = 0; c < D / 16; ++c)
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        float2 *p = reinterpret_cast<float2 *>(ep_o + (w * RB + 2 * t + r) * D + 16 * c + 2 * g);
                        if (fold) {
                            const float2 o = *p;
                            oacc[c][r] = oacc[c][r] * wa[r] + o.x * wb[r];
                            oacc[c][r + 2] = oacc[c][r + 2] * wa[r] + o.y * wb[r];
                        } else {
                            *p = make_float2(oacc[c][r], oacc[c][r + 2]);
                        }
                    }
            } else if constexpr (k8) {
                // even / odd column tiles of chunk c: lane (g, t) holds columns 16c + 4t .. 4t+3
#pragma unroll
                for (int c = 0; c < D / 16; ++c)
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        float4 *p = reinterpret_cast<float4 *>(ep_o + (w * RB + g + 8 * r) * D + 16 * c + 4 * t);
                        if (fold) {
                            const float4 o = *p;
                            oacc[2 * c][2 * r] = oacc[2 * c][2 * r] * wa[r] + o.x * wb[r];
                            oacc[2 * c + 1][2 * r] = oacc[2 * c + 1][2 * r] * wa[r] + o.y * wb[r];
                            oacc[2 * c][2 * r + 1] = oacc[2 * c][2 * r + 1] * wa[r] + o.z * wb[r];
                            oacc[2 * c + 1][2 * r + 1] = oacc[2 * c + 1][2 * r + 1] * wa[r] + o.w * wb[r];
                        } else {
                            *p = make_float4(oacc[2 * c][2 * r], oacc[2 * c + 1][2 * r], oacc[2 * c][2 * r + 1],
                                             oacc[2 * c + 1][2 * r + 1]);
                        }
                    }
            } else {
#pragma unroll
                for (int nt = 0; nt < S::kNTiles; ++nt)
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        float2 *p = reinterpret_cast<float2 *>(ep_o + (w * RB + g + 8 * r) * D + nt * 8 + 2 * t);
                        if (fold) {
                            const float2 o = *p;
                            oacc[nt][2 * r] = oacc[nt][2 * r] * wa[r] + o.x * wb[r];
                            oacc[nt][2 * r + 1] = oacc[nt][2 * r + 1] * wa[r] + o.y * wb[r];
                        } else {
                            *p = make_float2(oacc[nt][2 * r], oacc[nt][2 * r + 1]);
                        }
                    }
            }
            if (!fold && (kT8 ? g : t) == 0) {
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int row = kT8 ? 2 * t + r : g + 8 * r;
                    ep_m[w * RB + row] = m_run[r];
                    ep_l[w * RB + row] = l_run[r];
                }
            }
        };
        // (thread 0 may now block at a CTA barrier: what it has described must
        // be known to warps that gave up, so that they can reach it too)
        if (tid == 0) ctl.described(issued);
        __syncthreads();  // every warp is done with the slot's K, V and q (or the previous merge)
        if constexpr (S::kMergePhases == 2) {
            if (warp >= S::kMergeWarps) exchange(warp - S::kMergeWarps, false);
            __syncthreads();
            if (warp < S::kMergeWarps) exchange(warp, true);
            __syncthreads();  // the folded entries are read before they are overwritten
        }
        if (warp < S::kMergeWarps) exchange(warp, false);
        __syncthreads();
        const bool single = (mt.n_chunks == 1);
        const size_t pbase =
            ((size_t)blockIdx.x * 2 + ((int)blockIdx.x == mt.c_first ? 1 : 0)) * part_rows<RB>(a.rows);
        for (int idx = tid; idx < RB * D; idx += S::kThreads) {
            const int r = idx / D, d = idx % D;
            const int rg = mt.rb * RB + r;
            if (rg >= a.rows) continue;
            float M = kNegInf;
#pragma unroll
            for (int w = 0; w < S::kMergeWarps; ++w) M = fmaxf(M, ep_m[w * RB + r]);
            float num = 0.f, den = 0.f;
#pragma unroll
            for (int w = 0; w < S::kMergeWarps; ++w) {
                const float wt = safe_weight(ep_m[w * RB + r], M);
                num = fmaf(wt, ep_o[(w * RB + r) * D + d], num);
                den = fmaf(wt, ep_l[w * RB + r], den);
            }
            if (single) {
                if constexpr (k8)  // values are stored / v_scale
                    Tq::store(static_cast<T *>(a.out) + ((size_t)mt.bh * a.rows + rg) * D + d, num / den * a.kv_scale.y);
                else
                    Tq::store(static_cast<T *>(a.out) + ((size_t)mt.bh * a.rows + rg) * D + d, num / den);
            } else {
                float *pr = a.part + (pbase + r) * (D + 4);
                pr[d] = num;
                if (d == 0) {
                    pr[D] = M;
                    pr[D + 1] = den;
                }
            }
        }
        // the slot is free again (its generic writes ordered before the next bulk copy)
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0 && !gave_up) mbar_arrive(&empty[s]);
        if constexpr (kTicketMerge) {
            if (!single) {
                if (tid == 0 && n_pieces < 2) jobs[n_pieces] = MergeJob{mt.bh, mt.rb, mt.c_first, mt.n_chunks};
                ++n_pieces;
            }
        }
    }

    if (tid == 0) {  // (as above: the barriers below need every thread)
        ctl.described(issued);
        ctl.final_count(issued);
    }
    if constexpr (kTicketMerge) {
        n_pieces = min(n_pieces, 2);
        __syncthreads();
        if (tid == 0 && n_pieces > 0) {
            int *tickets = static_cast<int *>(a.merge_state);
            int seen[2];
#pragma unroll
            for (int i = 0; i < 2; ++i)
                if (i < n_pieces) seen[i] = atomic_add_acq_rel_gpu(tickets + (size_t)jobs[i].bh * a.n_rowblocks + jobs[i].rb, 1);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                if (i < n_pieces && seen[i] == jobs[i].n_chunks - 1)
                    tickets[(size_t)jobs[i].bh * a.n_rowblocks + jobs[i].rb] = 0;
                else
                    jobs[i].n_chunks = 0;
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const MergeJob job = jobs[i];
            if (i < n_pieces && job.n_chunks)
                merge_pieces<T, D, RB, S::kThreads, k8>(a, job, nullptr, tid);  // (16-row heads: no scratch)
        }
    }

    if (tid == 0 && gave_up && first_unwaited >= 0) {
        const uint64_t t0 = global_timer_ns();
        for (int p = first_unwaited; p < issued; ++p) {
            const uint32_t ph2 = (uint32_t)(p / S::kStages) & 1u;
            while (!mbar_try_wait(&full[p % S::kStages], ph2) && global_timer_ns() - t0 < kDrainLimitNs) {
            }
        }
    }
    // Let the next kernel on the stream launch only now: launched at the
    // start, the dependents' CTAs took SM slots this kernel's statically
    // balanced grid still needed (E4M3 long-context layer 74 -> 113 us).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename T, int D, bool kTicketMerge, bool kPaged, typename C = T, int kRows = 16>
AttnVariant make_mma_variant()
{
    using S = MmaShape<T, D, C, kRows>;
    AttnVariant v;
    v.fn = reinterpret_cast<const void *>(&attn_mma_kernel<T, D, false, kTicketMerge, kPaged, C, kRows>);
    v.fused_fn = reinterpret_cast<const void *>(&attn_mma_kernel<T, D, true, kTicketMerge, kPaged, C, kRows>);
    if constexpr (kTicketMerge) v.merge_fn = nullptr;
    else v.merge_fn = reinterpret_cast<const void *>(&attn_merge_kernel<T, D, S::kRB, S::k8>);
    v.threads = S::kThreads;
    v.fixed_smem_bytes = S::kFixedBytes;
    v.tile_keys = S::kTK;
    v.rows_per_block = S::kRB;
    v.piece_units = S::kPieceUnits;
    v.tma = true;
    return v;
}

// bf16 q / out over an E4M3 cache: D = 128, contiguous; heads of at most 8
// query rows in the swapped 8-row form.
template <bool kTicketMerge> bool pick_mma_e4m3_variant(int D, int rows, AttnVariant *v)
{
    if (D != 128) return false;
    *v = rows <= 8 ? make_mma_variant<__nv_bfloat16, 128, kTicketMerge, false, __nv_fp8_e4m3, 8>()
                   : make_mma_variant<__nv_bfloat16, 128, kTicketMerge, false, __nv_fp8_e4m3, 16>();
    return true;
}

template <typename T, bool kTicketMerge> bool pick_mma_variant(int D, bool paged, AttnVariant *v)
{
    switch (D) {
    case 64: *v = paged ? make_mma_variant<T, 64, kTicketMerge, true>() : make_mma_variant<T, 64, kTicketMerge, false>();
        return true;
    case 128:
        *v = paged ? make_mma_variant<T, 128, kTicketMerge, true>() : make_mma_variant<T, 128, kTicketMerge, false>();
        return true;
    default: return false;
    }
}

}  // namespace kvd
