// kvd_api.cu -- the C ABI (include/kvd.h): argument checks, the split-T plan,
// launches, and the in-place append kernel.
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include "kvd_attention.cuh"

namespace kvd {

// ---------------------------------------------------------------------------
// kv_append: cache[b, h, P_b + i, :] = new[b, h, i, :] for i < N, K and V.
// The cache is updated in place in its preallocated slots, as production
// engines do instead of concatenating ("7.1 自回归生成过程", section "Decode
// 阶段", the note under code 1-2).  One thread moves one 16-byte chunk of K and
// the matching chunk of V; consecutive threads cover consecutive chunks of a
// row, so loads and stores are fully coalesced 16-byte vector accesses.
struct AppendArgs {
    uint4 *k_cache;
    uint4 *v_cache;
    const uint4 *k_new;
    const uint4 *v_new;
    const int32_t *past_len;
    uint32_t *err_word;
    int H_kv, T_max, N, max_past_len;
    int row_chunks;   // 16-byte chunks per row
    long long total;  // B * H_kv * N * row_chunks
};

__global__ void __launch_bounds__(256) append_kernel(const AppendArgs a)
{
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < a.total;
         idx += stride) {
        const int c = (int)(idx % a.row_chunks);
        const long long row = idx / a.row_chunks;  // (bh, i)
        const int i = (int)(row % a.N);
        const long long bh = row / a.N;
        const int b = (int)(bh / a.H_kv);
        const int P = __ldg(a.past_len + b);
        if (!past_len_ok(P, a.N, a.T_max, a.max_past_len)) {
            if (c == 0 && i == 0 && bh % a.H_kv == 0) raise_error(a.err_word, KVD_DEVERR_PAST_LEN);
            continue;
        }
        const long long dst = (bh * a.T_max + P + i) * a.row_chunks + c;
        stg128(a.k_cache + dst, ldg128_nc(a.k_new + idx));
        stg128(a.v_cache + dst, ldg128_nc(a.v_new + idx));
    }
}

// ---------------------------------------------------------------------------
// Paged kv_append: token t = P_b + i of (b, h) goes to row t % page_size of head
// h in physical page block_table[b, t / page_size] of [num_pages, H_kv,
// page_size, D] pages (PagedAttention slot writes: "7.1 自回归生成过程", note
// under code 1-2).  Same thread mapping as append_kernel.
struct PagedAppendArgs {
    uint4 *k_pages;
    uint4 *v_pages;
    const uint4 *k_new;
    const uint4 *v_new;
    const int32_t *block_table;
    const int32_t *past_len;
    uint32_t *err_word;
    int H_kv, N, max_past_len;
    int page_shift, max_pages, num_pages;
    int row_chunks;
    long long total;
};

__global__ void __launch_bounds__(256) paged_append_kernel(const PagedAppendArgs a)
{
    const long long stride = (long long)gridDim.x * blockDim.x;
    const int capacity = a.max_pages << a.page_shift;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < a.total;
         idx += stride) {
        const int c = (int)(idx % a.row_chunks);
        const long long row = idx / a.row_chunks;  // (bh, i)
        const int i = (int)(row % a.N);
        const long long bh = row / a.N;
        const int b = (int)(bh / a.H_kv);
        const int h = (int)(bh % a.H_kv);
        const int P = __ldg(a.past_len + b);
        if (!past_len_ok(P, a.N, capacity, a.max_past_len)) {
            if (c == 0 && i == 0 && h == 0) raise_error(a.err_word, KVD_DEVERR_PAST_LEN);
            continue;
        }
        const int t = P + i;
        const int page = __ldg(a.block_table + (size_t)b * a.max_pages + (t >> a.page_shift));
        if (page < 0 || page >= a.num_pages) {
            if (c == 0) raise_error(a.err_word, KVD_DEVERR_PAGE);
            continue;
        }
        const long long slot = (((long long)page * a.H_kv + h) << a.page_shift) + (t & ((1 << a.page_shift) - 1));
        const long long dst = slot * a.row_chunks + c;
        stg128(a.k_pages + dst, ldg128_nc(a.k_new + idx));
        stg128(a.v_pages + dst, ldg128_nc(a.v_new + idx));
    }
}

// ---------------------------------------------------------------------------
// E4M3 kv_append: as append_kernel, with each new element x (type T) stored as
// the E4M3 code of x / scale (k_scale for K, v_scale for V).  One thread
// writes one 16-code chunk of K and of V (reading 16 elements of each).
struct AppendE4m3Args {
    uint4 *k_cache;
    uint4 *v_cache;
    const unsigned char *k_new;
    const unsigned char *v_new;
    const int32_t *past_len;
    uint32_t *err_word;
    int H_kv, T_max, N, max_past_len;
    int row_chunks;   // 16-code chunks per cache row (D / 16)
    float k_scale, v_scale;
    long long total;  // B * H_kv * N * row_chunks
};

template <typename T>
__global__ void __launch_bounds__(256) append_e4m3_kernel(const AppendE4m3Args a)
{
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < a.total;
         idx += stride) {
        const int c = (int)(idx % a.row_chunks);
        const long long row = idx / a.row_chunks;  // (bh, i)
        const int i = (int)(row % a.N);
        const long long bh = row / a.N;
        const int b = (int)(bh / a.H_kv);
        const int P = __ldg(a.past_len + b);
        if (!past_len_ok(P, a.N, a.T_max, a.max_past_len)) {
            if (c == 0 && i == 0 && bh % a.H_kv == 0) raise_error(a.err_word, KVD_DEVERR_PAST_LEN);
            continue;
        }
        const long long dst = (bh * a.T_max + P + i) * a.row_chunks + c;
        const size_t src = (size_t)idx * 16 * sizeof(T);  // 16 elements of T per chunk
        stg128(a.k_cache + dst, e4m3_chunk_from<T>(a.k_new + src, a.k_scale));
        stg128(a.v_cache + dst, e4m3_chunk_from<T>(a.v_new + src, a.v_scale));
    }
}

// ---------------------------------------------------------------------------
// Per-device facts, queried once.
namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxRows = 1024;  // (H_q / H_kv) * N supported per (b, h): 8 tcgen05 row blocks

std::mutex g_mu;
int g_sm_count[kMaxDevices];

struct OccEntry {
    int device;
    const void *fn;
    int smem;
    int ctas_per_sm;
};
OccEntry g_occ[256];
int g_occ_n = 0;

constexpr int kMaxSmemPerCta = 227 * 1024;
// Ranges longer than this many tile units per CTA use the separate merge pass.
constexpr int kLongRangeUnits = 32;
// The merge pass: at most this many four-warp CTAs per SM.
constexpr int kMergeCtasPerSm = 8;
// Query rows per KV head from which the tensor-core kernel (16-row blocks) is
// used, by head dim.  Measured on GB300 (bench.py, bf16): D=128 with 4 rows
// (the long-context workload) 106.4 us per layer against 113.6 on the CUDA
// cores, 8 rows 108.1 against 253.8, 16 rows 112.9 against 499.5; D=64 with 1
// row (GPT-2 batch 8) 14.6 against 10.3, so one-row decode stays on the CUDA
// cores and D=64 switches only where the CUDA-core kernel needs 8-row blocks.
constexpr int kMmaMinRows128 = 4;
constexpr int kMmaMinRows64 = 8;
// E4M3 caches (D = 128 only): widening the codes on the CUDA cores costs more
// than the saved bytes, so every row count goes to the tensor cores.
constexpr int kMmaMinRowsE4m3 = 1;
// Query rows per KV head from which bf16 / fp16 caches go to the tcgen05
// kernel (128-row blocks: every K/V tile read once for all rows), where the
// 16-row mma.sync blocks would read each tile once per block.
constexpr int kTc5MinRows = 17;
// Small layers (K/V bytes of one call, counted at max_past_len, at most
// kEarlyMaxBytes, a fifth of GB300's L2) run on the CUDA-core kernel with
// kArgEarly: the next kernel on the stream may launch as soon as this one
// starts, and kEarlyCtasPerSm CTAs per SM leave room for its CTAs.
#ifndef KVD_EARLY_CTAS_PER_SM
#define KVD_EARLY_CTAS_PER_SM 2
#endif
constexpr int kEarlyCtasPerSm = KVD_EARLY_CTAS_PER_SM;
#ifndef KVD_EARLY_MAX_BYTES
#define KVD_EARLY_MAX_BYTES (26LL << 20)
#endif
constexpr long long kEarlyMaxBytes = KVD_EARLY_MAX_BYTES;
// Small layers whose longest head needs at most kMaxCluster ring
// fills run in cluster mode: one thread-block cluster of C CTAs per
// sequence-head, C = tiles of the longest head / ring stages (rounded up), so
// that every CTA loads its whole share of the head at once (before the wait,
// with a stable history) and the pieces merge through distributed shared
// memory.  (8: the portable cluster size.)
#ifndef KVD_MAX_CLUSTER
#define KVD_MAX_CLUSTER 8
#endif
constexpr int kMaxCluster = KVD_MAX_CLUSTER;

// cuTensorMapEncodeTiled, looked up once through the runtime (no link to the
// driver library).
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
bool g_encode_looked_up = false;

kvd_status encode_fn(EncodeTiledFn *fn)
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode_looked_up) {
        g_encode_looked_up = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(p);
    }
    *fn = g_encode;
    return g_encode != nullptr ? KVD_OK : KVD_ERR_CUDA;
}

// A 2-D tensor map over a cache (or q) viewed as [rows, D] elements (16-bit,
// or 8-bit E4M3 codes), in boxes of box_rows rows x 128 bytes, 128-byte swizzle.
kvd_status encode_cache_map(CUtensorMap *map, const void *cache, long long rows, int D, kvd_dtype dtype,
                            int box_rows = 64)
{
    EncodeTiledFn fn;
    kvd_status st = encode_fn(&fn);
    if (st != KVD_OK) return st;
    const int es = dtype == KVD_E4M3 ? 1 : 2;
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D * es};
    const cuuint32_t box[2] = {(cuuint32_t)(128 / es), (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType ty = dtype == KVD_E4M3   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : dtype == KVD_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const CUresult r = fn(map, ty, 2,
                          const_cast<void *>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? KVD_OK : KVD_ERR_CUDA;
}

kvd_status current_device(int *dev)
{
    if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) return KVD_ERR_CUDA;
    return KVD_OK;
}

kvd_status sm_count(int dev, int *n)
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sm_count[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            return KVD_ERR_CUDA;
        g_sm_count[dev] = v;
    }
    *n = g_sm_count[dev];
    return KVD_OK;
}

// Resident CTAs per SM of `fn` with `smem` bytes of dynamic shared memory
// (the kernel is opted into the full 227 KB the first time it is seen).
kvd_status occupancy(int dev, const void *fn, int threads, int smem, int *ctas_per_sm)
{
    std::lock_guard<std::mutex> lk(g_mu);
    bool opted = false;
    for (int k = 0; k < g_occ_n; ++k) {
        if (g_occ[k].device == dev && g_occ[k].fn == fn) {
            opted = true;
            if (g_occ[k].smem == smem) {
                *ctas_per_sm = g_occ[k].ctas_per_sm;
                return KVD_OK;
            }
        }
    }
    if (!opted && cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kMaxSmemPerCta) != cudaSuccess)
        return KVD_ERR_CUDA;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, threads, smem) != cudaSuccess || occ <= 0)
        return KVD_ERR_CUDA;
    if (g_occ_n < 256) g_occ[g_occ_n++] = OccEntry{dev, fn, smem, occ};
    *ctas_per_sm = occ;
    return KVD_OK;
}

// Whether clusters of `c` CTAs of `fn` (threads, smem) can be resident at
// all (cudaOccupancyMaxActiveClusters > 0), cached per device.
struct ClusterEntry {
    int device;
    const void *fn;
    int smem, c;
    bool ok;
};
ClusterEntry g_cl[64];
int g_cl_n = 0;

kvd_status cluster_fits(int dev, const void *fn, int threads, int smem, int c, bool *ok)
{
    int dummy = 0;
    kvd_status st = occupancy(dev, fn, threads, smem, &dummy);  // (opts the kernel into large shared memory)
    if (st != KVD_OK) return st;
    std::lock_guard<std::mutex> lk(g_mu);
    for (int k = 0; k < g_cl_n; ++k) {
        if (g_cl[k].device == dev && g_cl[k].fn == fn && g_cl[k].smem == smem && g_cl[k].c == c) {
            *ok = g_cl[k].ok;
            return KVD_OK;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)c);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
    }
    if (g_cl_n < 64) g_cl[g_cl_n++] = ClusterEntry{dev, fn, smem, c, n > 0};
    *ok = n > 0;
    return KVD_OK;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

#ifdef KVD_TIMEOUT_TEST
int g_test_stall = 0;  // test builds: plant kArgTestStall in the next launches
#endif

int elem_bytes(kvd_dtype dt)
{
    switch (dt) {
    case KVD_F32: return 4;
    case KVD_BF16:
    case KVD_F16: return 2;
    case KVD_E4M3: return 1;
    default: return 0;
    }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The split-T plan of one decode_attention call.
struct Plan {
    AttnVariant v;
    int rows, rb, n_rowblocks;
    int grid, smem, launches, max_tiles;
    int sms;          // SMs of the device
    bool merge_pass;  // split heads merged by a second launch (else inside the kernel)
    bool mma;         // tensor-core kernel (16-row blocks, tiles by tensor map)
    bool tc5;         // tcgen05 kernel (128-row blocks, tiles and q by tensor map)
    bool early;       // small layer: kArgEarly, fewer CTAs per SM
    int cluster;      // > 0: cluster mode with this many CTAs per sequence-head
    size_t part_off, tickets_off, seg_off, ws_bytes;
};

kvd_status check_shapes(int B, int H_q, int H_kv, int D, int N, int max_past_len, kvd_dtype dtype)
{
    if (B < 0 || H_q < 1 || H_kv < 1 || N < 1 || max_past_len < 0) return KVD_ERR_INVALID_ARG;
    if (H_q % H_kv != 0) return KVD_ERR_INVALID_ARG;
    if (elem_bytes(dtype) == 0) return KVD_ERR_UNSUPPORTED;
    if (D != 64 && D != 128) return KVD_ERR_UNSUPPORTED;
    if ((long long)(H_q / H_kv) * N > kMaxRows) return KVD_ERR_UNSUPPORTED;
    return KVD_OK;
}

// The two builds of the kernels for one cache layout: with the separate
// merge pass (vp) and merging split heads themselves (vt); both have the same
// shared memory layout and tiles.
bool pick_builds(kvd_dtype dtype, int D, int rb, bool paged, AttnVariant *vp, AttnVariant *vt)
{
    switch (dtype) {
    case KVD_F32:
        return paged ? attn_variant_f32_paged(D, rb, vp) && attn_variant_f32_tk_paged(D, rb, vt)
                     : attn_variant_f32(D, rb, vp) && attn_variant_f32_tk(D, rb, vt);
    case KVD_BF16:
        return paged ? attn_variant_bf16_paged(D, rb, vp) && attn_variant_bf16_tk_paged(D, rb, vt)
                     : attn_variant_bf16(D, rb, vp) && attn_variant_bf16_tk(D, rb, vt);
    case KVD_F16:
        return paged ? attn_variant_f16_paged(D, rb, vp) && attn_variant_f16_tk_paged(D, rb, vt)
                     : attn_variant_f16(D, rb, vp) && attn_variant_f16_tk(D, rb, vt);
    case KVD_E4M3:  // bf16 q / out over an E4M3 cache, contiguous only
        return !paged && attn_variant_e4m3(D, rb, vp) && attn_variant_e4m3_tk(D, rb, vt);
    default:
        return false;
    }
}

// Lowest resident CTAs per SM over the attention and fused-step kernels of both builds.
kvd_status min_occupancy(int dev, const AttnVariant &vp, const AttnVariant &vt, int smem, int *occ)
{
    *occ = 1 << 30;
    for (const void *fn : {vp.fn, vp.fused_fn, vt.fn, vt.fused_fn}) {
        int o = 0;
        const kvd_status st = occupancy(dev, fn, vp.threads, smem, &o);
        if (st != KVD_OK) return st;
        if (o < *occ) *occ = o;
    }
    return KVD_OK;
}

kvd_status make_plan(int B, int H_q, int H_kv, int D, int N, int max_past_len, kvd_dtype dtype,
                     Plan *pl, bool paged = false)
{
    kvd_status st = check_shapes(B, H_q, H_kv, D, N, max_past_len, dtype);
    if (st != KVD_OK) return st;
    pl->rows = (H_q / H_kv) * N;
    // Many query rows per KV head (chunked decode with GQA): the tensor cores,
    // in blocks of 16 rows (mma.sync; E4M3 heads of at most 8 rows in the
    // swapped 8-row form) or, for 16-bit caches from kTc5MinRows rows, of 128
    // rows (tcgen05).  The choice does not depend on the cache layout, so
    // paged and contiguous calls give the same bits.
    const bool f16_family = dtype == KVD_BF16 || dtype == KVD_F16;
    pl->tc5 = f16_family && pl->rows >= kTc5MinRows;
    pl->mma = !pl->tc5 && ((pl->rows >= (D == 128 ? kMmaMinRows128 : kMmaMinRows64) && f16_family) ||
                           (dtype == KVD_E4M3 && D == 128 && pl->rows >= kMmaMinRowsE4m3));
    pl->rb = pl->tc5 ? 128 : pl->mma ? 16 : pl->rows <= 1 ? 1 : pl->rows <= 2 ? 2 : (pl->rows <= 4 || dtype == KVD_E4M3) ? 4 : 8;
    pl->n_rowblocks = (pl->rows + pl->rb - 1) / pl->rb;
    AttnVariant vp, vt, op, ot;  // this layout's builds, and the other layout's
    if (pl->tc5) {
        const auto builds = [&](bool pg, AttnVariant *p, AttnVariant *t) {
            return dtype == KVD_BF16 ? attn_variant_tc5_bf16(D, pg, p) && attn_variant_tc5_bf16_tk(D, pg, t)
                                     : attn_variant_tc5_f16(D, pg, p) && attn_variant_tc5_f16_tk(D, pg, t);
        };
        if (!builds(paged, &vp, &vt) || !builds(!paged, &op, &ot)) return KVD_ERR_UNSUPPORTED;
    } else if (pl->mma && dtype == KVD_E4M3) {
        if (!attn_variant_mma_e4m3(D, pl->rows, &vp) || !attn_variant_mma_e4m3_tk(D, pl->rows, &vt))
            return KVD_ERR_UNSUPPORTED;
        op = vp;
        ot = vt;
        pl->rb = vp.rows_per_block;  // (16, or 8 in the swapped form)
        pl->n_rowblocks = (pl->rows + pl->rb - 1) / pl->rb;
    } else if (pl->mma) {
        const auto builds = [&](bool pg, AttnVariant *p, AttnVariant *t) {
            return dtype == KVD_BF16 ? attn_variant_mma_bf16(D, pg, p) && attn_variant_mma_bf16_tk(D, pg, t)
                                     : attn_variant_mma_f16(D, pg, p) && attn_variant_mma_f16_tk(D, pg, t);
        };
        if (!builds(paged, &vp, &vt) || !builds(!paged, &op, &ot)) return KVD_ERR_UNSUPPORTED;
    } else {
        if (!pick_builds(dtype, D, pl->rb, paged, &vp, &vt)) return KVD_ERR_UNSUPPORTED;
        if (!pick_builds(dtype, D, pl->rb, !paged, &op, &ot)) {  // (no other layout: E4M3)
            op = vp;
            ot = vt;
        }
    }
    pl->v = vp;

    // Shared memory holds the ring plus two per-sequence tables (B + 1 tile
    // prefix sums, B history lengths).
    const size_t smem = (size_t)pl->v.fixed_smem_bytes + (((size_t)2 * B + 1) * 4 + 15) / 16 * 16;
    if (smem > (size_t)kMaxSmemPerCta) return KVD_ERR_UNSUPPORTED;
    pl->smem = (int)smem;

    int dev = 0, sms = 0, occ = 0, occ_other = 0;
    if ((st = current_device(&dev)) != KVD_OK) return st;
    if ((st = sm_count(dev, &sms)) != KVD_OK) return st;
    pl->sms = sms;
    // The attention and the fused-step kernels of both builds share the plan:
    // size the grid for the one with the lowest occupancy.  The workspace is
    // sized for the larger grid of the two cache layouts, so that one size
    // (kvd_decode_workspace_bytes) serves contiguous and paged calls.
    if ((st = min_occupancy(dev, vp, vt, pl->smem, &occ)) != KVD_OK) return st;
    if ((st = min_occupancy(dev, op, ot, pl->smem, &occ_other)) != KVD_OK) return st;

    // One CTA per resident slot; each takes an equal share of all tiles.
    // Small layers leave room on every SM for the calls that follow.
    const long long kv_bytes_hint =
        2LL * B * H_kv * ((long long)max_past_len + N) * D * elem_bytes(dtype);
    pl->early = !pl->mma && !pl->tc5 && kv_bytes_hint <= kEarlyMaxBytes;
    pl->grid = sms * (pl->early && occ > kEarlyCtasPerSm ? kEarlyCtasPerSm : occ);
    const long long t_hint = (long long)max_past_len + N;
    pl->max_tiles = (int)((t_hint + pl->v.tile_keys - 1) / pl->v.tile_keys);
    // Heads split across CTAs: merged inside the kernel by the CTA that
    // finishes a head last, unless the ranges are long (at most
    // kLongRangeUnits tile units per CTA, counted at max_past_len), where a
    // second, early-launched merge pass measured faster than the merge at the
    // tail of the last CTA.
    const long long units_hint =
        (long long)B * H_kv * pl->n_rowblocks * (pl->max_tiles + pl->v.piece_units);
    pl->merge_pass = !pl->early && units_hint > (long long)kLongRangeUnits * pl->grid;
    pl->launches = pl->merge_pass ? 2 : 1;
    if (!pl->merge_pass) pl->v = vt;
    pl->cluster = 0;
    if (pl->early && pl->v.cluster_fn != nullptr && pl->v.stages > 0) {
        const int c = (pl->max_tiles + pl->v.stages - 1) / pl->v.stages;
        const long long ctas = (long long)B * H_kv * pl->n_rowblocks * c;
        // (the pieces, c x RB rows of D + 2 floats, take the place of the tables)
        const size_t pieces = round_up((size_t)c * pl->rb * (D + 2) * sizeof(float), 16);
        const size_t smem_cl = (size_t)pl->v.fixed_smem_bytes +
                               (pieces > smem - pl->v.fixed_smem_bytes ? pieces : smem - pl->v.fixed_smem_bytes);
        bool fits = false;
        if (c >= 2 && c <= kMaxCluster && ctas <= 8LL * sms && smem_cl <= (size_t)kMaxSmemPerCta) {
            if ((st = cluster_fits(dev, pl->v.cluster_fn, pl->v.threads, (int)smem_cl, c, &fits)) != KVD_OK)
                return st;
            bool fits2 = false;
            if (fits &&
                (st = cluster_fits(dev, pl->v.cluster_fused_fn, pl->v.threads, (int)smem_cl, c, &fits2)) != KVD_OK)
                return st;
            fits = fits && fits2;
        }
        if (fits) {
            pl->cluster = c;
            pl->grid = (int)ctas;
            pl->smem = (int)smem_cl;
        }
    }

    // (partial slots of blocks of 16 or more rows -- the tensor-core kernels'
    // but the 8-row E4M3 form -- hold only a block's real rows: the kernels'
    // part_rows<RB>)
    const int part_rows = pl->rb >= 16 && pl->rows < pl->rb ? pl->rows : pl->rb;
    const size_t pieces = (size_t)sms * (occ > occ_other ? occ : occ_other) * 2 * part_rows;
    size_t off = 0;
    pl->part_off = off;  // per piece row: o[D], m, l, 2 floats of padding (16-byte rows)
    off += round_up(pieces * (D + 4) * sizeof(float), 256);
    pl->tickets_off = off;
    off += round_up((size_t)B * H_kv * pl->n_rowblocks * sizeof(int), 256);
    pl->seg_off = off;
    off += round_up((size_t)B * H_kv * pl->n_rowblocks * sizeof(int2), 256);
    pl->ws_bytes = off;
    return KVD_OK;
}

}  // namespace
}  // namespace kvd

using namespace kvd;

extern "C" {

kvd_status kvd_append(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                      const int32_t *past_len, int B, int H_kv, int T_max, int D, int N,
                      int max_past_len, kvd_dtype dtype, uint32_t *err_word, void *stream)
{
    const int s = elem_bytes(dtype);
    if (s == 0) return KVD_ERR_UNSUPPORTED;
    if (!k_cache || !v_cache || !k_new || !v_new || !past_len) return KVD_ERR_INVALID_ARG;
    if (B < 0 || H_kv < 1 || T_max < 1 || D < 1 || N < 1 || max_past_len < 0)
        return KVD_ERR_INVALID_ARG;
    if (((long long)D * s) % 16 != 0) return KVD_ERR_UNSUPPORTED;
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new))
        return KVD_ERR_INVALID_ARG;
    if ((long long)max_past_len + N > T_max) return KVD_ERR_CAPACITY;
    if (B == 0) return KVD_OK;

    int dev = 0, sms = 0;
    kvd_status st;
    if ((st = current_device(&dev)) != KVD_OK) return st;
    if ((st = sm_count(dev, &sms)) != KVD_OK) return st;

    AppendArgs a;
    a.k_cache = static_cast<uint4 *>(k_cache);
    a.v_cache = static_cast<uint4 *>(v_cache);
    a.k_new = static_cast<const uint4 *>(k_new);
    a.v_new = static_cast<const uint4 *>(v_new);
    a.past_len = past_len;
    a.err_word = err_word;
    a.H_kv = H_kv;
    a.T_max = T_max;
    a.N = N;
    a.max_past_len = max_past_len;
    a.row_chunks = (int)(((long long)D * s) / 16);
    a.total = (long long)B * H_kv * N * a.row_chunks;
    const int threads = 256;
    long long blocks = (a.total + threads - 1) / threads;
    if (blocks > 8LL * sms) blocks = 8LL * sms;
    void *args[] = {&a};
    return cudaLaunchKernel(reinterpret_cast<const void *>(&append_kernel), dim3((unsigned)blocks),
                            dim3(threads), args, 0, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? KVD_OK
               : KVD_ERR_CUDA;
}

size_t kvd_decode_workspace_bytes(int B, int H_q, int H_kv, int D, int N, int max_past_len,
                                  kvd_dtype dtype)
{
    Plan pl;
    if (make_plan(B, H_q, H_kv, D, N, max_past_len, dtype, &pl) != KVD_OK) return 0;
    return pl.ws_bytes;
}

kvd_status kvd_decode_plan(int B, int H_q, int H_kv, int D, int N, int max_past_len,
                           kvd_dtype dtype, kvd_plan_info *info)
{
    if (info == nullptr) return KVD_ERR_INVALID_ARG;
    Plan pl;
    const kvd_status st = make_plan(B, H_q, H_kv, D, N, max_past_len, dtype, &pl);
    if (st != KVD_OK) return st;
    info->tile_keys = pl.v.tile_keys;
    info->max_tiles = pl.max_tiles;
    info->grid = pl.grid;
    info->threads = pl.v.threads;
    info->smem_bytes = pl.smem;
    info->launches = pl.launches;
    info->workspace_bytes = pl.ws_bytes;
    info->rows_per_block = pl.rb;
    info->tensor_cores = pl.tc5 ? 2 : pl.mma ? 1 : 0;
    info->early_start = pl.early ? 1 : 0;
    info->cluster = pl.cluster;
    return KVD_OK;
}

}  // extern "C"

namespace {

// Attention (k_new == v_new == null) or the fused step (append inside).
// A paged cache: block table and pool geometry (null table = contiguous cache).
struct PagedCache {
    const int32_t *block_table;
    int page_size, max_pages, num_pages;
};

// Checks of the paged geometry; on success *T_max = max_pages * page_size.
kvd_status check_paged(const PagedCache &pc, int *T_max, int *page_shift)
{
    if (pc.block_table == nullptr || pc.max_pages < 1 || pc.num_pages < 1) return KVD_ERR_INVALID_ARG;
    if (pc.page_size < 64 || (pc.page_size & (pc.page_size - 1)) != 0 || pc.page_size > (1 << 24))
        return KVD_ERR_INVALID_ARG;
    const long long cap = (long long)pc.max_pages * pc.page_size;
    if (cap > 0x7fffffffLL) return KVD_ERR_INVALID_ARG;
    *T_max = (int)cap;
    int sh = 0;
    while ((1 << sh) < pc.page_size) ++sh;
    *page_shift = sh;
    return KVD_OK;
}

}  // namespace

// Host checks of a kvd_decode_attention call (contiguous cache, no E4M3) and
// the workspace it needs, without launching anything: the bytes, and the
// region [*zero_off, *zero_off + *zero_bytes) that must be zero when the
// kernel starts (the merge counters; every complete call leaves them zero).
// For the entry point whose workspace is built into the library.
namespace kvd {
kvd_status decode_attention_prepare(const void *q, const void *k_cache, const void *v_cache, const void *out,
                                    const int32_t *past_len, int B, int H_q, int H_kv, int T_max, int D, int N,
                                    int max_past_len, kvd_dtype dtype, size_t *ws_bytes, size_t *zero_off,
                                    size_t *zero_bytes)
{
    *ws_bytes = *zero_off = *zero_bytes = 0;
    if (!q || !k_cache || !v_cache || !out || !past_len) return KVD_ERR_INVALID_ARG;
    kvd_status st = check_shapes(B, H_q, H_kv, D, N, max_past_len, dtype);
    if (st != KVD_OK) return st;
    if (dtype == KVD_E4M3) return KVD_ERR_UNSUPPORTED;
    if (T_max < 1) return KVD_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return KVD_ERR_INVALID_ARG;
    if ((long long)max_past_len + N > T_max) return KVD_ERR_CAPACITY;
    if (B == 0) return KVD_OK;
    Plan pl;
    if ((st = make_plan(B, H_q, H_kv, D, N, max_past_len, dtype, &pl)) != KVD_OK) return st;
    *ws_bytes = pl.ws_bytes;
    *zero_off = pl.tickets_off;
    *zero_bytes = pl.seg_off - pl.tickets_off;
    return KVD_OK;
}
}  // namespace kvd

namespace {

kvd_status decode_launch(const void *q, const void *k_cache, const void *v_cache, const void *k_new,
                         const void *v_new, void *out, const int32_t *past_len, int B, int H_q, int H_kv,
                         int T_max, int D, int N, int max_past_len, float scale, kvd_dtype dtype,
                         void *workspace, size_t workspace_bytes, uint32_t *err_word, void *stream,
                         const PagedCache *paged = nullptr, const float *e4m3_scales = nullptr,
                         uint32_t step_flags = 0u)
{
    if (!q || !k_cache || !v_cache || !out || !past_len) return KVD_ERR_INVALID_ARG;
    kvd_status st = check_shapes(B, H_q, H_kv, D, N, max_past_len, dtype);
    if (st != KVD_OK) return st;
    // An E4M3 cache only through the _e4m3 entry points (which pass its scales).
    if ((dtype == KVD_E4M3) != (e4m3_scales != nullptr)) return KVD_ERR_UNSUPPORTED;
    if (e4m3_scales != nullptr &&
        !(e4m3_scales[0] > 0.f && e4m3_scales[0] < INFINITY && e4m3_scales[1] > 0.f && e4m3_scales[1] < INFINITY))
        return KVD_ERR_INVALID_ARG;
    int page_shift = 0;
    if (paged != nullptr && (st = check_paged(*paged, &T_max, &page_shift)) != KVD_OK) return st;
    if (T_max < 1) return KVD_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return KVD_ERR_INVALID_ARG;
    if ((long long)max_past_len + N > T_max) return KVD_ERR_CAPACITY;
    if (B == 0) return KVD_OK;

    Plan pl;
    if ((st = make_plan(B, H_q, H_kv, D, N, max_past_len, dtype, &pl, paged != nullptr)) != KVD_OK) return st;
    if (workspace == nullptr || workspace_bytes < pl.ws_bytes ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return KVD_ERR_WORKSPACE;

    char *ws = static_cast<char *>(workspace);
    AttnArgs a;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.out = out;
    a.past_len = past_len;
    a.k_new = k_new;
    a.v_new = v_new;
    a.part = reinterpret_cast<float *>(ws + pl.part_off);
    // Separate regions: the tickets must stay zero while the same workspace
    // serves calls in the other mode.
    a.merge_state = ws + (pl.merge_pass ? pl.seg_off : pl.tickets_off);
    if (e4m3_scales != nullptr)
        a.kv_scale = make_float2(e4m3_scales[0], e4m3_scales[1]);
    else
        a.block_table = paged != nullptr ? paged->block_table : nullptr;
    a.num_pages = paged != nullptr ? paged->num_pages : 0;
    a.page_shift = (short)page_shift;
    a.flags = pl.early ? kArgEarly : 0;
    // (a promise about the history only helps the fused step of a small
    // contiguous layer: its K/V tiles then load before the wait)
    if (pl.early && k_new != nullptr && paged == nullptr && (step_flags & KVD_STEP_HISTORY_STABLE))
        a.flags |= kArgHistoryStable;
#ifdef KVD_TIMEOUT_TEST
    if (g_test_stall) a.flags |= kArgTestStall;
#endif
    a.err_word = err_word;
    a.B = B;
    a.H_kv = H_kv;
    a.T_max = T_max;
    a.N = N;
    a.max_past_len = max_past_len;
    a.rows = pl.rows;
    a.n_rowblocks = pl.n_rowblocks;
    const float sc = (scale > 0.f) ? scale : 1.0f / sqrtf((float)D);
    // (E4M3: key = k_scale x stored code, folded into the q pre-scale)
    a.qscale = sc * kLog2e * (e4m3_scales != nullptr ? e4m3_scales[0] : 1.0f);

    // Both kernels are programmatic dependents of whatever precedes them on
    // the stream: they start early and wait (griddepcontrol.wait) before
    // touching any input, which hides their launch latency.
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = static_cast<cudaStream_t>(stream);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {&a};
    if (pl.cluster > 0) {  // one cluster of pl.cluster CTAs per sequence-head
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)pl.cluster;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
        cfg.gridDim = dim3((unsigned)pl.grid);
        cfg.blockDim = dim3(pl.v.threads);
        cfg.dynamicSmemBytes = (size_t)pl.smem;
        return cudaLaunchKernelExC(&cfg, k_new != nullptr ? pl.v.cluster_fused_fn : pl.v.cluster_fn, args) ==
                       cudaSuccess
                   ? KVD_OK
                   : KVD_ERR_CUDA;
    }

    cfg.gridDim = dim3((unsigned)pl.grid);
    cfg.blockDim = dim3(pl.v.threads);
    cfg.dynamicSmemBytes = (size_t)pl.smem;
    if (pl.v.tma) {
        // the K and V tensor maps, passed by value after the arguments (rows:
        // the contiguous cache's B*H_kv*T_max, or the pool's pages x heads x slots)
        const long long rows_total = paged != nullptr ? (long long)paged->num_pages * H_kv * paged->page_size
                                                      : (long long)B * H_kv * T_max;
        if (rows_total + 64 > 0x7fffffffLL) return KVD_ERR_UNSUPPORTED;  // 32-bit box coordinates
        alignas(64) CUtensorMap tmk, tmv;
        if ((st = encode_cache_map(&tmk, k_cache, rows_total, D, dtype)) != KVD_OK) return st;
        if ((st = encode_cache_map(&tmv, v_cache, rows_total, D, dtype)) != KVD_OK) return st;
        alignas(64) CUtensorMap tmq;
        void *targs[] = {&a, &tmk, &tmv, &tmq};
        if (pl.v.q_map) {  // q viewed as [B * H_q * N, D], 128-row boxes (one row block)
            const long long q_rows = (long long)B * H_kv * pl.rows;
            if (q_rows + pl.rb > 0x7fffffffLL) return KVD_ERR_UNSUPPORTED;
            if ((st = encode_cache_map(&tmq, q, q_rows, D, dtype, pl.rb)) != KVD_OK) return st;
        }
        if (cudaLaunchKernelExC(&cfg, k_new != nullptr ? pl.v.fused_fn : pl.v.fn, targs) != cudaSuccess)
            return KVD_ERR_CUDA;
    } else if (cudaLaunchKernelExC(&cfg, k_new != nullptr ? pl.v.fused_fn : pl.v.fn, args) != cudaSuccess) {
        return KVD_ERR_CUDA;
    }
    if (pl.merge_pass) {
        // four-warp CTAs striding over the real query rows, a warp per row
        // up to kMergeCtasPerSm CTAs per SM (then kMergeRows rows per warp at
        // a time), so that the whole grid is resident soon after the
        // attention kernel's CTAs leave (a warp per padded row slot, most of
        // them empty, cost several microseconds per layer)
        const long long rows_total = (long long)B * H_kv * pl.rows;
        const long long ctas = std::min<long long>((rows_total + 3) / 4, (long long)pl.sms * kMergeCtasPerSm);
        cfg.gridDim = dim3((unsigned)std::max<long long>(ctas, 1));
        cfg.blockDim = dim3(128);
        cfg.dynamicSmemBytes = 0;
        if (cudaLaunchKernelExC(&cfg, pl.v.merge_fn, args) != cudaSuccess) return KVD_ERR_CUDA;
    }
    return KVD_OK;
}

}  // namespace

extern "C" {

kvd_status kvd_decode_attention(const void *q, const void *k_cache, const void *v_cache,
                                void *out, const int32_t *past_len, int B, int H_q, int H_kv,
                                int T_max, int D, int N, int max_past_len, float scale,
                                kvd_dtype dtype, void *workspace, size_t workspace_bytes,
                                uint32_t *err_word, void *stream)
{
    return decode_launch(q, k_cache, v_cache, nullptr, nullptr, out, past_len, B, H_q, H_kv, T_max, D, N,
                         max_past_len, scale, dtype, workspace, workspace_bytes, err_word, stream);
}

kvd_status kvd_decode_step(const void *q, void *k_cache, void *v_cache, const void *k_new,
                           const void *v_new, void *out, const int32_t *past_len, int B, int H_q,
                           int H_kv, int T_max, int D, int N, int max_past_len, float scale,
                           kvd_dtype dtype, void *workspace, size_t workspace_bytes,
                           uint32_t *err_word, void *stream)
{
    if (!k_new || !v_new) return KVD_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new)) return KVD_ERR_INVALID_ARG;
    return decode_launch(q, k_cache, v_cache, k_new, v_new, out, past_len, B, H_q, H_kv, T_max, D, N,
                         max_past_len, scale, dtype, workspace, workspace_bytes, err_word, stream);
}

kvd_status kvd_decode_step_flags(const void *q, void *k_cache, void *v_cache, const void *k_new,
                                 const void *v_new, void *out, const int32_t *past_len, int B, int H_q,
                                 int H_kv, int T_max, int D, int N, int max_past_len, float scale,
                                 kvd_dtype dtype, uint32_t flags, void *workspace, size_t workspace_bytes,
                                 uint32_t *err_word, void *stream)
{
    if ((flags & ~(uint32_t)KVD_STEP_HISTORY_STABLE) != 0u) return KVD_ERR_INVALID_ARG;
    if (!k_new || !v_new) return KVD_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new)) return KVD_ERR_INVALID_ARG;
    return decode_launch(q, k_cache, v_cache, k_new, v_new, out, past_len, B, H_q, H_kv, T_max, D, N,
                         max_past_len, scale, dtype, workspace, workspace_bytes, err_word, stream, nullptr,
                         nullptr, flags);
}

kvd_status kvd_paged_append(void *k_pages, void *v_pages, const void *k_new, const void *v_new,
                            const int32_t *block_table, const int32_t *past_len, int B, int H_kv,
                            int D, int N, int page_size, int max_pages, int num_pages,
                            int max_past_len, kvd_dtype dtype, uint32_t *err_word, void *stream)
{
    const int s = elem_bytes(dtype);
    if (s == 0) return KVD_ERR_UNSUPPORTED;
    if (!k_pages || !v_pages || !k_new || !v_new || !past_len) return KVD_ERR_INVALID_ARG;
    if (B < 0 || H_kv < 1 || D < 1 || N < 1 || max_past_len < 0) return KVD_ERR_INVALID_ARG;
    int T_max = 0, page_shift = 0;
    kvd_status st = check_paged(PagedCache{block_table, page_size, max_pages, num_pages}, &T_max, &page_shift);
    if (st != KVD_OK) return st;
    if (((long long)D * s) % 16 != 0) return KVD_ERR_UNSUPPORTED;
    if (!aligned16(k_pages) || !aligned16(v_pages) || !aligned16(k_new) || !aligned16(v_new))
        return KVD_ERR_INVALID_ARG;
    if ((long long)max_past_len + N > T_max) return KVD_ERR_CAPACITY;
    if (B == 0) return KVD_OK;

    int dev = 0, sms = 0;
    if ((st = current_device(&dev)) != KVD_OK) return st;
    if ((st = sm_count(dev, &sms)) != KVD_OK) return st;

    PagedAppendArgs a;
    a.k_pages = static_cast<uint4 *>(k_pages);
    a.v_pages = static_cast<uint4 *>(v_pages);
    a.k_new = static_cast<const uint4 *>(k_new);
    a.v_new = static_cast<const uint4 *>(v_new);
    a.block_table = block_table;
    a.past_len = past_len;
    a.err_word = err_word;
    a.H_kv = H_kv;
    a.N = N;
    a.max_past_len = max_past_len;
    a.page_shift = page_shift;
    a.max_pages = max_pages;
    a.num_pages = num_pages;
    a.row_chunks = (int)(((long long)D * s) / 16);
    a.total = (long long)B * H_kv * N * a.row_chunks;
    const int threads = 256;
    long long blocks = (a.total + threads - 1) / threads;
    if (blocks > 8LL * sms) blocks = 8LL * sms;
    void *args[] = {&a};
    return cudaLaunchKernel(reinterpret_cast<const void *>(&paged_append_kernel), dim3((unsigned)blocks),
                            dim3(threads), args, 0, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? KVD_OK
               : KVD_ERR_CUDA;
}

kvd_status kvd_paged_decode_attention(const void *q, const void *k_pages, const void *v_pages,
                                      void *out, const int32_t *block_table,
                                      const int32_t *past_len, int B, int H_q, int H_kv, int D,
                                      int N, int page_size, int max_pages, int num_pages,
                                      int max_past_len, float scale, kvd_dtype dtype,
                                      void *workspace, size_t workspace_bytes, uint32_t *err_word,
                                      void *stream)
{
    const PagedCache pc{block_table, page_size, max_pages, num_pages};
    return decode_launch(q, k_pages, v_pages, nullptr, nullptr, out, past_len, B, H_q, H_kv, 0, D, N,
                         max_past_len, scale, dtype, workspace, workspace_bytes, err_word, stream, &pc);
}

kvd_status kvd_paged_decode_step(const void *q, void *k_pages, void *v_pages, const void *k_new,
                                 const void *v_new, void *out, const int32_t *block_table,
                                 const int32_t *past_len, int B, int H_q, int H_kv, int D, int N,
                                 int page_size, int max_pages, int num_pages, int max_past_len,
                                 float scale, kvd_dtype dtype, void *workspace,
                                 size_t workspace_bytes, uint32_t *err_word, void *stream)
{
    if (!k_new || !v_new) return KVD_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new)) return KVD_ERR_INVALID_ARG;
    const PagedCache pc{block_table, page_size, max_pages, num_pages};
    return decode_launch(q, k_pages, v_pages, k_new, v_new, out, past_len, B, H_q, H_kv, 0, D, N,
                         max_past_len, scale, dtype, workspace, workspace_bytes, err_word, stream, &pc);
}

kvd_status kvd_append_e4m3(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                           const int32_t *past_len, int B, int H_kv, int T_max, int D, int N,
                           int max_past_len, kvd_dtype new_dtype, float k_scale, float v_scale,
                           uint32_t *err_word, void *stream)
{
    if (new_dtype != KVD_F32 && new_dtype != KVD_BF16 && new_dtype != KVD_F16) return KVD_ERR_UNSUPPORTED;
    if (!k_cache || !v_cache || !k_new || !v_new || !past_len) return KVD_ERR_INVALID_ARG;
    if (B < 0 || H_kv < 1 || T_max < 1 || D < 1 || N < 1 || max_past_len < 0) return KVD_ERR_INVALID_ARG;
    if (!(k_scale > 0.f && k_scale < INFINITY && v_scale > 0.f && v_scale < INFINITY)) return KVD_ERR_INVALID_ARG;
    if (D % 16 != 0) return KVD_ERR_UNSUPPORTED;
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new))
        return KVD_ERR_INVALID_ARG;
    if ((long long)max_past_len + N > T_max) return KVD_ERR_CAPACITY;
    if (B == 0) return KVD_OK;

    int dev = 0, sms = 0;
    kvd_status st;
    if ((st = current_device(&dev)) != KVD_OK) return st;
    if ((st = sm_count(dev, &sms)) != KVD_OK) return st;

    AppendE4m3Args a;
    a.k_cache = static_cast<uint4 *>(k_cache);
    a.v_cache = static_cast<uint4 *>(v_cache);
    a.k_new = static_cast<const unsigned char *>(k_new);
    a.v_new = static_cast<const unsigned char *>(v_new);
    a.past_len = past_len;
    a.err_word = err_word;
    a.H_kv = H_kv;
    a.T_max = T_max;
    a.N = N;
    a.max_past_len = max_past_len;
    a.row_chunks = D / 16;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.total = (long long)B * H_kv * N * a.row_chunks;
    const int threads = 256;
    long long blocks = (a.total + threads - 1) / threads;
    if (blocks > 8LL * sms) blocks = 8LL * sms;
    const void *fn = new_dtype == KVD_F32    ? reinterpret_cast<const void *>(&append_e4m3_kernel<float>)
                     : new_dtype == KVD_BF16 ? reinterpret_cast<const void *>(&append_e4m3_kernel<__nv_bfloat16>)
                                             : reinterpret_cast<const void *>(&append_e4m3_kernel<__half>);
    void *args[] = {&a};
    return cudaLaunchKernel(fn, dim3((unsigned)blocks), dim3(threads), args, 0, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? KVD_OK
               : KVD_ERR_CUDA;
}

kvd_status kvd_decode_attention_e4m3(const void *q, const void *k_cache, const void *v_cache, void *out,
                                     const int32_t *past_len, int B, int H_q, int H_kv, int T_max, int D,
                                     int N, int max_past_len, float scale, float k_scale, float v_scale,
                                     void *workspace, size_t workspace_bytes, uint32_t *err_word,
                                     void *stream)
{
    const float scales[2] = {k_scale, v_scale};
    return decode_launch(q, k_cache, v_cache, nullptr, nullptr, out, past_len, B, H_q, H_kv, T_max, D, N,
                         max_past_len, scale, KVD_E4M3, workspace, workspace_bytes, err_word, stream, nullptr,
                         scales);
}

kvd_status kvd_decode_step_e4m3(const void *q, void *k_cache, void *v_cache, const void *k_new,
                                const void *v_new, void *out, const int32_t *past_len, int B, int H_q,
                                int H_kv, int T_max, int D, int N, int max_past_len, float scale,
                                float k_scale, float v_scale, void *workspace, size_t workspace_bytes,
                                uint32_t *err_word, void *stream)
{
    if (!k_new || !v_new) return KVD_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new)) return KVD_ERR_INVALID_ARG;
    const float scales[2] = {k_scale, v_scale};
    return decode_launch(q, k_cache, v_cache, k_new, v_new, out, past_len, B, H_q, H_kv, T_max, D, N,
                         max_past_len, scale, KVD_E4M3, workspace, workspace_bytes, err_word, stream, nullptr,
                         scales);
}

kvd_status kvd_workspace_init(void *workspace, size_t workspace_bytes, void *stream)
{
    if (workspace_bytes == 0) return KVD_OK;
    if (workspace == nullptr) return KVD_ERR_WORKSPACE;
    return cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? KVD_OK
               : KVD_ERR_CUDA;
}

size_t kvd_cache_bytes(int L, int B, int H_kv, int D, int T, kvd_dtype dtype)
{
    const int s = elem_bytes(dtype);
    if (s == 0 || L < 0 || B < 0 || H_kv < 0 || D < 0 || T < 0) return 0;
    return (size_t)2 * (size_t)L * (size_t)H_kv * (size_t)D * (size_t)T * (size_t)B * (size_t)s;
}

#ifdef KVD_TIMEOUT_TEST
// Test builds only (not part of include/kvd.h): make the next launches stall
// the first pipeline stage of every CTA so that the bounded waits run out.
void kvd_test_inject_stall(int on) { g_test_stall = on; }
#endif

// Staging layout of kvd_decode_step_host: q, k_new, v_new, past_len, out,
// each region 256-byte aligned.
size_t kvd_host_staging_bytes(int B, int H_q, int H_kv, int D, int N, kvd_dtype dtype)
{
    if (dtype == KVD_E4M3 || check_shapes(B, H_q, H_kv, D, N, 0, dtype) != KVD_OK) return 0;
    const size_t s = (size_t)elem_bytes(dtype);
    const size_t qb = (size_t)B * H_q * N * D * s, nb = (size_t)B * H_kv * N * D * s;
    return round_up(qb, 256) * 2 + round_up(nb, 256) * 2 + round_up((size_t)B * 4, 256);
}

size_t kvd_host_staging_inputs_bytes(int B, int H_q, int H_kv, int D, int N, kvd_dtype dtype)
{
    if (dtype == KVD_E4M3 || check_shapes(B, H_q, H_kv, D, N, 0, dtype) != KVD_OK) return 0;
    const size_t s = (size_t)elem_bytes(dtype);
    const size_t qb = (size_t)B * H_q * N * D * s, nb = (size_t)B * H_kv * N * D * s;
    return round_up(qb, 256) + round_up(nb, 256) * 2 + (size_t)B * 4;
}

namespace {
// Page-locked host memory (cudaHostAlloc / cudaHostRegister): a copy from or
// to it never blocks the host.
bool page_locked(const void *p)
{
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeHost;
}
}  // namespace

namespace {
// kvd_decode_step_host and _packed: `packed` (one host block in the staging
// layout's input part, at q_host) or the four inputs at their own addresses.
kvd_status host_step(const void *q_host, const void *k_new_host, const void *v_new_host, const int32_t *past_len_host,
                     bool packed, void *k_cache, void *v_cache, void *out_host, int B, int H_q, int H_kv, int T_max,
                     int D, int N, int max_past_len, float scale, kvd_dtype dtype, void *staging,
                     size_t staging_bytes, void *workspace, size_t workspace_bytes, uint32_t *err_word, void *stream)
{
    // Every check before anything is queued.
    if (!q_host || !k_new_host || !v_new_host || !out_host || !past_len_host || !k_cache || !v_cache)
        return KVD_ERR_INVALID_ARG;
    kvd_status st = check_shapes(B, H_q, H_kv, D, N, max_past_len, dtype);
    if (st != KVD_OK) return st;
    if (dtype == KVD_E4M3) return KVD_ERR_UNSUPPORTED;
    if (T_max < 1) return KVD_ERR_INVALID_ARG;
    if ((long long)max_past_len + N > T_max) return KVD_ERR_CAPACITY;
    if (B == 0) return KVD_OK;  // (nothing to copy or compute)
    const size_t need = kvd_host_staging_bytes(B, H_q, H_kv, D, N, dtype);
    if (staging == nullptr || (reinterpret_cast<uintptr_t>(staging) & 255u) != 0 || staging_bytes < need)
        return KVD_ERR_WORKSPACE;
    const size_t s = (size_t)elem_bytes(dtype);
    const size_t qb = (size_t)B * H_q * N * D * s, nb = (size_t)B * H_kv * N * D * s, pb = (size_t)B * 4;
    char *q_d = static_cast<char *>(staging);
    char *kn_d = q_d + round_up(qb, 256);
    char *vn_d = kn_d + round_up(nb, 256);
    int32_t *pl_d = reinterpret_cast<int32_t *>(vn_d + round_up(nb, 256));
    char *out_d = reinterpret_cast<char *>(pl_d) + round_up(pb, 256);
    const size_t in_bytes = (size_t)(reinterpret_cast<char *>(pl_d) - q_d) + pb;  // the inputs part
    size_t ws_need = 0, zero_off = 0, zero_bytes = 0;
    st = kvd::decode_attention_prepare(q_d, k_cache, v_cache, out_d, pl_d, B, H_q, H_kv, T_max, D, N,
                                       max_past_len, dtype, &ws_need, &zero_off, &zero_bytes);
    if (st != KVD_OK) return st;
    if (workspace == nullptr || workspace_bytes < ws_need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return KVD_ERR_WORKSPACE;
    if (!page_locked(q_host) || !page_locked(out_host) ||
        (packed ? !page_locked(static_cast<const char *>(q_host) + in_bytes - 1)
                : (!page_locked(k_new_host) || !page_locked(v_new_host) || !page_locked(past_len_host))))
        return KVD_ERR_INVALID_ARG;

    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (packed) {
        if (cudaMemcpyAsync(q_d, q_host, in_bytes, cudaMemcpyHostToDevice, cs) != cudaSuccess) return KVD_ERR_CUDA;
    } else if (cudaMemcpyAsync(q_d, q_host, qb, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
               cudaMemcpyAsync(kn_d, k_new_host, nb, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
               cudaMemcpyAsync(vn_d, v_new_host, nb, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
               cudaMemcpyAsync(pl_d, past_len_host, pb, cudaMemcpyHostToDevice, cs) != cudaSuccess) {
        return KVD_ERR_CUDA;
    }
    st = kvd_decode_step(q_d, k_cache, v_cache, kn_d, vn_d, out_d, pl_d, B, H_q, H_kv, T_max, D, N, max_past_len,
                         scale, dtype, workspace, workspace_bytes, err_word, stream);
    if (st != KVD_OK) return st;
    return cudaMemcpyAsync(out_host, out_d, qb, cudaMemcpyDeviceToHost, cs) == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}
}  // namespace

kvd_status kvd_decode_step_host(const void *q_host, void *k_cache, void *v_cache, const void *k_new_host,
                                const void *v_new_host, void *out_host, const int32_t *past_len_host, int B,
                                int H_q, int H_kv, int T_max, int D, int N, int max_past_len, float scale,
                                kvd_dtype dtype, void *staging, size_t staging_bytes, void *workspace,
                                size_t workspace_bytes, uint32_t *err_word, void *stream)
{
    return host_step(q_host, k_new_host, v_new_host, past_len_host, false, k_cache, v_cache, out_host, B, H_q, H_kv,
                     T_max, D, N, max_past_len, scale, dtype, staging, staging_bytes, workspace, workspace_bytes,
                     err_word, stream);
}

kvd_status kvd_decode_step_host_packed(const void *inputs_host, void *k_cache, void *v_cache, void *out_host, int B,
                                       int H_q, int H_kv, int T_max, int D, int N, int max_past_len, float scale,
                                       kvd_dtype dtype, void *staging, size_t staging_bytes, void *workspace,
                                       size_t workspace_bytes, uint32_t *err_word, void *stream)
{
    // (the inputs' own addresses inside the block only matter for the null
    // checks: the block is copied in one piece)
    const void *p = inputs_host;
    return host_step(p, p, p, static_cast<const int32_t *>(p), true, k_cache, v_cache, out_host, B, H_q, H_kv, T_max,
                     D, N, max_past_len, scale, dtype, staging, staging_bytes, workspace, workspace_bytes, err_word,
                     stream);
}

const char *kvd_status_string(kvd_status status)
{
    switch (status) {
    case KVD_OK: return "KVD_OK";
    case KVD_ERR_INVALID_ARG: return "KVD_ERR_INVALID_ARG";
    case KVD_ERR_CAPACITY: return "KVD_ERR_CAPACITY";
    case KVD_ERR_UNSUPPORTED: return "KVD_ERR_UNSUPPORTED";
    case KVD_ERR_WORKSPACE: return "KVD_ERR_WORKSPACE";
    case KVD_ERR_CUDA: return "KVD_ERR_CUDA";
    default: return "KVD_UNKNOWN_STATUS";
    }
}

}  // extern "C"
