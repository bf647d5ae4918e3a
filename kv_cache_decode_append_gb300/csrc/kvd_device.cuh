// kvd_device.cuh -- device helpers shared by the decode-step kernels (sm_103a).
//
// Inline PTX for the Blackwell bulk-copy (TMA) engine and shared-memory
// mbarriers, bf16 widening, and the bounded wait used by every pipeline.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the library calls no driver entry point directly)
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvd.h"

namespace kvd {

constexpr float kLog2e = 1.4426950408889634f;

// A pipeline wait gives up after this long (ns of %globaltimer), sets
// KVD_DEVERR_TIMEOUT and lets the kernel wind down.  A healthy wait ends in
// microseconds; the bound only exists so that no kernel can spin forever.
// (A test build, KVD_TIMEOUT_TEST, shortens it so that a test can make a
// pipeline wait run out.)  The waits of the wind-down itself -- for copies and
// MMAs still in flight before the CTA exits -- keep the long bound.
#ifdef KVD_TIMEOUT_TEST
constexpr uint64_t kWaitLimitNs = 2000000ull;
#else
constexpr uint64_t kWaitLimitNs = 2000000000ull;
#endif
constexpr uint64_t kDrainLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make the mbarrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n"
        "  .reg .pred p;\n"
        "  mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "  selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Non-blocking test of phase `parity` of `bar`.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n"
        "  .reg .pred p;\n"
        "  mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "  selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait until phase `parity` of `bar` has completed.  Bounded: returns false
// after kWaitLimitNs without completion.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0u && global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// The wind-down's wait for work still in flight: bounded by kDrainLimitNs.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t *bar, uint32_t parity)
{
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > kDrainLimitNs) return false;
    return true;
}

// Wait for phase `parity` of `bar`, giving up after kWaitLimitNs or when
// *abort_flag is set by another thread: 0 the phase completed, 1 this wait
// timed out, 2 another thread gave up.
__device__ __forceinline__ int mbar_wait_or_abort(uint64_t *bar, uint32_t parity, const volatile int *abort_flag)
{
    if (mbar_try_wait(bar, parity)) return 0;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return 0;
        if ((it & 63u) == 0u) {
            if (*abort_flag != 0) return 2;
            if (global_timer_ns() - t0 > kWaitLimitNs) return 1;
        }
    }
}

// Shared-memory int with release (store) / acquire (load) semantics at CTA
// scope: what the writer stored before is visible to the reader after.
__device__ __forceinline__ void st_release_cta(volatile int *p, int v)
{
    asm volatile("st.release.cta.shared.u32 [%0], %1;" ::"r"(smem_addr((const void *)p)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_cta(const volatile int *p)
{
    int v;
    asm volatile("ld.acquire.cta.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr((const void *)p)) : "memory");
    return v;
}

// 2^x with the hardware approximation (ex2.approx.ftz.f32, one MUFU op).
__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// L2 policy for data that is read exactly once (K/V streams).
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// One bulk (TMA) copy global -> shared of `bytes` (multiple of 16, both
// addresses 16-byte aligned), completing as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_load_g2s(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// 2-D tiled bulk (TMA) load of one box of a tensor map (a kernel parameter)
// at element coordinates (x, y) into shared memory, completing on bar.
__device__ __forceinline__ void tma_load_2d(void *dst, const void *tmap, int x, int y, uint64_t *bar,
                                            uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Generic-proxy writes to shared memory made visible to later bulk (async
// proxy) writes of the same bytes.
__device__ __forceinline__ void fence_proxy_async_shared()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Four 8x8 16-bit matrices from shared memory (row addresses from lanes
// 8m..8m+7 for matrix m); trans: each matrix transposed.
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void *p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_addr(p)));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], const void *p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_addr(p)));
}
// the same, from a shared-space address
__device__ __forceinline__ void ldmatrix_x4_addr(uint32_t (&r)[4], uint32_t a)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a));
}
__device__ __forceinline__ void ldmatrix_x4_trans_addr(uint32_t (&r)[4], uint32_t a)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a));
}
// The 8x8 matrix of 16-bit elements held in ldmatrix's fragment layout (lane
// (g, t): row g, columns 2t, 2t+1), transposed across the warp: the result
// is lane (g, t)'s pair of rows 2t, 2t+1 at column g.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x)
{
    uint32_t r;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
    return r;
}
// 16-byte store to a shared-space address
__device__ __forceinline__ void sts128(uint32_t a, const uint4 &v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// d = a(16x16, row) * b(16x8, col) + d on the tensor cores, fp32 accumulators;
// T selects bf16 or fp16 operands.
template <typename T> __device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4],
                                                               uint32_t b0, uint32_t b1);
template <> __device__ __forceinline__ void mma_16816<__nv_bfloat16>(float (&d)[4], const uint32_t (&a)[4],
                                                                     uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <> __device__ __forceinline__ void mma_16816<__half>(float (&d)[4], const uint32_t (&a)[4],
                                                              uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two fp32 values as one 16-bit pair of type T (lo in the low half), rounded
// to nearest even.
template <typename T> __device__ __forceinline__ uint32_t pack_pair(float lo, float hi);
template <> __device__ __forceinline__ uint32_t pack_pair<__nv_bfloat16>(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
template <> __device__ __forceinline__ uint32_t pack_pair<__half>(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint4 lds128(const void *p)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_addr(p)));
    return v;
}

__device__ __forceinline__ uint4 ldg128_nc(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void stg128(void *p, uint4 v)
{
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// Two fp32 values in one 64-bit register pair, for the packed fp32 pipe of
// sm_100-class GPUs: one f32x2 instruction performs two IEEE fp32 operations
// with the same rounding as two scalar ones.
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pack2(float lo, float hi)
{
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpack2(f32x2 v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c)
{
    f32x2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b)
{
    f32x2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Element type traits: how a 16-byte chunk widens to fp32.
template <typename T> struct Elem;

template <> struct Elem<float> {
    static constexpr int kBytes = 4;
    static constexpr int kPerChunk = 4;
    __device__ __forceinline__ static void widen(const uint4 &c, float *f)
    {
        f[0] = __uint_as_float(c.x);
        f[1] = __uint_as_float(c.y);
        f[2] = __uint_as_float(c.z);
        f[3] = __uint_as_float(c.w);
    }
    // the chunk as two fp32 pairs (elements 0,1 and 2,3)
    __device__ __forceinline__ static void widen2(const uint4 &c, f32x2 *f)
    {
        f[0] = pack2(__uint_as_float(c.x), __uint_as_float(c.y));
        f[1] = pack2(__uint_as_float(c.z), __uint_as_float(c.w));
    }
    __device__ __forceinline__ static void store(float *dst, float v) { *dst = v; }
};

template <> struct Elem<__nv_bfloat16> {
    static constexpr int kBytes = 2;
    static constexpr int kPerChunk = 8;
    // A bf16 is the upper half of an fp32: element 2k sits in the low half of
    // word k (little endian), element 2k+1 in the high half.
    __device__ __forceinline__ static void widen(const uint4 &c, float *f)
    {
        const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            f[2 * k] = __uint_as_float(w[k] << 16);
            f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        }
    }
    // the chunk as four fp32 pairs (elements 2k, 2k+1 of word k)
    __device__ __forceinline__ static void widen2(const uint4 &c, f32x2 *f)
    {
        const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
            f[k] = pack2(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xffff0000u));
    }
    __device__ __forceinline__ static void store(__nv_bfloat16 *dst, float v)
    {
        *dst = __float2bfloat16_rn(v);
    }
};

template <> struct Elem<__half> {
    static constexpr int kBytes = 2;
    static constexpr int kPerChunk = 8;
    // element 2k in the low half of word k, element 2k+1 in the high half
    __device__ __forceinline__ static float2 pair(uint32_t w)
    {
        __half2 h;
        memcpy(&h, &w, sizeof h);
        return __half22float2(h);
    }
    __device__ __forceinline__ static void widen(const uint4 &c, float *f)
    {
        const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 p = pair(w[k]);
            f[2 * k] = p.x;
            f[2 * k + 1] = p.y;
        }
    }
    __device__ __forceinline__ static void widen2(const uint4 &c, f32x2 *f)
    {
        const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 p = pair(w[k]);
            f[k] = pack2(p.x, p.y);
        }
    }
    __device__ __forceinline__ static void store(__half *dst, float v) { *dst = __float2half_rn(v); }
};

// E4M3 codes (8-bit floating point: 1 sign, 4 exponent, 3 fraction bits, no
// infinities, largest finite 448), 16 to a 16-byte chunk, widened exactly
// with the hardware conversion (two codes to an f16 pair, then to fp32).
template <> struct Elem<__nv_fp8_e4m3> {
    static constexpr int kBytes = 1;
    static constexpr int kPerChunk = 16;
    __device__ __forceinline__ static float2 pair(uint32_t two_codes)
    {
        uint32_t h2;
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((unsigned short)two_codes));
        __half2 h;
        memcpy(&h, &h2, sizeof h);
        return __half22float2(h);
    }
    // the chunk as eight fp32 pairs (codes 2k, 2k+1)
    __device__ __forceinline__ static void widen2(const uint4 &c, f32x2 *f)
    {
        const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 lo = pair(w[k] & 0xffffu), hi = pair(w[k] >> 16);
            f[2 * k] = pack2(lo.x, lo.y);
            f[2 * k + 1] = pack2(hi.x, hi.y);
        }
    }
};

// Two E4M3 codes (the low 16 bits) as an fp16 pair, exactly (every E4M3
// value is an fp16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes)
{
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((unsigned short)two_codes));
    return h2;
}

// Two fp32 values as two E4M3 codes, lo in the low byte: round to nearest
// even, magnitudes beyond 448 saturate to 448.
__device__ __forceinline__ uint32_t e4m3x2_from_f32(float lo, float hi)
{
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// One 16-code E4M3 chunk from the 16 elements of type T at src (16-byte
// aligned): each element x is stored as the code of the fp32 quotient
// x / scale (IEEE division).  Used by the E4M3 append and by the fused step,
// so both store the same bits.
template <typename T>
__device__ __forceinline__ uint4 e4m3_chunk_from(const unsigned char *src, float scale)
{
    constexpr int kIn = 16 / Elem<T>::kPerChunk;  // input chunks of T
    float x[16];
#pragma unroll
    for (int c = 0; c < kIn; ++c) Elem<T>::widen(ldg128_nc(src + c * 16), x + c * Elem<T>::kPerChunk);
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t lo = e4m3x2_from_f32(__fdiv_rn(x[4 * k], scale), __fdiv_rn(x[4 * k + 1], scale));
        const uint32_t hi = e4m3x2_from_f32(__fdiv_rn(x[4 * k + 2], scale), __fdiv_rn(x[4 * k + 3], scale));
        w[k] = lo | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Atomic add at GPU scope with acquire-release semantics; returns the old
// value.  Writes that precede it (this thread's, and those it has seen through
// a CTA barrier) are visible to a thread whose own acquire-release atomic on
// the same word reads this one's result, and so are that thread's later reads
// (and, after a CTA barrier, its CTA's).
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int *p, int v)
{
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// ---- thread-block clusters ----
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
// fp32 store into the shared memory of CTA `rank` of this cluster, at the
// offset that p has in this CTA's shared memory.
__device__ __forceinline__ void st_cluster_f32(void *p, uint32_t rank, float v)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(p)), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}
// Cluster barrier, all threads of the CTA: arrive, releasing this thread's
// earlier shared-memory writes (local and remote) ...
__device__ __forceinline__ void cluster_arrive_release()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
// ... and wait until every thread of the cluster that has not exited has
// arrived, acquiring their writes.
__device__ __forceinline__ void cluster_wait_acquire()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void raise_error(uint32_t *err_word, uint32_t bit)
{
    if (err_word != nullptr) atomicOr(err_word, bit);
}

__device__ __forceinline__ bool past_len_ok(int P, int N, int T_max, int max_past_len)
{
    return P >= 0 && P <= max_past_len && P + N <= T_max;
}

}  // namespace kvd
