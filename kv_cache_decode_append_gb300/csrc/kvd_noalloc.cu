// kvd_noalloc.cu -- decode attention whose scratch memory is built into the
// library, for callers that must not allocate device memory.
//
// Some callers cannot allocate device memory where they call us: a plugin
// running inside a host engine that owns every device buffer through its own
// pool and hands extensions no allocator; or a latency-critical serving loop
// where cudaMalloc could block on the device or fail with out-of-memory in the
// middle of a run.  kvd_decode_attention_noalloc serves them: its scratch is a
// fixed array compiled into this file instead of a caller-provided workspace.
//
// Costs and rules of the built-in scratch:
//   * every device that loads the library holds kNoAllocScratchBytes (4 MiB)
//     of device memory for it until the process exits;
//   * all calls on a device share that one array: calls whose GPU work can
//     overlap (different streams without ordering between them) race on it;
//   * the array keeps whatever the previous call left in it; the part of it
//     that must start at zero (the counters the kernel uses to merge heads
//     split across CTAs, a few bytes per sequence-head) is cleared with
//     cudaMemsetAsync before each launch, once the host checks have passed;
//     the rest (partial results) is always written before it is read;
//   * shapes needing more than kNoAllocScratchBytes are rejected with
//     KVD_ERR_WORKSPACE, and invalid arguments with their status, before
//     anything is queued on the stream;
//   * the scratch's device address is looked up once per device and kept:
//     the entry point must not be used on a device after cudaDeviceReset.
#include <mutex>

#include <cuda_runtime.h>

#include "kvd.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;
constexpr int kNoAllocMaxDevices = 64;

// The scratch itself.  Host code must not use this name as an address: on the
// host it is only a stand-in; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void *g_noalloc_dev_ptr[kNoAllocMaxDevices];  // device address of g_noalloc_scratch, per device

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and remembered.
kvd_status noalloc_scratch(void **ptr)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return KVD_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_dev_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return KVD_ERR_CUDA;
        g_noalloc_dev_ptr[dev] = p;
    }
    *ptr = g_noalloc_dev_ptr[dev];
    return KVD_OK;
}

}  // namespace

namespace kvd {
kvd_status decode_attention_prepare(const void *q, const void *k_cache, const void *v_cache, const void *out,
                                    const int32_t *past_len, int B, int H_q, int H_kv, int T_max, int D, int N,
                                    int max_past_len, kvd_dtype dtype, size_t *ws_bytes, size_t *zero_off,
                                    size_t *zero_bytes);
}

extern "C" kvd_status kvd_decode_attention_noalloc(const void *q, const void *k_cache,
                                                   const void *v_cache, void *out,
                                                   const int32_t *past_len, int B, int H_q,
                                                   int H_kv, int T_max, int D, int N,
                                                   int max_past_len, float scale, kvd_dtype dtype,
                                                   uint32_t *err_word, void *stream)
{
    // Every host check first: an invalid call returns without queuing anything.
    size_t need = 0, zero_off = 0, zero_bytes = 0;
    kvd_status st = kvd::decode_attention_prepare(q, k_cache, v_cache, out, past_len, B, H_q, H_kv, T_max, D, N,
                                                  max_past_len, dtype, &need, &zero_off, &zero_bytes);
    if (st != KVD_OK) return st;
    if (B == 0) return KVD_OK;
    if (need > kNoAllocScratchBytes) return KVD_ERR_WORKSPACE;
    void *scratch = nullptr;
    if ((st = noalloc_scratch(&scratch)) != KVD_OK) return st;
    // The merge counters must start at zero (a call that gave up on a
    // timeout may have left some set); a memset allocates nothing.
    if (zero_bytes != 0 &&
        cudaMemsetAsync(static_cast<unsigned char *>(scratch) + zero_off, 0, zero_bytes,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return KVD_ERR_CUDA;
    return kvd_decode_attention(q, k_cache, v_cache, out, past_len, B, H_q, H_kv, T_max, D, N,
                                max_past_len, scale, dtype, scratch, kNoAllocScratchBytes, err_word,
                                stream);
}
