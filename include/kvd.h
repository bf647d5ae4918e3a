/*
 * kvd.h -- C ABI of the GB300 (sm_103a) KV-cache decode step.
 *
 * One decode step of GPT-style attention for one layer:
 *   1. kvd_append            writes the K/V of N new tokens in place into a
 *                            preallocated [B, H_kv, T_max, D] cache;
 *   2. kvd_decode_attention  attends the N new query rows over the whole
 *                            cached history (scaled q.K^T, softmax, .V) with
 *                            the history-offset causal mask and GQA grouping.
 *
 * Sources (page title and section):
 *   - The cache holds the K/V of past tokens, which do not change; decode feeds
 *     only the new tokens and appends their K/V: gitcode.csdn.net
 *     miniONNXRuntime article, section "KV Cache 原理"; shapes [1,H,T,D] +
 *     [1,H,1,D] -> [1,H,T+1,D] on the time axis: section "Decode Shape 示例".
 *   - Real engines write new K/V in place into preallocated slots rather than
 *     concatenating: jennyma11.github.io/infra/ch07-01 "7.1 自回归生成过程",
 *     section "Decode 阶段", note under code 1-2; openai-hub.com/news/2435
 *     "GPT-2缓存实测：千倍计算只快6倍", section "显存测量最容易被分配器误导".
 *   - Decode attention q.K^T/sqrt(D), softmax, .V with H_q query heads and
 *     H_kv KV heads: "7.1 自回归生成过程", code 1-2.
 *   - With P cached and N new tokens, new row i sees P+i+1 keys:
 *     "GPT-2缓存实测", section "一个很容易漏掉的错误".
 *   - Cache size 2 x layers x KV heads x head dim x tokens x batch x bytes:
 *     "GPT-2缓存实测", section "GPT-2缓存要占多少显存".
 *
 * Conventions for every entry point
 *   - Layouts are dense row-major: caches [B, H_kv, T_max, D]; q and out
 *     [B, H_q, N, D]; k_new and v_new [B, H_kv, N, D].  One dtype (fp32, bf16
 *     or fp16) covers q, caches, new K/V and out; arithmetic accumulates in fp32.
 *   - Pointers named as device pointers must be CUDA device memory of the
 *     current device and 16-byte aligned.  Every buffer is owned by the caller;
 *     the library allocates nothing, keeps no pointer after the call returns,
 *     and never synchronises the host with the device.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     All device work of a call is enqueued on it, in order.
 *   - The kernels are launched with programmatic stream serialization: each
 *     waits for the work queued before it (griddepcontrol.wait) before it
 *     touches anything that work may write, and lets the next kernel on the
 *     stream launch before it has finished.  A kernel of the caller's, launched
 *     next on the stream with the programmatic-serialization attribute, must
 *     itself wait (cudaGridDependencySynchronize) before it reads what these
 *     calls wrote; kernels launched without that attribute, copies and events
 *     are ordered as usual.  (KVD_STEP_HISTORY_STABLE, below, lets a call read
 *     the cached history before that wait.)
 *   - Argument errors are found on the host before anything is launched and are
 *     returned as a status; nothing is written then.  A launch failure returns
 *     KVD_ERR_CUDA.
 *   - past_len lives in device memory, so per-sequence violations are detected
 *     on the device: a sequence b with past_len[b] < 0, past_len[b] >
 *     max_past_len or past_len[b] + N > T_max is skipped (nothing of it is
 *     written) and KVD_DEVERR_PAST_LEN is OR-ed into *err_word when err_word is
 *     not NULL.  The kernels never trap and every wait they contain is bounded.
 *   - GQA: query head hq reads KV head hq / (H_q / H_kv).
 */
#ifndef KVD_H
#define KVD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvd_status {
    KVD_OK = 0,
    KVD_ERR_INVALID_ARG = 1, /* null pointer, bad size, H_q % H_kv != 0, N < 1, misalignment */
    KVD_ERR_CAPACITY = 2,    /* max_past_len + N > T_max, or max_past_len < 0 */
    KVD_ERR_UNSUPPORTED = 3, /* D not in {64, 128}, unknown dtype, too many query rows */
    KVD_ERR_WORKSPACE = 4,   /* workspace missing, misaligned or smaller than required */
    KVD_ERR_CUDA = 5         /* a CUDA call or launch failed */
} kvd_status;

/* Element types.  KVD_E4M3 is a cache format only (see the _e4m3 calls). */
typedef enum kvd_dtype { KVD_F32 = 0, KVD_BF16 = 1, KVD_F16 = 2, KVD_E4M3 = 3 } kvd_dtype;

/* Bits OR-ed into the device error word. */
#define KVD_DEVERR_PAST_LEN 1u /* a sequence had an out-of-range past_len and was skipped */
#define KVD_DEVERR_TIMEOUT 2u  /* a bounded shared-memory pipeline wait gave up */
#define KVD_DEVERR_PAGE 4u     /* a paged call met a block-table entry outside [0, num_pages) */
#define KVD_DEVERR_INTERNAL 8u /* a launch found an internal invariant broken and did nothing */

/*
 * kvd_append -- in-place cache update (step 1 of a decode step).
 *
 * For every sequence b < B, KV head h < H_kv and new token i < N:
 *   k_cache[b, h, past_len[b] + i, :] = k_new[b, h, i, :]   (bit copy)
 *   v_cache[b, h, past_len[b] + i, :] = v_new[b, h, i, :]
 * No other slot is touched; nothing is reallocated or concatenated.
 *
 *   k_cache, v_cache  device, [B, H_kv, T_max, D], modified in place
 *   k_new, v_new      device, [B, H_kv, N, D]
 *   past_len          device int32[B]: tokens cached BEFORE this append
 *   max_past_len      host bound on every past_len[b] (checked on the device)
 *   err_word          device uint32 or NULL (see conventions)
 * Returns KVD_OK, KVD_ERR_INVALID_ARG, KVD_ERR_CAPACITY, KVD_ERR_UNSUPPORTED or
 * KVD_ERR_CUDA.  D may be any positive multiple of 8 (bf16, fp16) or 4 (fp32).
 */
kvd_status kvd_append(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                      const int32_t *past_len, int B, int H_kv, int T_max, int D, int N,
                      int max_past_len, kvd_dtype dtype, uint32_t *err_word, void *stream);

/*
 * kvd_decode_workspace_bytes -- scratch size for kvd_decode_attention with the
 * same shape arguments on the current device (0 when the arguments are
 * invalid).  The split-T plan depends on the shapes and on the device's SM
 * count, so query it on the device that will run the call.
 */
size_t kvd_decode_workspace_bytes(int B, int H_q, int H_kv, int D, int N, int max_past_len,
                                  kvd_dtype dtype);

/*
 * kvd_decode_attention -- split-T attention of the new rows (step 2).
 *
 * Call after kvd_append with the SAME (pre-append) past_len.  For b < B,
 * query head hq < H_q, new row i < N, with h = hq / (H_q / H_kv) and
 * P = past_len[b]:
 *   s_j = scale * q[b,hq,i,:] . k_cache[b,h,j,:]     for j = 0 .. P+i
 *   out[b,hq,i,:] = sum_j softmax(s)_j * v_cache[b,h,j,:]
 * Slots j > P+i (including any stale or NaN slot past P+N-1) are never read.
 *
 *   q, out            device, [B, H_q, N, D]; out gets the input dtype
 *                     (bf16 / fp16 rounded to nearest even from the fp32 result)
 *   k_cache, v_cache  device, [B, H_kv, T_max, D], already appended
 *   scale             softmax scale; <= 0 selects 1/sqrt(D)
 *   workspace         device scratch of at least kvd_decode_workspace_bytes(...)
 *                     bytes, 256-byte aligned, zero-filled before its first use
 *                     (kvd_workspace_init or any zero fill); every complete call
 *                     leaves it zero-filled again, so it is reused as is.  Zero
 *                     it again after a call that reported KVD_DEVERR_TIMEOUT.
 *                     Calls that run concurrently need distinct workspaces.
 * Supported: D in {64, 128}; dtype fp32, bf16 or fp16; H_q % H_kv == 0;
 * (H_q / H_kv) * N <= 1024 (query rows per KV head; chunked prefill).
 * Returns KVD_OK or the first argument error found (see kvd_status).
 * The workspace size does not depend on the cache layout: the paged calls
 * below use the same kvd_decode_workspace_bytes.
 */
kvd_status kvd_decode_attention(const void *q, const void *k_cache, const void *v_cache,
                                void *out, const int32_t *past_len, int B, int H_q, int H_kv,
                                int T_max, int D, int N, int max_past_len, float scale,
                                kvd_dtype dtype, void *workspace, size_t workspace_bytes,
                                uint32_t *err_word, void *stream);

/*
 * kvd_decode_step -- kvd_append followed by kvd_decode_attention, in one
 * launch (the layer step of a decode iteration).
 *
 * Same result as calling kvd_append(k_cache, v_cache, k_new, v_new, past_len,
 * ...) and then kvd_decode_attention(q, k_cache, v_cache, out, past_len, ...)
 * with the same pre-append past_len: afterwards the cache slots P..P+N-1 of
 * every valid sequence hold k_new / v_new and out holds the attention of the
 * new rows.  The tile holding a sequence's new keys takes them from k_new /
 * v_new directly and writes them to their cache slots from shared memory, so
 * no separate append pass runs.  Arguments are those of the two calls;
 * workspace as for kvd_decode_attention (kvd_decode_workspace_bytes).
 * Sequences with an out-of-range past_len are skipped entirely (no cache write,
 * no output) and flagged with KVD_DEVERR_PAST_LEN.
 */
kvd_status kvd_decode_step(const void *q, void *k_cache, void *v_cache, const void *k_new,
                           const void *v_new, void *out, const int32_t *past_len, int B, int H_q,
                           int H_kv, int T_max, int D, int N, int max_past_len, float scale,
                           kvd_dtype dtype, void *workspace, size_t workspace_bytes,
                           uint32_t *err_word, void *stream);

/*
 * kvd_decode_step_flags -- kvd_decode_step with caller guarantees that let
 * the kernel start its reads before the work queued ahead of it on `stream`
 * has finished.  No counterpart in the source pages: the pages time the
 * cached decode step and name launch and scheduling overhead as what remains
 * of its cost ("GPT-2缓存实测：千倍计算只快6倍", section
 * "千倍计算量为何只换来6倍速度"; "7.1 自回归生成过程", section "Decode 阶段");
 * this call lets a layer's cache reads overlap that overhead.
 *
 * flags (bitwise OR; any other bit returns KVD_ERR_INVALID_ARG):
 *   KVD_STEP_HISTORY_STABLE -- no work queued on `stream` before this call
 *     writes past_len or the cache rows below past_len[b] (the history).
 *     Typical in a model: the kernels ahead of a layer's step write q, k_new
 *     and v_new (and other layers' caches), and past_len advances once per
 *     token after the last layer.  For a small layer (kvd_plan_info.early_start
 *     = 1) on a contiguous cache the kernel then reads past_len and loads its
 *     first K/V tiles before it waits for the previous kernel; q, k_new,
 *     v_new, the workspace and every write still wait.  Elsewhere the flag is
 *     accepted and changes nothing.  Breaking the guarantee gives wrong results
 *     (the history may be read before it is written); nothing is checked.
 * Everything else, including the result bit for bit, is kvd_decode_step's.
 */
#define KVD_STEP_HISTORY_STABLE 1u
kvd_status kvd_decode_step_flags(const void *q, void *k_cache, void *v_cache, const void *k_new,
                                 const void *v_new, void *out, const int32_t *past_len, int B, int H_q,
                                 int H_kv, int T_max, int D, int N, int max_past_len, float scale,
                                 kvd_dtype dtype, uint32_t flags, void *workspace, size_t workspace_bytes,
                                 uint32_t *err_word, void *stream);

/*
 * kvd_decode_step_host -- kvd_decode_step with the call's own inputs and its
 * output in host memory: the whole step as the pages time it per token, the
 * new token's q, K and V coming from the host side and the attention result
 * going back ("GPT-2缓存实测：千倍计算只快6倍", section "实验到底测了什么";
 * the decode step itself: "7.1 自回归生成过程", section "Decode 阶段").
 *
 *   q_host, k_new_host, v_new_host   page-locked host memory, read; layouts as
 *                                    for kvd_decode_step
 *   past_len_host                    page-locked host int32[B], read
 *   out_host                         page-locked host memory, written
 *   k_cache, v_cache                 device, as for kvd_decode_step (updated in
 *                                    place)
 *   staging                          device scratch of at least
 *                                    kvd_host_staging_bytes(B, H_q, H_kv, D, N,
 *                                    dtype) bytes, 256-byte aligned, owned by
 *                                    the caller; it holds the device copies of
 *                                    q, k_new, v_new, past_len and out
 *   workspace, workspace_bytes       as for kvd_decode_step
 *
 * Enqueues on `stream`, in order: copies of q, k_new, v_new and past_len from
 * the host into `staging` (cudaMemcpyAsync), kvd_decode_step on the staged
 * copies, and the copy of out back to out_host (five copies in all; see
 * kvd_decode_step_host_packed for one copy of the inputs).  Like every call here it
 * returns at once: out_host holds the result once `stream` has passed the
 * call, and the host buffers must stay valid and unchanged until then.  The
 * result is kvd_decode_step's, bit for bit.
 *
 * Errors, all found before anything is queued: every argument error of
 * kvd_decode_step (E4M3 caches are not taken: KVD_ERR_UNSUPPORTED); a host
 * buffer that is not page-locked (cudaHostAlloc / cudaHostRegister), so that
 * no copy can block the host: KVD_ERR_INVALID_ARG; staging null, misaligned
 * or too small: KVD_ERR_WORKSPACE.  A failed copy or launch: KVD_ERR_CUDA.
 */
kvd_status kvd_decode_step_host(const void *q_host, void *k_cache, void *v_cache, const void *k_new_host,
                                const void *v_new_host, void *out_host, const int32_t *past_len_host, int B,
                                int H_q, int H_kv, int T_max, int D, int N, int max_past_len, float scale,
                                kvd_dtype dtype, void *staging, size_t staging_bytes, void *workspace,
                                size_t workspace_bytes, uint32_t *err_word, void *stream);

/*
 * kvd_decode_step_host_packed -- kvd_decode_step_host with the four inputs in
 * one page-locked host block, copied to the device in one piece:
 *
 *   inputs_host   one page-locked host allocation of at least
 *                 kvd_host_staging_inputs_bytes(B, H_q, H_kv, D, N, dtype)
 *                 bytes, laid out as the staging buffer's input part: q at
 *                 offset 0, then k_new, v_new and past_len (int32[B]), each
 *                 starting on the next 256-byte boundary after the previous
 *                 one (kvd_host_staging_bytes gives the full layout)
 *
 * Everything else (arguments, result, errors) is kvd_decode_step_host's.  The
 * block must be a single allocation: a copy may not span two page-locked
 * allocations, even adjacent ones (the call then fails with KVD_ERR_CUDA).
 */
kvd_status kvd_decode_step_host_packed(const void *inputs_host, void *k_cache, void *v_cache, void *out_host, int B,
                                       int H_q, int H_kv, int T_max, int D, int N, int max_past_len, float scale,
                                       kvd_dtype dtype, void *staging, size_t staging_bytes, void *workspace,
                                       size_t workspace_bytes, uint32_t *err_word, void *stream);

/*
 * kvd_host_staging_bytes -- device bytes of kvd_decode_step_host's staging
 * buffer for these shapes: in this order q (B * H_q * N * D elements), k_new
 * and v_new (B * H_kv * N * D each), past_len (B int32) and out (as q), each
 * region starting on a 256-byte boundary.  0 for invalid shapes or dtypes
 * (E4M3 included).
 *
 * kvd_host_staging_inputs_bytes -- the bytes of that layout up to the end of
 * past_len (the four inputs): the size of kvd_decode_step_host_packed's
 * input block.
 */
size_t kvd_host_staging_bytes(int B, int H_q, int H_kv, int D, int N, kvd_dtype dtype);
size_t kvd_host_staging_inputs_bytes(int B, int H_q, int H_kv, int D, int N, kvd_dtype dtype);

/*
 * kvd_decode_plan -- how kvd_decode_attention would run these shapes on the
 * current device, without launching anything: keys per tile, the most tiles
 * one sequence-head can have (from max_past_len + N), the persistent grid
 * (one CTA per resident slot; each CTA streams an equal share of all tiles)
 * and block, dynamic shared memory, kernels launched per call (2 when the
 * ranges are long and a separate merge pass combines the heads split across
 * CTAs, else 1: the kernel merges them itself), the workspace size, the query
 * rows per block and whether the tensor-core kernel runs.  Returns the same
 * argument errors as kvd_decode_attention.
 */
typedef struct kvd_plan_info {
    int tile_keys;
    int max_tiles;
    int grid;
    int threads;
    int smem_bytes;
    int launches;
    size_t workspace_bytes;
    int rows_per_block;  /* query rows of a (b, h) handled together */
    int tensor_cores;    /* 2: the tcgen05 kernel (bf16 / fp16 caches, contiguous or paged,
                            with (H_q / H_kv) * N >= 17 query rows per KV head: blocks of
                            128 rows, each K/V tile read once per block of rows);
                            1: the mma.sync tensor-core kernel (bf16 / fp16 caches with
                            4 .. 16 rows for D = 128, 8 .. 16 for D = 64; E4M3 caches
                            with D = 128, in blocks of 8 rows when a KV head has at
                            most 8, else of 16); 0: the CUDA-core kernel */
    int early_start;     /* 1: a small layer (K/V of at most 26 MiB at max_past_len, on the
                            CUDA-core kernel): the next kernel on the stream may launch as
                            soon as this one starts, so its CTAs take free SM slots and,
                            with KVD_STEP_HISTORY_STABLE, start loading before this one ends */
    int cluster;         /* > 0: such a layer whose longest head fits in a few ring fills
                            runs as one thread-block cluster of `cluster` CTAs per
                            (b, h_kv, row block): each CTA loads its equal share of the
                            head's keys at once and the shares merge through distributed
                            shared memory (the workspace is then unused) */
} kvd_plan_info;

kvd_status kvd_decode_plan(int B, int H_q, int H_kv, int D, int N, int max_past_len,
                           kvd_dtype dtype, kvd_plan_info *info);

/*
 * kvd_decode_attention_noalloc -- kvd_decode_attention without a caller
 * workspace, for callers that cannot allocate device memory.
 *
 * The source pages describe no such entry point; it exists for callers that
 * may not allocate on their hot path, such as a plugin inside a host engine
 * that owns all device memory through its own pool and offers no allocator,
 * or a serving loop where cudaMalloc could block on the device or run out of
 * memory mid-run.  Arguments, semantics and results are those of
 * kvd_decode_attention, minus the workspace: the scratch is a 4 MiB array
 * built into the library (every device that loads the library holds it
 * until the process exits).  The function allocates nothing and calls no
 * allocating routine.
 *
 *   - Invalid arguments return their status, and shapes whose
 *     kvd_decode_workspace_bytes exceeds 4 MiB return KVD_ERR_WORKSPACE,
 *     before anything is queued on `stream`.
 *   - The first call on each device looks up that device's scratch address
 *     (cudaGetSymbolAddress, with the device current) and keeps it; make that
 *     first call before any stream capture on the device, and do not use this
 *     entry point on a device after cudaDeviceReset.
 *   - All calls on a device share the one scratch array: calls whose GPU work
 *     can overlap (unordered streams) race and give undefined results.
 *   - The scratch keeps the previous call's contents; each call clears the
 *     part that must start at zero (its merge counters, a few bytes per
 *     sequence-head) with cudaMemsetAsync on `stream` before it launches.
 */
kvd_status kvd_decode_attention_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                        void *out, const int32_t *past_len, int B, int H_q,
                                        int H_kv, int T_max, int D, int N, int max_past_len,
                                        float scale, kvd_dtype dtype, uint32_t *err_word,
                                        void *stream);

/*
 * Paged cache.  Real serving engines keep the cache in fixed-size pages and
 * write new tokens into their page slots in place (PagedAttention:
 * "7.1 自回归生成过程", section "Decode 阶段", note under code 1-2;
 * "GPT-2缓存实测", section "显存测量最容易被分配器误导").  Here:
 *
 *   k_pages, v_pages  device, [num_pages, H_kv, page_size, D]: one page holds
 *                     page_size consecutive tokens of one sequence for every KV
 *                     head, each head's rows contiguous (a tile of keys is one
 *                     contiguous run of a page)
 *   block_table       device int32 [B, max_pages]: logical page j of sequence b
 *                     is physical page block_table[b * max_pages + j]; token t
 *                     of (b, h) is row t % page_size of head h in logical page
 *                     t / page_size.  Only the entries of pages that hold tokens
 *                     0 .. past_len[b] + N - 1 are read.
 *   page_size         a power of two, >= 64 (a multiple of every tile size)
 *   max_pages         entries per block-table row; the capacity of a sequence is
 *                     max_pages * page_size tokens (the T_max of the contiguous
 *                     calls: max_past_len + N must fit, else KVD_ERR_CAPACITY)
 *   num_pages         pages in the pool
 *
 * Every other argument, the results and the workspace are those of the
 * contiguous call of the same name.  A block-table entry outside
 * [0, num_pages) that a sequence needs is found on the device: KVD_DEVERR_PAGE
 * is OR-ed into *err_word, nothing is written to or read from outside the pool,
 * and that sequence's cache writes for the bad page are skipped and its output
 * rows are unspecified.
 */
kvd_status kvd_paged_append(void *k_pages, void *v_pages, const void *k_new, const void *v_new,
                            const int32_t *block_table, const int32_t *past_len, int B, int H_kv,
                            int D, int N, int page_size, int max_pages, int num_pages,
                            int max_past_len, kvd_dtype dtype, uint32_t *err_word, void *stream);

kvd_status kvd_paged_decode_attention(const void *q, const void *k_pages, const void *v_pages,
                                      void *out, const int32_t *block_table,
                                      const int32_t *past_len, int B, int H_q, int H_kv, int D,
                                      int N, int page_size, int max_pages, int num_pages,
                                      int max_past_len, float scale, kvd_dtype dtype,
                                      void *workspace, size_t workspace_bytes, uint32_t *err_word,
                                      void *stream);

kvd_status kvd_paged_decode_step(const void *q, void *k_pages, void *v_pages, const void *k_new,
                                 const void *v_new, void *out, const int32_t *block_table,
                                 const int32_t *past_len, int B, int H_q, int H_kv, int D, int N,
                                 int page_size, int max_pages, int num_pages, int max_past_len,
                                 float scale, kvd_dtype dtype, void *workspace,
                                 size_t workspace_bytes, uint32_t *err_word, void *stream);

/*
 * 8-bit cache (E4M3).  Serving stacks also keep the cache in FP8, and decode is
 * where quantization pays most ("GPT-2缓存实测", section "实验到底测了什么", the
 * paragraph after the configuration table; "7.1 自回归生成过程", section "Decode
 * 阶段").  Here the K and V caches hold E4M3 codes (1 sign, 4 exponent, 3
 * fraction bits, bias 7, no infinities, largest finite value 448) with one
 * scale per cache: a stored code c stands for k_scale * value(c) (K) or
 * v_scale * value(c) (V).  q, new K/V and out are bf16 (the append also takes
 * fp32 or fp16 new rows), arithmetic is fp32.
 *
 *   k_cache, v_cache  device, [B, H_kv, T_max, D] bytes (E4M3 codes), D a
 *                     multiple of 16; contiguous layout only
 *   k_scale, v_scale  positive, finite
 *
 * kvd_append_e4m3 stores, for each new element x, the code of the fp32
 * quotient x / scale rounded to the nearest E4M3 value (ties to the even code,
 * magnitudes beyond 448 saturate to 448).  kvd_decode_attention_e4m3 and
 * kvd_decode_step_e4m3 are kvd_decode_attention / kvd_decode_step over such a
 * cache (the fused step quantizes the new rows exactly as kvd_append_e4m3
 * does).  Workspace: kvd_decode_workspace_bytes(..., KVD_E4M3).  Query rows
 * per KV head are processed in blocks of at most 4 (D = 64) or of 16 (D = 128,
 * on the tensor cores: kvd_plan_info.tensor_cores = 1).  Other arguments, errors
 * and device-side checks as for the bf16 calls; any other entry point given
 * KVD_E4M3 returns KVD_ERR_UNSUPPORTED, except kvd_append / kvd_paged_append,
 * which copy already-quantized rows bit for bit.
 */
kvd_status kvd_append_e4m3(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                           const int32_t *past_len, int B, int H_kv, int T_max, int D, int N,
                           int max_past_len, kvd_dtype new_dtype, float k_scale, float v_scale,
                           uint32_t *err_word, void *stream);

kvd_status kvd_decode_attention_e4m3(const void *q, const void *k_cache, const void *v_cache, void *out,
                                     const int32_t *past_len, int B, int H_q, int H_kv, int T_max, int D,
                                     int N, int max_past_len, float scale, float k_scale, float v_scale,
                                     void *workspace, size_t workspace_bytes, uint32_t *err_word,
                                     void *stream);

kvd_status kvd_decode_step_e4m3(const void *q, void *k_cache, void *v_cache, const void *k_new,
                                const void *v_new, void *out, const int32_t *past_len, int B, int H_q,
                                int H_kv, int T_max, int D, int N, int max_past_len, float scale,
                                float k_scale, float v_scale, void *workspace, size_t workspace_bytes,
                                uint32_t *err_word, void *stream);

/* kvd_workspace_init -- zero-fill a workspace on `stream` (asynchronous), as
 * kvd_decode_attention and kvd_decode_step need before a workspace's first use. */
kvd_status kvd_workspace_init(void *workspace, size_t workspace_bytes, void *stream);

/*
 * kvd_cache_bytes -- bytes of K and V caches for L layers:
 *   2 * L * H_kv * D * T * B * (4 for fp32, 2 for bf16 and fp16); 0 on invalid input.
 */
size_t kvd_cache_bytes(int L, int B, int H_kv, int D, int T, kvd_dtype dtype);

/* kvd_status_string -- a static, human-readable name for a status code. */
const char *kvd_status_string(kvd_status status);

#ifdef __cplusplus
}
#endif

#endif /* KVD_H */
