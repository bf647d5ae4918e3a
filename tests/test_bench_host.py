"""bench.py's host-side arithmetic (CPU): the algorithmic bytes the roofline divides by,
the whole-job throughput, and the comment-insensitive kernel-source hash that decides
whether the committed ncu summary still describes the kernels."""
import bench
from kv_cache_decode_append_gb300 import workloads as wl


def test_long_context_algorithmic_bytes():
    """The default workload's per-layer bytes, counted term by term."""
    w = wl.WORKLOADS["gqa_longctx_b32_bf16"]
    past = wl.past_lens(w).tolist()
    assert sum(past) == 166230                                   # the seeded history lengths
    kv = 2 * 8 * 128 * 2 * (166230 + 32 * 1)                     # K and V over P_b + N keys, 8 KV heads
    qo = 2 * 32 * 32 * 1 * 128 * 2                               # q read and out written, 32 query heads
    app = 4 * 32 * 8 * 1 * 128 * 2                               # new K/V read and written
    assert bench.attn_bytes(w, past) == kv + qo == 681_533_440
    assert bench.layer_bytes(w, past) == kv + qo + app == 681_795_584


def test_e4m3_cache_bytes():
    """E4M3 cache: K/V and the appended codes count one byte, q / out / new K/V two."""
    w = wl.WORKLOADS["gqa_longctx_b32_bf16"]
    past = wl.past_lens(w).tolist()
    kv = 2 * 8 * 128 * 1 * (166230 + 32)
    qo = 2 * 32 * 32 * 128 * 2
    app = 2 * 32 * 8 * 128 * (2 + 1)
    assert bench.layer_bytes(w, past, cache_elem=1) == kv + qo + app == 341_225_472


def test_whole_job_throughput():
    # weak scaling: every rank moves the same bytes; the slowest rank's time counts
    assert bench.whole_job_gbs(10**9, 4, 2.0, 1) == 2.0
    assert bench.whole_job_gbs(10**9, 4, 2.0, 8) == 16.0


def test_code_only_ignores_comments_and_layout():
    a = 'asm volatile("x // kept" ::: "memory"); // note\n  int  k = 1; /* block\n comment */ k++;'
    b = 'asm volatile("x // kept" ::: "memory");\nint k = 1; k++;   // other note'
    assert bench._code_only(a) == bench._code_only(b)
    assert '"x // kept"' in bench._code_only(a)                   # string literals stay
    assert bench._code_only("int k = 1;") != bench._code_only("int k = 2;")
    assert bench._code_only('s = "a\\"b"; // c') == 's = "a\\"b";'  # escaped quote inside a string


def test_kernel_source_hash_is_stable():
    h = bench.kernel_source_hash()
    assert len(h) == 16 and h == bench.kernel_source_hash()
