"""The tcgen05 kernel (128-row blocks, scores and output accumulators in tensor
memory) on the GPU: chunked decode and chunked prefill with more than 16 query rows
per KV head, bf16 and fp16, D = 64 and 128, contiguous and paged caches, against the
oracle; the fused step bit-identical to append + attention, paged bit-identical to
contiguous; both merge modes."""
import pytest
import torch

import kv_cache_decode_append_gb300 as kvd
from kv_cache_decode_append_gb300 import workloads as wl
import test_gpu_paged
import test_gpu_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    import __graft_entry__
    __graft_entry__.build()
    import oracle
    return oracle.load()


# (B, H_q, H_kv, D, N, T_max, past, dtype)
TC5_CASES = [
    (3, 8, 1, 128, 4, 700, [512, 0, 695], "bf16"),           # 32 rows, empty history
    (2, 16, 2, 64, 3, 1100, [1000, 61], "bf16"),             # D=64, 24 rows
    (1, 32, 4, 128, 16, 600, [583], "bf16"),                 # 128 rows: chunk of 16 over two tiles
    (2, 4, 4, 128, 17, 300, [0, 283], "f16"),                # 17 rows (MHA chunk), fp16, P + N = T_max
    (2, 12, 12, 64, 32, 1024, [992, 100], "f16"),            # GPT-2 shapes, chunk of 32, fp16
    (4, 32, 8, 128, 8, 2100, [2092, 7, 1000, 64], "bf16"),   # 32 rows, ragged
    (1, 4, 4, 128, 128, 400, [200], "bf16"),                 # chunked prefill: 128 new keys, 3 tiles
    (2, 16, 1, 64, 8, 520, [512, 1], "bf16"),                # D=64, 128 rows
    (2, 8, 2, 128, 5, 69, [0, 64], "f16"),                   # 20 rows, whole history in the masked tile
    (1, 8, 2, 128, 64, 400, [300], "bf16"),                  # chunked prefill: 256 rows, two row blocks
    (2, 10, 2, 64, 32, 300, [200, 17], "f16"),               # 160 rows (GQA 5), D=64: a full and a partial block
]


@pytest.mark.parametrize("case", TC5_CASES, ids=[f"tc5_{i}" for i in range(len(TC5_CASES))])
def test_tc5_parity(orc, case):
    B, H_q, H_kv, D, N, T_max, past, dtype = case
    plan = kvd.kvd_decode_plan(B, H_q, H_kv, D, N, max(past), dtype)
    assert plan["tensor_cores"] == 2 and plan["rows_per_block"] == 128
    w = wl.Workload(0, "tc5", L=1, B=B, H_q=H_q, H_kv=H_kv, D=D, N=N, dtype=dtype, T_max=T_max, P=0)
    test_gpu_step._check(orc, w, past, seed=9600 + D + N)


# The last two: 64 x 8 heads x 17 rows = 8704 real rows, more than the merge
# pass's capped grid has warps (8 four-warp CTAs per SM: 4864 on 152 SMs), so
# its warps take two rows at a time and the last group of each head holds one.
@pytest.mark.parametrize("case", [(32, 64, 4, 128, 2, 6200, 6100, 2), (4, 32, 2, 128, 2, 1100, 1000, 1),
                                  (64, 8, 8, 128, 17, 560, 540, 2), (64, 8, 8, 64, 17, 560, 540, 2)],
                         ids=["merge_pass", "in_kernel", "merge_pass_two_rows_per_warp",
                              "merge_pass_two_rows_per_warp_d64"])
def test_tc5_merge_modes(orc, case):
    B, H_q, H_kv, D, N, T_max, max_past, launches = case
    plan = kvd.kvd_decode_plan(B, H_q, H_kv, D, N, max_past, "bf16")
    assert plan["tensor_cores"] == 2 and plan["launches"] == launches
    gen = torch.Generator().manual_seed(9650 + launches)
    past = torch.randint(0, max_past + 1, (B,), generator=gen, dtype=torch.int32)
    past[1] = max_past
    w = wl.Workload(0, "tc5m", L=1, B=B, H_q=H_q, H_kv=H_kv, D=D, N=N, dtype="bf16", T_max=T_max, P=0)
    test_gpu_step._check(orc, w, past, seed=9660 + launches)


# (B, H_q, H_kv, D, N, T_max, past, dtype, page_size)
TC5_PAGED_CASES = [
    (2, 8, 1, 128, 4, 1000, [999 - 4, 130], "bf16", 64),     # 32 rows, 64-token pages
    (2, 12, 12, 64, 24, 1024, [1000, 333], "f16", 128),      # 24 rows (MHA chunk), fp16
    (1, 8, 2, 128, 64, 512, [400], "bf16", 64),              # 256 rows: two row blocks
]


@pytest.mark.parametrize("case", TC5_PAGED_CASES, ids=[f"tc5_paged{i}" for i in range(len(TC5_PAGED_CASES))])
def test_tc5_paged(orc, case):
    B, H_q, H_kv, D, N, T_max, past, dtype, ps = case
    assert kvd.kvd_decode_plan(B, H_q, H_kv, D, N, max(past), dtype)["tensor_cores"] == 2
    w = wl.Workload(0, "tc5p", L=1, B=B, H_q=H_q, H_kv=H_kv, D=D, N=N, dtype=dtype, T_max=T_max, P=0)
    test_gpu_paged._check(orc, w, past, ps, seed=9700 + ps + N)


def test_tc5_gqa_longctx_chunk8_full_size(orc):
    """The long-context workload's shapes and lengths at full size, 8 new tokens (32 rows
    per KV head), in the launch configuration bench.py --n-new 8 times."""
    w = wl.with_n(wl.WORKLOADS["gqa_longctx_b32_bf16"], 8)
    assert kvd.kvd_decode_plan(w.B, w.H_q, w.H_kv, w.D, w.N, max(wl.past_lens(w).tolist()), "bf16")["tensor_cores"] == 2
    test_gpu_step._check(orc, w, wl.past_lens(w), device_inputs=True)


@pytest.mark.parametrize("n_new", [16, 32], ids=["n16_64rows", "n32_128rows"])
def test_tc5_gqa_longctx_chunk_full_size(orc, n_new):
    """The long-context workload at full size with 16 and 32 new tokens: 64 and 128 rows
    per KV head (the launch configurations bench.py --n-new 16 / 32 time)."""
    w = wl.with_n(wl.WORKLOADS["gqa_longctx_b32_bf16"], n_new)
    plan = kvd.kvd_decode_plan(w.B, w.H_q, w.H_kv, w.D, w.N, max(wl.past_lens(w).tolist()), "bf16")
    assert plan["tensor_cores"] == 2 and plan["rows_per_block"] == 128
    test_gpu_step._check(orc, w, wl.past_lens(w), device_inputs=True)
