"""The tensor-core kernel (16-row blocks, mma.sync, tiles by TMA tensor maps) on the
GPU: grouped / chunked decode with 4+ (D = 128) or 8+ (D = 64) query rows per KV
head, bf16 and fp16, against the oracle; the fused step bit-identical to append +
attention; both merge modes."""
import pytest
import torch

import kv_cache_decode_append_gb300 as kvd
from kv_cache_decode_append_gb300 import workloads as wl
import test_gpu_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    import __graft_entry__
    __graft_entry__.build()
    import oracle
    return oracle.load()


# (B, H_q, H_kv, D, N, T_max, past, dtype) -- 4 .. 16 rows per KV head (more go to
# the tcgen05 kernel: test_gpu_tc5.py)
MMA_CASES = [
    (2, 32, 2, 128, 1, 900, [899, 130], "bf16"),           # 16 rows: one full block
    (3, 8, 1, 128, 2, 700, [512, 0, 695], "bf16"),         # 16 rows, chunk of 2, empty history
    (2, 16, 2, 64, 2, 1100, [1000, 61], "bf16"),           # D=64, 16 rows
    (1, 32, 8, 128, 3, 600, [583], "bf16"),                # 12 rows: chunk of 3, 4 padding rows
    (2, 12, 12, 64, 16, 1024, [1008, 512], "f16"),         # GPT-2 shapes, chunk of 16, fp16
    (4, 64, 4, 128, 1, 2000, [1999, 7, 1000, 64], "f16"),  # 16 rows, fp16, ragged
    (3, 16, 4, 128, 1, 800, [799, 0, 257], "bf16"),        # 4 rows: GQA decode, 12 padding rows
    (2, 8, 8, 64, 8, 640, [600, 33], "bf16"),              # D=64, 8 rows
]


@pytest.mark.parametrize("case", MMA_CASES, ids=[f"mma{i}" for i in range(len(MMA_CASES))])
def test_mma_parity(orc, case):
    B, H_q, H_kv, D, N, T_max, past, dtype = case
    plan = kvd.kvd_decode_plan(B, H_q, H_kv, D, N, max(past), dtype)
    assert plan["tensor_cores"] == 1 and plan["rows_per_block"] == 16
    w = wl.Workload(0, "mma", L=1, B=B, H_q=H_q, H_kv=H_kv, D=D, N=N, dtype=dtype, T_max=T_max, P=0)
    test_gpu_step._check(orc, w, past, seed=9400 + D + N)


# The last: 128 x 8 heads x 5 rows = 5120 real rows, more than the merge pass's
# capped grid has warps (4864 on 152 SMs): two rows per warp at a time, the last
# group of each head holding one.
@pytest.mark.parametrize("case", [(32, 64, 4, 128, 6200, 6100, 2), (16, 32, 2, 128, 1100, 1000, 1),
                                  (128, 40, 8, 128, 1100, 1000, 2)],
                         ids=["merge_pass", "in_kernel", "merge_pass_two_rows_per_warp"])
def test_mma_merge_modes(orc, case):
    B, H_q, H_kv, D, T_max, max_past, launches = case
    plan = kvd.kvd_decode_plan(B, H_q, H_kv, D, 1, max_past, "bf16")
    assert plan["tensor_cores"] == 1 and plan["launches"] == launches
    gen = torch.Generator().manual_seed(9450 + launches)
    past = torch.randint(0, max_past + 1, (B,), generator=gen, dtype=torch.int32)
    past[1] = max_past
    w = wl.Workload(0, "mmam", L=1, B=B, H_q=H_q, H_kv=H_kv, D=D, N=1, dtype="bf16", T_max=T_max, P=0)
    test_gpu_step._check(orc, w, past, seed=9460 + launches)


def test_kernel_choice():
    assert kvd.kvd_decode_plan(4, 32, 8, 128, 1, 1000, "bf16")["tensor_cores"] == 1   # 4 rows, D=128
    assert kvd.kvd_decode_plan(4, 16, 8, 128, 1, 1000, "bf16")["tensor_cores"] == 0   # 2 rows
    assert kvd.kvd_decode_plan(8, 12, 12, 64, 1, 1000, "bf16")["tensor_cores"] == 0   # 1 row, D=64
    assert kvd.kvd_decode_plan(4, 32, 2, 128, 1, 1000, "f32")["tensor_cores"] == 0    # fp32 cache
    assert kvd.kvd_decode_plan(4, 32, 2, 128, 1, 1000, "bf16")["tensor_cores"] == 1   # 16 rows
    assert kvd.kvd_decode_plan(4, 17, 1, 128, 1, 1000, "bf16")["tensor_cores"] == 2   # 17 rows: tcgen05
    assert kvd.kvd_decode_plan(4, 8, 8, 64, 3, 1000, "f16")["tensor_cores"] == 0      # 3 rows, D=64
