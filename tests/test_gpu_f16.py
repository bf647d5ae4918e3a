"""fp16 caches (q, new K/V and out fp16) on the GPU: the contiguous two-call and
fused paths against the oracle, fused bit-identical to two calls, and the paged
path bit-identical to the contiguous one (the same checks as the bf16 / fp32
tests, through their helpers)."""
import pytest

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


# (B, H_q, H_kv, D, N, T_max, past, page_size)
F16_CASES = [
    (8, 12, 12, 64, 1, 1024, [1023, 0, 512, 1, 64, 900, 333, 1000], 64),  # GPT-2 shapes, batch 8
    (4, 32, 8, 128, 1, 3000, [2999, 17, 1500, 2048], 128),                # GQA, ragged
    (2, 8, 2, 128, 4, 700, [63, 600], 64),                                # chunk of 4 across a tile
    (1, 32, 4, 128, 16, 600, [583], 256),                                 # 128 query rows
]


@pytest.mark.parametrize("case", F16_CASES, ids=[f"f16_{i}" for i in range(len(F16_CASES))])
def test_f16_contiguous_and_fused(orc, case):
    B, H_q, H_kv, D, N, T_max, past, _ = case
    w = wl.Workload(0, "f16", L=1, B=B, H_q=H_q, H_kv=H_kv, D=D, N=N, dtype="f16", T_max=T_max, P=0)
    test_gpu_step._check(orc, w, past, seed=9200 + D + N)


@pytest.mark.parametrize("case", F16_CASES, ids=[f"f16_{i}" for i in range(len(F16_CASES))])
def test_f16_paged(orc, case):
    B, H_q, H_kv, D, N, T_max, past, ps = case
    w = wl.Workload(0, "f16p", L=1, B=B, H_q=H_q, H_kv=H_kv, D=D, N=N, dtype="f16", T_max=T_max, P=0)
    test_gpu_paged._check(orc, w, past, ps, seed=9300 + D + N)
