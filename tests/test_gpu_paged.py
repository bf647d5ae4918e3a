"""Paged cache on the GPU: kvd_paged_append / kvd_paged_decode_attention /
kvd_paged_decode_step against the paged oracle, and against the contiguous path.

Pages come from the contiguous inputs laid out as a shuffled pool with unused
NaN pages (workloads.to_paged).  Over the same logical data the paged kernels
run the same tiles in the same order as the contiguous ones (the planner picks
the CUDA-core or the tensor-core kernel from the shapes alone, whatever the
layout), so their outputs must match the contiguous outputs bit for bit; the
paged append must write exactly the page slots the oracle writes and nothing
else.
"""
import numpy as np
import pytest
import torch

import kv_cache_decode_append_gb300 as kvd
from kv_cache_decode_append_gb300 import workloads as wl
from helpers import TOL, row_rel_err, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def orc():
    import __graft_entry__
    __graft_entry__.build()
    import oracle
    return oracle.load()


def _same_bits(a: torch.Tensor, b: torch.Tensor) -> bool:
    return np.array_equal(to_np(a).view(np.uint8), to_np(b).view(np.uint8))


def _inputs(w, past, page_size, seed, device="cpu"):
    past = torch.as_tensor(past, dtype=torch.int32)
    t = wl.layer_inputs(w, 0, past, device=device, seed_base=seed)
    kp, vp, table = wl.to_paged(t["k_cache"], t["v_cache"], page_size, extra_pages=3, seed=seed)
    return past, t, kp, vp, table


def _run(w, past, t, kp, vp, table, fused=False):
    """Paged path on copies of the inputs; returns (out, k_pages, v_pages, err)."""
    max_past = int(past.max())
    g = {k: v.to(DEV) for k, v in t.items()}
    kpd, vpd, tbl = kp.to(DEV).clone(), vp.to(DEV).clone(), table.to(DEV)
    past_d = past.to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = kvd.alloc_workspace(w.B, w.H_q, w.H_kv, w.D, w.N, max_past, w.torch_dtype, DEV)
    out = torch.full_like(g["q"], float("nan"))
    if fused:
        kvd.kvd_paged_decode_step(g["q"], kpd, vpd, g["k_new"], g["v_new"], out, tbl, past_d, max_past, 0.0, ws, err)
    else:
        kvd.kvd_paged_append(kpd, vpd, g["k_new"], g["v_new"], tbl, past_d, max_past, err)
        kvd.kvd_paged_decode_attention(g["q"], kpd, vpd, out, tbl, past_d, max_past, 0.0, ws, err)
    torch.cuda.synchronize()
    return out, kpd, vpd, int(err.item())


def _contiguous(w, past, t):
    max_past = int(past.max())
    g = {k: v.to(DEV).clone() for k, v in t.items()}
    past_d = past.to(DEV)
    ws = kvd.alloc_workspace(w.B, w.H_q, w.H_kv, w.D, w.N, max_past, w.torch_dtype, DEV)
    out = torch.full_like(g["q"], float("nan"))
    kvd.kvd_append(g["k_cache"], g["v_cache"], g["k_new"], g["v_new"], past_d, max_past)
    kvd.kvd_decode_attention(g["q"], g["k_cache"], g["v_cache"], out, past_d, max_past, 0.0, ws)
    torch.cuda.synchronize()
    return out


def _check(orc, w, past, page_size, seed):
    past, t, kp, vp, table = _inputs(w, past, page_size, seed)
    out, kpd, vpd, err = _run(w, past, t, kp, vp, table)
    assert err == 0
    # append: exactly the oracle's page slots, everything else untouched
    h = {k: to_np(v) for k, v in t.items()}
    kpo, vpo = to_np(kp), to_np(vp)
    assert orc.paged_append(kpo, vpo, h["k_new"], h["v_new"], to_np(table), past.numpy(), w.dtype) == 0
    assert np.array_equal(to_np(kpd).view(np.uint8), kpo.view(np.uint8))
    assert np.array_equal(to_np(vpd).view(np.uint8), vpo.view(np.uint8))
    # attention: the paged oracle within tolerance, the contiguous kernel bit for bit
    ref, st = orc.paged_decode_attention(h["q"], kpo, vpo, to_np(table), past.numpy(), w.dtype)
    assert st == 0
    assert row_rel_err(out.double().cpu().numpy(), ref) <= TOL[w.dtype]
    assert _same_bits(out, _contiguous(w, past, t))
    # fused step: same pages and same output bits as append + attention
    out2, kpd2, vpd2, err2 = _run(w, past, t, kp, vp, table, fused=True)
    assert err2 == 0
    assert _same_bits(kpd2, kpd) and _same_bits(vpd2, vpd) and _same_bits(out2, out)


# (B, H_q, H_kv, D, N, T_max, past, dtype, page_size)
PAGED_CASES = [
    (3, 8, 2, 128, 1, 1000, [999, 0, 412], "bf16", 64),      # P+N = T_max, empty history
    (2, 12, 12, 64, 1, 1024, [1023, 700], "bf16", 128),      # GPT-2 shapes, last slot
    (2, 8, 4, 64, 5, 700, [63, 600], "f32", 64),             # new keys straddle a page
    (1, 32, 4, 128, 16, 600, [583], "bf16", 256),            # 128 query rows, chunk of 16
    (4, 6, 2, 64, 7, 1100, [1000, 3, 640, 64], "bf16", 512), # 3 row blocks, big pages
    (2, 2, 1, 128, 1, 2200, [2047, 2048], "f32", 64),        # MQA, fp32 D=128 (32-key tiles)
]


@pytest.mark.parametrize("case", PAGED_CASES, ids=[f"paged{i}" for i in range(len(PAGED_CASES))])
def test_paged_parity(orc, case):
    B, H_q, H_kv, D, N, T_max, past, dtype, ps = case
    w = wl.Workload(0, "paged", L=1, B=B, H_q=H_q, H_kv=H_kv, D=D, N=N, dtype=dtype, T_max=T_max, P=0)
    _check(orc, w, past, ps, seed=8100 + ps + N)


@pytest.mark.parametrize("name", ["gpt2s_b8_p1023_bf16", "gpt2s_12layer_p1000_f32"])
def test_paged_workloads(orc, name):
    w = wl.WORKLOADS[name]
    _check(orc, w, wl.past_lens(w), 64, seed=8300 + w.wid)


def test_paged_gqa_longctx_full_size(orc):
    """The long-context workload at full size, 64-token pages: the attention against
    the oracle (on the same data, contiguous) and bit for bit against the contiguous
    path, the fused step bit-identical to append + attention."""
    w = wl.WORKLOADS["gqa_longctx_b32_bf16"]
    past = wl.past_lens(w)
    _, t, kp, vp, table = _inputs(w, past, 64, seed=8500, device=DEV)
    out, _, _, err = _run(w, past, t, kp, vp, table)
    assert err == 0
    h = {k: to_np(v) for k, v in t.items()}
    assert orc.append(h["k_cache"], h["v_cache"], h["k_new"], h["v_new"], past.numpy(), w.dtype) == 0
    ref, st = orc.decode_attention(h["q"], h["k_cache"], h["v_cache"], past.numpy(), w.dtype)
    assert st == 0
    assert row_rel_err(out.double().cpu().numpy(), ref) <= TOL[w.dtype]
    assert _same_bits(out, _contiguous(w, past, t))
    out2, _, _, err2 = _run(w, past, t, kp, vp, table, fused=True)
    assert err2 == 0 and _same_bits(out2, out)


@pytest.mark.parametrize("case", [(16, 32, 8, 128, 6200, 6100, 2), (16, 32, 8, 128, 1100, 1000, 1)],
                         ids=["merge_pass", "in_kernel"])
def test_paged_merge_modes(orc, case):
    B, H_q, H_kv, D, T_max, max_past, launches = case
    assert kvd.kvd_decode_plan(B, H_q, H_kv, D, 1, max_past, "bf16")["launches"] == launches
    gen = torch.Generator().manual_seed(8700 + launches)
    past = torch.randint(0, max_past + 1, (B,), generator=gen, dtype=torch.int32)
    past[5] = max_past
    w = wl.Workload(0, "pmerge", L=1, B=B, H_q=H_q, H_kv=H_kv, D=D, N=1, dtype="bf16", T_max=T_max, P=0)
    _check(orc, w, past, 128, seed=8710 + launches)


def test_paged_bad_page_is_flagged_and_contained():
    """A needed block-table entry outside the pool: KVD_DEVERR_PAGE, no write outside
    the sequence's valid pages, the other sequences exact."""
    w = wl.Workload(0, "bad", L=1, B=3, H_q=4, H_kv=2, D=64, N=2, dtype="bf16", T_max=512, P=0)
    past = torch.tensor([300, 200, 100], dtype=torch.int32)
    past_, t, kp, vp, table = _inputs(w, past, 64, seed=8800)
    good, kpd_good, _, err = _run(w, past, t, kp, vp, table)
    assert err == 0
    bad_table = table.clone()
    bad_table[1, 3] = kp.shape[0] + 7      # sequence 1 needs pages 0..3 (tokens 0..201)
    for fused in (False, True):
        out, kpd, vpd, err = _run(w, past, t, kp, vp, bad_table, fused=fused)
        assert err & kvd.KVD_DEVERR_PAGE
        assert _same_bits(out[0], good[0]) and _same_bits(out[2], good[2])
        # sequence 1's new tokens go to its page 3, which is invalid: the pool is
        # exactly the good run's pool except that page
        page3 = int(table[1, 3])
        keep = torch.ones(kp.shape[0], dtype=torch.bool)
        keep[page3] = False
        assert _same_bits(kpd[keep.to(DEV)], kpd_good[keep.to(DEV)])
        assert _same_bits(kpd[page3], kp[page3])


@pytest.mark.parametrize("ps,N,tc", [(64, 1, 1), (256, 1, 1), (64, 5, 2)],
                         ids=["mma_ps64", "mma_ps256", "tcgen05_ps64"])
def test_paged_tensor_core_bad_page(ps, N, tc):
    """A bad block-table entry on the tensor-core kernels (4 rows per KV head: mma.sync;
    20 rows: tcgen05): flagged, contained to its sequence, no write into the pool for it."""
    w = wl.Workload(0, "badm", L=1, B=3, H_q=16, H_kv=4, D=128, N=N, dtype="bf16", T_max=1024, P=0)
    assert kvd.kvd_decode_plan(3, 16, 4, 128, N, 700, "bf16")["tensor_cores"] == tc
    past = torch.tensor([700, 300, 64], dtype=torch.int32)
    _, t, kp, vp, table = _inputs(w, past, ps, seed=8900 + ps + N)
    good, kpd_good, _, err = _run(w, past, t, kp, vp, table, fused=True)
    assert err == 0
    bad_table = table.clone()
    last = 300 // ps                      # sequence 1's page holding its new token
    bad_table[1, last] = kp.shape[0] + 3
    out, kpd, _, err = _run(w, past, t, kp, vp, bad_table, fused=True)
    assert err & kvd.KVD_DEVERR_PAGE
    assert _same_bits(out[0], good[0]) and _same_bits(out[2], good[2])
    page = int(table[1, last])
    keep = torch.ones(kp.shape[0], dtype=torch.bool)
    keep[page] = False
    assert _same_bits(kpd[keep.to(DEV)], kpd_good[keep.to(DEV)])
    assert _same_bits(kpd[page], kp[page])
