"""Decode attention on the GPU against the oracle, element by element.

Every case runs the whole step as a user would: kvd_append, then
kvd_decode_attention with the same pre-append past_len, through the C ABI.
Cache slots past each sequence's history hold NaN, so any masked slot that
leaked into the arithmetic would poison the output.  Tolerances (row-normwise
relative error, see helpers.TOL): 1e-5 for fp32, 1e-2 for bf16.
"""
import numpy as np
import pytest
import torch

import kv_cache_decode_append_gb300 as kvd
from kv_cache_decode_append_gb300 import workloads as wl
from helpers import TOL, elem_rel_err, row_rel_err, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def orc():
    import __graft_entry__
    __graft_entry__.build()
    import oracle
    return oracle.load()


def gpu_step(t, past, max_past=None, scale=0.0, err=None):
    """Append + attention on the GPU; returns (out, device caches)."""
    g = {k: v.to(DEV) for k, v in t.items()}
    q = g["q"]
    B, H_q, N, D = q.shape
    H_kv = g["k_cache"].shape[1]
    max_past = int(past.max()) if max_past is None else max_past
    past_d = past.to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV) if err is None else err
    ws = kvd.alloc_workspace(B, H_q, H_kv, D, N, max_past, q.dtype, DEV)
    out = torch.full_like(q, float("nan"))
    kvd.kvd_append(g["k_cache"], g["v_cache"], g["k_new"], g["v_new"], past_d, max_past, err)
    kvd.kvd_decode_attention(q, g["k_cache"], g["v_cache"], out, past_d, max_past, scale, ws, err)
    torch.cuda.synchronize()
    return out, g, int(err.item())


def oracle_step(orc, t, past, dtype, scale=None):
    h = {k: to_np(v) for k, v in t.items()}
    assert orc.append(h["k_cache"], h["v_cache"], h["k_new"], h["v_new"], past.numpy(), dtype) == 0
    ref, st = orc.decode_attention(h["q"], h["k_cache"], h["v_cache"], past.numpy(), dtype, scale)
    assert st == 0
    return ref


def check(orc, w, past, scale=0.0, device_inputs=False, seed_base=None):
    past = torch.as_tensor(past, dtype=torch.int32)
    t = wl.layer_inputs(w, 0, past, device=DEV if device_inputs else "cpu", seed_base=seed_base)
    out, _, err = gpu_step(t, past, scale=scale)
    assert err == 0
    ref = oracle_step(orc, t, past, w.dtype, scale if scale > 0 else None)
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    rel = row_rel_err(got, ref)
    assert rel <= TOL[w.dtype], f"{w.describe()}: row-normwise rel err {rel:.3e} (elementwise {elem_rel_err(got, ref):.3e})"
    return rel


@pytest.mark.parametrize("name", [n for n in wl.WORKLOADS if n != "gqa_longctx_b32_bf16"])
def test_workloads(orc, name):
    w = wl.WORKLOADS[name]
    ns = wl.CHUNKED_N if name == "gpt2s_chunked_p512_f32" else (w.N,)
    for N in ns:
        ww = wl.with_n(w, N)
        check(orc, ww, wl.past_lens(ww))


def test_gqa_longctx_full_size(orc):
    """The long-context GQA workload at full size (B=32, P~U[1024,8192]), one layer,
    in the launch configuration the benchmark times; every output row is checked."""
    w = wl.WORKLOADS["gqa_longctx_b32_bf16"]
    check(orc, w, wl.past_lens(w), device_inputs=True)


# (B, H_q, H_kv, D, N, T_max, past, dtype, scale)
EDGE_CASES = [
    (1, 4, 4, 64, 1, 1, [0], "f32", 0.0),                 # empty history, T_max = 1
    (2, 4, 2, 128, 5, 16, [0, 11], "bf16", 0.0),          # empty history with a chunk; P+N = T_max
    (3, 8, 8, 64, 1, 300, [77, 299, 1], "f32", 0.0),      # ragged lengths, last slot filled
    (2, 16, 2, 128, 1, 5000, [4999, 130], "bf16", 0.0),   # group 8, long and short, many splits
    (2, 8, 4, 64, 3, 700, [513, 0], "f32", 0.0),          # group 2, chunk of 3
    (1, 32, 4, 128, 16, 600, [583], "bf16", 0.0),         # 128 query rows per KV head
    (4, 6, 2, 64, 7, 1100, [1000, 3, 640, 64], "bf16", 0.0),  # 21 rows -> 3 row blocks
    (1, 12, 12, 64, 2, 1024, [1022], "f32", 0.37),        # explicit scale
    (2, 2, 1, 128, 1, 2200, [2047, 2048], "f32", 0.0),    # MQA, tile-boundary lengths
]


@pytest.mark.parametrize("case", EDGE_CASES, ids=[f"edge{i}" for i in range(len(EDGE_CASES))])
def test_edge_cases(orc, case):
    B, H_q, H_kv, D, N, T_max, past, dtype, scale = case
    w = wl.Workload(0, "edge", L=1, B=B, H_q=H_q, H_kv=H_kv, D=D, N=N, dtype=dtype, T_max=T_max, P=0)
    check(orc, w, past, scale=scale, seed_base=7000 + len(past) * 13 + D)


@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_groups_and_head_dims(orc, group, D):
    w = wl.Workload(0, "g", L=1, B=2, H_q=2 * group, H_kv=2, D=D, N=1, dtype="bf16", T_max=900, P=0)
    check(orc, w, [899, 450], seed_base=100 * group + D)


def test_single_token_permutation_invariance():
    """N = 1: permuting the (K, V) pairs of the visible slots leaves the GPU output unchanged."""
    w = wl.Workload(0, "perm", L=1, B=1, H_q=8, H_kv=2, D=128, N=1, dtype="f32", T_max=700, P=0)
    past = torch.tensor([600], dtype=torch.int32)
    t = wl.layer_inputs(w, 0, past, seed_base=9100)
    out, g, _ = gpu_step(t, past)
    perm = torch.randperm(601, generator=torch.Generator().manual_seed(5)).to(DEV)
    out2 = torch.empty_like(out)
    kc, vc = g["k_cache"].clone(), g["v_cache"].clone()
    kc[:, :, :601] = g["k_cache"][:, :, perm]
    vc[:, :, :601] = g["v_cache"][:, :, perm]
    p_d = past.to(DEV)
    ws = kvd.alloc_workspace(1, 8, 2, 128, 1, 600, torch.float32, DEV)
    kvd.kvd_decode_attention(g["q"], kc, vc, out2, p_d, 600, 0.0, ws)
    torch.cuda.synchronize()
    assert row_rel_err(out2.double().cpu().numpy(), out.double().cpu().numpy()) < 1e-5


def test_chunk_reversed_order_changes_result(orc):
    """N > 1: a cache holding new||old instead of old||new gives a different output."""
    w = wl.Workload(0, "rev", L=1, B=1, H_q=4, H_kv=4, D=64, N=8, dtype="f32", T_max=64, P=0)
    past = torch.tensor([40], dtype=torch.int32)
    t = wl.layer_inputs(w, 0, past, seed_base=9200)
    out, g, _ = gpu_step(t, past)
    kc, vc = g["k_cache"].clone(), g["v_cache"].clone()
    kc[0, :, :48] = torch.cat([g["k_cache"][0, :, 40:48], g["k_cache"][0, :, :40]], dim=1)
    vc[0, :, :48] = torch.cat([g["v_cache"][0, :, 40:48], g["v_cache"][0, :, :40]], dim=1)
    out2 = torch.empty_like(out)
    kvd.kvd_decode_attention(g["q"], kc, vc, out2, past.to(DEV), 40, 0.0,
                             kvd.alloc_workspace(1, 4, 4, 64, 8, 40, torch.float32, DEV))
    torch.cuda.synchronize()
    assert row_rel_err(out2.double().cpu().numpy(), out.double().cpu().numpy()) > 1e-2


def test_device_rejects_bad_sequences():
    """A sequence whose past_len breaks the host promise is skipped and flagged."""
    w = wl.Workload(0, "bad", L=1, B=3, H_q=4, H_kv=2, D=64, N=1, dtype="bf16", T_max=600, P=0)
    past = torch.tensor([100, 400, 50], dtype=torch.int32)
    t = wl.layer_inputs(w, 0, past, seed_base=9300)
    g = {k: v.to(DEV) for k, v in t.items()}
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.full_like(g["q"], 7.0)
    ws = kvd.alloc_workspace(3, 4, 2, 64, 1, 300, torch.bfloat16, DEV)
    kvd.kvd_append(g["k_cache"], g["v_cache"], g["k_new"], g["v_new"], past.to(DEV), 300, err)
    kvd.kvd_decode_attention(g["q"], g["k_cache"], g["v_cache"], out, past.to(DEV), 300, 0.0, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) & kvd.KVD_DEVERR_PAST_LEN
    assert bool((out[1] == 7.0).all())          # skipped: untouched
    assert bool(torch.isfinite(out[0]).all() and torch.isfinite(out[2]).all())


def test_workspace_errors():
    w = wl.Workload(0, "ws", L=1, B=2, H_q=4, H_kv=2, D=128, N=1, dtype="bf16", T_max=4096, P=0)
    past = torch.tensor([4000, 4000], dtype=torch.int32)
    t = {k: v.to(DEV) for k, v in wl.layer_inputs(w, 0, past).items()}
    need = kvd.kvd_decode_workspace_bytes(2, 4, 2, 128, 1, 4000, "bf16")
    assert need > 0
    out = torch.empty_like(t["q"])
    small = torch.zeros(need - 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(kvd.KvdError) as e:
        kvd.kvd_decode_attention(t["q"], t["k_cache"], t["v_cache"], out, past.to(DEV), 4000, 0.0, small)
    assert e.value.status == kvd.KVD_ERR_WORKSPACE
    with pytest.raises(kvd.KvdError) as e:
        kvd.kvd_decode_attention(t["q"], t["k_cache"], t["v_cache"], out, past.to(DEV), 4000, 0.0, None)
    assert e.value.status == kvd.KVD_ERR_WORKSPACE


def test_repeated_calls_reuse_workspace(orc):
    """The same workspace serves consecutive calls and layers (no stale state)."""
    w = wl.Workload(0, "rep", L=1, B=3, H_q=8, H_kv=2, D=128, N=2, dtype="bf16", T_max=3000, P=0)
    past = torch.tensor([2900, 17, 1500], dtype=torch.int32)
    ws = kvd.alloc_workspace(3, 8, 2, 128, 2, 2900, torch.bfloat16, DEV)
    for layer in range(3):
        t = wl.layer_inputs(w, 0, past, seed_base=9400 + layer)
        g = {k: v.to(DEV) for k, v in t.items()}
        out = torch.empty_like(g["q"])
        kvd.kvd_append(g["k_cache"], g["v_cache"], g["k_new"], g["v_new"], past.to(DEV), 2900)
        kvd.kvd_decode_attention(g["q"], g["k_cache"], g["v_cache"], out, past.to(DEV), 2900, 0.0, ws)
        torch.cuda.synchronize()
        ref = oracle_step(orc, t, past, "bf16")
        assert row_rel_err(out.double().cpu().numpy(), ref) <= TOL["bf16"]


# Heads split across CTAs are merged inside the kernel on short ranges and by a
# second launch on long ones: both ways, on ragged lengths.
# (B, H_q, H_kv, D, T_max, max_past, launches)
MERGE_MODES = [
    (16, 32, 8, 128, 6200, 6100, 2),   # ~40 tile units per CTA: separate merge pass
    (16, 32, 8, 128, 1100, 1000, 1),   # ~8 tile units per CTA: merged in the kernel
]


@pytest.mark.parametrize("case", MERGE_MODES, ids=["merge_pass", "in_kernel"])
def test_merge_modes(orc, case):
    B, H_q, H_kv, D, T_max, max_past, launches = case
    assert kvd.kvd_decode_plan(B, H_q, H_kv, D, 1, max_past, "bf16")["launches"] == launches
    gen = torch.Generator().manual_seed(9900 + launches)
    past = torch.randint(0, max_past + 1, (B,), generator=gen, dtype=torch.int32)
    past[3] = max_past
    w = wl.Workload(0, "merge", L=1, B=B, H_q=H_q, H_kv=H_kv, D=D, N=1, dtype="bf16", T_max=T_max, P=0)
    check(orc, w, past, seed_base=9910 + launches)
