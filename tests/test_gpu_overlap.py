"""Consecutive decode steps that start before the previous kernel finishes.

Small layers (kvd_plan_info.early_start) let the next kernel on the stream
launch early: with KVD_STEP_HISTORY_STABLE their CTAs read past_len and load
their first K/V tiles before they wait for the previous kernel.  The tcgen05
cases chain layers through the merge pass's early release of the next launch
(the flag changes nothing there).  Only what the previous kernel may write has to wait: q, the
new rows, the workspace.  These tests chain layers whose q, k_new and v_new
are the previous layer's output, so a read issued before the wait would see
stale data, and require the chained results to be bit-identical to layers run
one at a time with the device synchronised in between (which the step tests
tie to the oracle).
"""
import numpy as np
import pytest
import torch

import kv_cache_decode_append_gb300 as kvd
from kv_cache_decode_append_gb300 import workloads as wl
from helpers import TOL, row_rel_err, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _same_bits(a: torch.Tensor, b: torch.Tensor) -> bool:
    return np.array_equal(to_np(a).view(np.uint8), to_np(b).view(np.uint8))


def _chain(w, past, layers, flags, graph=False, seed=9100):
    """Run `layers` fused steps on one stream; layer l > 0 takes the output of
    layer l - 1 as its q, k_new and v_new (MHA shapes: H_q == H_kv)."""
    assert w.H_q == w.H_kv
    past = torch.as_tensor(past, dtype=torch.int32)
    max_past = int(past.max())
    past_d = past.to(DEV)
    ins = [wl.layer_inputs(w, l, past, device=DEV, seed_base=seed + l) for l in range(layers)]
    outs = [torch.full_like(ins[0]["q"], float("nan")) for _ in range(layers)]
    ws = kvd.alloc_workspace(w.B, w.H_q, w.H_kv, w.D, w.N, max_past, w.torch_dtype, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)

    def run(sync_each):
        for l in range(layers):
            x = ins[l]
            q = x["q"] if l == 0 else outs[l - 1]
            kn = x["k_new"] if l == 0 else outs[l - 1]
            kvd.kvd_decode_step(q, x["k_cache"], x["v_cache"], kn, kn, outs[l], past_d, max_past, 0.0, ws, err,
                                flags=flags)
            if sync_each:
                torch.cuda.synchronize()

    if graph:
        for _ in range(2):  # (idempotent: the same rows are appended again)
            run(False)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run(False)
        for o in outs:
            o.fill_(float("nan"))
        g.replay()
    else:
        run(flags is None)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return ins, outs


CASES = [  # (B, H, D, N, T_max, past, dtype)
    (8, 12, 64, 1, 1024, [1023] * 8, "bf16"),               # GPT-2 Small batch 8 at the context limit
    (1, 12, 64, 1, 1024, [1000], "f32"),                    # GPT-2 Small at the pages' measured point
    (1, 12, 64, 4, 1024, [512], "f32"),                     # chunked decode
    (3, 4, 128, 2, 700, [31, 697, 300], "bf16"),            # ragged histories, new keys across tiles
    (2, 6, 64, 3, 300, [0, 257], "f16"),                    # empty history
    (3, 4, 128, 20, 700, [300, 677, 0], "bf16"),            # 20 rows per head: tcgen05, new keys across tiles
    (2, 2, 64, 40, 900, [860, 1], "f16"),                   # 40 rows, fp16: tcgen05
    (32, 8, 128, 20, 4100, [4000 - 97 * i for i in range(32)], "bf16"),  # tcgen05, long ranges: merge pass
]


@pytest.mark.parametrize("case", CASES, ids=[f"c{i}" for i in range(len(CASES))])
@pytest.mark.parametrize("flags", [0, kvd.KVD_STEP_HISTORY_STABLE], ids=["plain", "stable"])
@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
def test_chained_layers_match_serial(case, flags, graph):
    B, H, D, N, T_max, past, dtype = case
    w = wl.Workload(0, "chain", L=1, B=B, H_q=H, H_kv=H, D=D, N=N, dtype=dtype, T_max=T_max, P=0)
    plan = kvd.kvd_decode_plan(B, H, H, D, N, max(past), w.torch_dtype)
    assert plan["early_start"] == 1 or plan["tensor_cores"] == 2
    layers = 6
    ins_ref, ref = _chain(w, past, layers, None)
    ins, got = _chain(w, past, layers, flags, graph=graph)
    for l in range(layers):
        assert _same_bits(got[l], ref[l]), f"layer {l}"
        assert _same_bits(ins[l]["k_cache"], ins_ref[l]["k_cache"]), f"layer {l} K cache"
        assert _same_bits(ins[l]["v_cache"], ins_ref[l]["v_cache"]), f"layer {l} V cache"


@pytest.mark.parametrize("name", ["gpt2s_b8_p1023_bf16", "gpt2s_12layer_p1000_f32", "gpt2s_chunked_p512_f32"])
def test_small_workloads_run_in_cluster_mode(name):
    """The GPT-2 Small layers are small enough for cluster mode (one cluster of
    CTAs per KV head, shares merged in distributed shared memory)."""
    w = wl.WORKLOADS[name]
    plan = kvd.kvd_decode_plan(w.B, w.H_q, w.H_kv, w.D, w.N, int(wl.past_lens(w).max()), w.torch_dtype)
    assert plan["early_start"] == 1 and plan["cluster"] >= 2
    assert plan["grid"] == w.B * w.H_kv * -(-w.group * w.N // plan["rows_per_block"]) * plan["cluster"]


def test_stable_flag_matches_oracle(oracle_lib):
    """One stable-history step against the oracle directly (GPT-2 b8 shape, bf16)."""
    w = wl.WORKLOADS["gpt2s_b8_p1023_bf16"]
    past = wl.past_lens(w)
    t = wl.layer_inputs(w, 3, past)
    g = {k: v.to(DEV) for k, v in t.items()}
    out = torch.empty_like(g["q"])
    ws = kvd.alloc_workspace(w.B, w.H_q, w.H_kv, w.D, w.N, int(past.max()), w.torch_dtype, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvd.kvd_decode_step(g["q"], g["k_cache"], g["v_cache"], g["k_new"], g["v_new"], out, past.to(DEV),
                        int(past.max()), 0.0, ws, err, flags=kvd.KVD_STEP_HISTORY_STABLE)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    h = {k: to_np(v) for k, v in t.items()}
    assert oracle_lib.append(h["k_cache"], h["v_cache"], h["k_new"], h["v_new"], past.numpy(), "bf16") == 0
    assert _same_bits(g["k_cache"], torch.from_numpy(h["k_cache"]).view(torch.bfloat16))
    ref, st = oracle_lib.decode_attention(h["q"], h["k_cache"], h["v_cache"], past.numpy(), "bf16")
    assert st == 0
    assert row_rel_err(out.double().cpu().numpy(), ref) <= TOL["bf16"]


def test_stable_flag_rejects_unknown_bits():
    w = wl.Workload(0, "x", L=1, B=1, H_q=2, H_kv=2, D=64, N=1, dtype="bf16", T_max=64, P=0)
    past = torch.tensor([10], dtype=torch.int32)
    t = wl.layer_inputs(w, 0, past, device=DEV)
    ws = kvd.alloc_workspace(1, 2, 2, 64, 1, 10, torch.bfloat16, DEV)
    with pytest.raises(kvd.KvdError):
        kvd.kvd_decode_step(t["q"], t["k_cache"], t["v_cache"], t["k_new"], t["v_new"], torch.empty_like(t["q"]),
                            past.to(DEV), 10, 0.0, ws, None, flags=0x80)


def test_stable_bad_past_len_reported_after_wait():
    """An out-of-range past_len under KVD_STEP_HISTORY_STABLE: the sequence is
    skipped and the error bit lands in an error word zeroed just before the call."""
    w = wl.Workload(0, "bad", L=1, B=3, H_q=4, H_kv=4, D=64, N=1, dtype="bf16", T_max=600, P=0)
    past = torch.tensor([100, 400, 50], dtype=torch.int32)   # 400 > max_past_len = 300
    t = wl.layer_inputs(w, 0, past.clamp_max(300), seed_base=9300)
    g = {k: v.to(DEV) for k, v in t.items()}
    before = g["k_cache"].clone()
    out = torch.full_like(g["q"], 7.0)
    err = torch.full((1,), 123, dtype=torch.int32, device=DEV)
    ws = kvd.alloc_workspace(3, 4, 4, 64, 1, 300, torch.bfloat16, DEV)
    err.zero_()
    kvd.kvd_decode_step(g["q"], g["k_cache"], g["v_cache"], g["k_new"], g["v_new"], out, past.to(DEV), 300,
                        0.0, ws, err, flags=kvd.KVD_STEP_HISTORY_STABLE)
    torch.cuda.synchronize()
    assert int(err.item()) == kvd.KVD_DEVERR_PAST_LEN
    assert _same_bits(g["k_cache"][1], before[1])
    assert bool((out[1] == 7.0).all())
    assert bool(torch.isfinite(out[0]).all() and torch.isfinite(out[2]).all())
