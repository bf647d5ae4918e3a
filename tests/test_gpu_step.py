"""kvd_decode_step (append + attention in one launch) on the GPU.

The fused step must leave exactly the cache kvd_append leaves (bit for bit,
including every untouched slot) and produce exactly the output of
kvd_append + kvd_decode_attention: the tile holding the new keys reads them
from k_new / v_new instead of the cache, so the arithmetic sees the same bits.
It is also compared with the oracle within the parity tolerance.
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


def _both_paths(w, past, seed=None, device_inputs=False):
    past = torch.as_tensor(past, dtype=torch.int32)
    t = wl.layer_inputs(w, 0, past, device=DEV if device_inputs else "cpu", seed_base=seed)
    max_past = int(past.max())
    past_d = past.to(DEV)
    ws = kvd.alloc_workspace(w.B, w.H_q, w.H_kv, w.D, w.N, max_past, w.torch_dtype, DEV)
    # separate calls
    g1 = {k: v.to(DEV).clone() for k, v in t.items()}
    out1 = torch.full_like(g1["q"], float("nan"))
    err1 = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvd.kvd_append(g1["k_cache"], g1["v_cache"], g1["k_new"], g1["v_new"], past_d, max_past, err1)
    kvd.kvd_decode_attention(g1["q"], g1["k_cache"], g1["v_cache"], out1, past_d, max_past, 0.0, ws, err1)
    # fused step
    g2 = {k: v.to(DEV).clone() for k, v in t.items()}
    out2 = torch.full_like(g2["q"], float("nan"))
    err2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvd.kvd_decode_step(g2["q"], g2["k_cache"], g2["v_cache"], g2["k_new"], g2["v_new"], out2, past_d,
                        max_past, 0.0, ws, err2)
    torch.cuda.synchronize()
    return t, past, (g1, out1, int(err1.item())), (g2, out2, int(err2.item()))


def _same_bits(a: torch.Tensor, b: torch.Tensor) -> bool:
    return np.array_equal(to_np(a).view(np.uint8), to_np(b).view(np.uint8))


def _check(orc, w, past, seed=None, device_inputs=False):
    t, past, (g1, out1, e1), (g2, out2, e2) = _both_paths(w, past, seed, device_inputs)
    assert e1 == 0 and e2 == 0
    assert _same_bits(g1["k_cache"], g2["k_cache"]) and _same_bits(g1["v_cache"], g2["v_cache"])
    assert _same_bits(out1, out2)
    # and against the oracle
    h = {k: to_np(v) for k, v in t.items()}
    assert orc.append(h["k_cache"], h["v_cache"], h["k_new"], h["v_new"], past.numpy(), w.dtype) == 0
    assert np.array_equal(to_np(g2["k_cache"]).view(np.uint8), h["k_cache"].view(np.uint8))
    assert np.array_equal(to_np(g2["v_cache"]).view(np.uint8), h["v_cache"].view(np.uint8))
    ref, st = orc.decode_attention(h["q"], h["k_cache"], h["v_cache"], past.numpy(), w.dtype)
    assert st == 0
    assert row_rel_err(out2.double().cpu().numpy(), ref) <= TOL[w.dtype]


@pytest.mark.parametrize("name", [n for n in wl.WORKLOADS if n != "gqa_longctx_b32_bf16"])
def test_step_workloads(orc, name):
    w = wl.WORKLOADS[name]
    ns = wl.CHUNKED_N if name == "gpt2s_chunked_p512_f32" else (w.N,)
    for N in ns:
        ww = wl.with_n(w, N)
        _check(orc, ww, wl.past_lens(ww))


def test_step_gqa_longctx_full_size(orc):
    w = wl.WORKLOADS["gqa_longctx_b32_bf16"]
    _check(orc, w, wl.past_lens(w), device_inputs=True)


# new keys straddling a tile boundary, P = 0, P + N = T_max, several row blocks
STEP_EDGES = [
    (2, 4, 2, 64, 5, 140, [62, 0], "f32"),
    (3, 8, 2, 128, 3, 700, [31, 697, 5], "bf16"),
    (1, 32, 4, 128, 16, 600, [583], "bf16"),
    (2, 6, 2, 64, 7, 1100, [1000, 60], "bf16"),
    (1, 2, 2, 128, 1, 1, [0], "f32"),
    (1, 4, 4, 64, 144, 300, [100], "f32"),           # chunked prefill on the CUDA cores: 144 rows, 18 row blocks
]


@pytest.mark.parametrize("case", STEP_EDGES, ids=[f"edge{i}" for i in range(len(STEP_EDGES))])
def test_step_edges(orc, case):
    B, H_q, H_kv, D, N, T_max, past, dtype = case
    w = wl.Workload(0, "edge", L=1, B=B, H_q=H_q, H_kv=H_kv, D=D, N=N, dtype=dtype, T_max=T_max, P=0)
    _check(orc, w, past, seed=7700 + D + N)


def test_step_skips_bad_sequences():
    """A rejected sequence gets no cache write and no output; the others are done."""
    w = wl.Workload(0, "bad", L=1, B=3, H_q=4, H_kv=2, D=64, N=2, dtype="bf16", T_max=600, P=0)
    past = torch.tensor([100, 400, 50], dtype=torch.int32)   # 400 > max_past_len = 300
    t = wl.layer_inputs(w, 0, past.clamp_max(300), seed_base=7800)
    g = {k: v.to(DEV) for k, v in t.items()}
    before = g["k_cache"].clone()
    out = torch.full_like(g["q"], 7.0)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = kvd.alloc_workspace(3, 4, 2, 64, 2, 300, torch.bfloat16, DEV)
    kvd.kvd_decode_step(g["q"], g["k_cache"], g["v_cache"], g["k_new"], g["v_new"], out, past.to(DEV), 300,
                        0.0, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) & kvd.KVD_DEVERR_PAST_LEN
    assert _same_bits(g["k_cache"][1], before[1])
    assert bool((out[1] == 7.0).all())
    assert _same_bits(g["k_cache"][0, :, 100:102], g["k_new"][0])
    assert bool(torch.isfinite(out[0]).all() and torch.isfinite(out[2]).all())


# (B, H_q, H_kv, D, N, T_max, past, dtype): a 4-row tensor-core step and an fp32
# CUDA-core step with a split head
HOST_CASES = [(4, 8, 2, 128, 1, 300, [100, 0, 297, 50], "bf16"),
              (2, 12, 12, 64, 3, 1100, [1000, 7], "f32")]


@pytest.mark.parametrize("case", HOST_CASES, ids=["bf16_tensor_cores", "f32"])
def test_step_host_buffers(orc, case):
    """kvd_decode_step_host: inputs and output in page-locked host memory, copied by
    the library through its staging buffer; bit-identical to kvd_decode_step."""
    B, H_q, H_kv, D, N, T_max, past, dtype = case
    w = wl.Workload(0, "host", L=1, B=B, H_q=H_q, H_kv=H_kv, D=D, N=N, dtype=dtype, T_max=T_max, P=0)
    past = torch.as_tensor(past, dtype=torch.int32)
    t = wl.layer_inputs(w, 0, past, device="cpu", seed_base=9900 + N)
    max_past = int(past.max())
    ws = kvd.alloc_workspace(B, H_q, H_kv, D, N, max_past, w.torch_dtype, DEV)
    # device path
    g1 = {k: v.to(DEV).clone() for k, v in t.items()}
    out1 = torch.full_like(g1["q"], float("nan"))
    kvd.kvd_decode_step(g1["q"], g1["k_cache"], g1["v_cache"], g1["k_new"], g1["v_new"], out1, past.to(DEV),
                        max_past, 0.0, ws)
    # host path (its own caches and workspace)
    kc, vc = t["k_cache"].to(DEV).clone(), t["v_cache"].to(DEV).clone()
    host = {k: t[k].pin_memory() for k in ("q", "k_new", "v_new")}
    past_h = past.pin_memory()
    out_h = torch.full(t["q"].shape, float("nan"), dtype=t["q"].dtype).pin_memory()
    staging = kvd.alloc_host_staging(B, H_q, H_kv, D, N, w.torch_dtype, DEV)
    ws2 = kvd.alloc_workspace(B, H_q, H_kv, D, N, max_past, w.torch_dtype, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvd.kvd_decode_step_host(host["q"], kc, vc, host["k_new"], host["v_new"], out_h, past_h, max_past, staging,
                             0.0, ws2, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert _same_bits(out_h, out1)
    assert _same_bits(kc, g1["k_cache"]) and _same_bits(vc, g1["v_cache"])
    ref, st = orc.decode_attention(to_np(t["q"]), to_np(g1["k_cache"]), to_np(g1["v_cache"]), past.numpy(), dtype)
    assert st == 0 and row_rel_err(out_h.double().numpy(), ref) <= TOL[dtype]

    # the four inputs in one block laid out as the staging buffer's: one copy
    hp = kvd.alloc_host_inputs(B, H_q, H_kv, D, N, t["q"].dtype)
    for key in ("q", "k_new", "v_new"):
        hp[key].copy_(t[key])
    hp["past_len"].copy_(past)
    kc2, vc2 = t["k_cache"].to(DEV).clone(), t["v_cache"].to(DEV).clone()
    out_p = torch.full(t["q"].shape, float("nan"), dtype=t["q"].dtype).pin_memory()
    kvd.kvd_decode_step_host_packed(hp, kc2, vc2, out_p, max_past, staging, 0.0, ws2, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert _same_bits(out_p, out1) and _same_bits(kc2, g1["k_cache"]) and _same_bits(vc2, g1["v_cache"])

    # errors return before anything is queued: out_h keeps its bits
    before = out_h.clone()
    raw = kvd.raw
    code = {torch.bfloat16: kvd.KVD_BF16, torch.float32: kvd.KVD_F32}[t["q"].dtype]

    def call(q_ptr, staging_bytes, ws_bytes):
        return raw.kvd_decode_step_host(q_ptr, kc.data_ptr(), vc.data_ptr(), host["k_new"].data_ptr(),
                                        host["v_new"].data_ptr(), out_h.data_ptr(), past_h.data_ptr(), B, H_q, H_kv,
                                        T_max, D, N, max_past, 0.0, code, staging.data_ptr(), staging_bytes,
                                        ws2.data_ptr(), ws_bytes, None, None)
    pageable = t["q"].clone()
    assert call(pageable.data_ptr(), staging.numel(), ws2.numel()) == kvd.KVD_ERR_INVALID_ARG
    assert call(host["q"].data_ptr(), staging.numel() - 1, ws2.numel()) == kvd.KVD_ERR_WORKSPACE
    assert call(host["q"].data_ptr(), staging.numel(), 16) == kvd.KVD_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert _same_bits(out_h, before)
