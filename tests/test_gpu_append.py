"""kv_append on the GPU against the oracle: the whole cache bit for bit."""
import numpy as np
import pytest
import torch

import kv_cache_decode_append_gb300 as kvd
from kv_cache_decode_append_gb300 import workloads as wl
from helpers import to_np

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def orc():
    import __graft_entry__
    __graft_entry__.build()
    import oracle
    return oracle.load()


def _run(orc, w, past, device_inputs=False, tail="nan"):
    """Append one layer on the GPU and with the oracle; compare every byte of both caches."""
    past = torch.as_tensor(past, dtype=torch.int32)
    t = wl.layer_inputs(w, 0, past, device=DEV if device_inputs else "cpu", tail_fill=tail)
    g = {k: v.to(DEV) for k, v in t.items()}
    host = {k: to_np(v) for k, v in t.items()}
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    max_past = int(past.max()) if past.numel() else 0
    kvd.kvd_append(g["k_cache"], g["v_cache"], g["k_new"], g["v_new"], past.to(DEV), max_past, err)
    torch.cuda.synchronize()
    st = orc.append(host["k_cache"], host["v_cache"], host["k_new"], host["v_new"], past.numpy(), w.dtype)
    assert st == 0
    assert int(err.item()) == 0
    assert np.array_equal(to_np(g["k_cache"]).view(np.uint8), host["k_cache"].view(np.uint8))
    assert np.array_equal(to_np(g["v_cache"]).view(np.uint8), host["v_cache"].view(np.uint8))


@pytest.mark.parametrize("name", [n for n in wl.WORKLOADS if n != "gqa_longctx_b32_bf16"])
def test_append_workloads(orc, name):
    w = wl.WORKLOADS[name]
    ns = wl.CHUNKED_N if name == "gpt2s_chunked_p512_f32" else (w.N,)
    for N in ns:
        ww = wl.with_n(w, N)
        _run(orc, ww, wl.past_lens(ww))


def test_append_gqa_longctx_full_size(orc):
    """The long-context workload at full size (one layer, 2 x 545 MB of cache)."""
    w = wl.WORKLOADS["gqa_longctx_b32_bf16"]
    _run(orc, w, wl.past_lens(w), device_inputs=True, tail="zero")


@pytest.mark.parametrize("dtype,D", [("f32", 4), ("bf16", 8), ("f32", 64), ("bf16", 128), ("bf16", 72)])
def test_append_edges(orc, dtype, D):
    # empty history, a sequence that fills the last slot, ragged lengths
    w = wl.Workload(0, "edge", L=1, B=4, H_q=3, H_kv=3, D=D, N=5, dtype=dtype, T_max=37, P=0)
    _run(orc, w, [0, 32, 17, 1])


def test_append_rejects_bad_sequences_on_device(orc):
    """past_len out of range: that sequence is untouched, the rest appended, error bit set."""
    w = wl.Workload(0, "bad", L=1, B=4, H_q=2, H_kv=2, D=64, N=3, dtype="bf16", T_max=20, P=0)
    past = torch.tensor([5, 18, -1, 9], dtype=torch.int32)   # 18 + 3 > 20, -1 < 0
    t = wl.layer_inputs(w, 0, past.clamp_min(0), device="cpu")
    g = {k: v.to(DEV) for k, v in t.items()}
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvd.kvd_append(g["k_cache"], g["v_cache"], g["k_new"], g["v_new"], past.to(DEV), 17, err)
    torch.cuda.synchronize()
    assert int(err.item()) & kvd.KVD_DEVERR_PAST_LEN
    got = to_np(g["k_cache"])
    ref = to_np(t["k_cache"])
    for b in (1, 2):  # rejected: bit-identical to before
        assert np.array_equal(got[b].view(np.uint8), ref[b].view(np.uint8))
    for b in (0, 3):
        P = int(past[b])
        assert np.array_equal(got[b, :, P:P + 3], to_np(t["k_new"])[b])
    # max_past_len is a host promise checked on the device too
    err.zero_()
    kvd.kvd_append(g["k_cache"], g["v_cache"], g["k_new"], g["v_new"],
                   torch.tensor([5, 9, 9, 9], dtype=torch.int32, device=DEV), 6, err)
    torch.cuda.synchronize()
    assert int(err.item()) & kvd.KVD_DEVERR_PAST_LEN


def test_append_host_errors_do_not_launch():
    w = wl.Workload(0, "h", L=1, B=2, H_q=2, H_kv=2, D=64, N=2, dtype="f32", T_max=8, P=0)
    t = {k: v.to(DEV) for k, v in wl.layer_inputs(w, 0, torch.zeros(2, dtype=torch.int32)).items()}
    before = t["k_cache"].clone()
    with pytest.raises(kvd.KvdError) as e:
        kvd.kvd_append(t["k_cache"], t["v_cache"], t["k_new"], t["v_new"],
                       torch.zeros(2, dtype=torch.int32, device=DEV), 7)
    assert e.value.status == kvd.KVD_ERR_CAPACITY
    torch.cuda.synchronize()
    assert torch.equal(before.isnan(), t["k_cache"].isnan())
