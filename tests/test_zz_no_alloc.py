"""kvd_decode_attention_noalloc: decode attention with the library's built-in scratch.

This entry point is for callers that cannot allocate device memory where they
call the library (for example a plugin inside an engine that owns all device
memory, or a serving loop that must not risk cudaMalloc mid-run).  It must give
the same results as kvd_decode_attention with a caller-allocated workspace.

The file is named to be collected last, so that a run stopping at its first
failure has already run every other test.  Each case calls the new entry point
through the C ABI twice in a row (different shapes, so the second call finds
the first call's leftovers in the shared scratch) and compares both outputs
with the workspace entry point's: within the parity tolerance of the other
tests, and bit for bit, since both run the same plan and kernels on the same
inputs (the split heads' pieces are merged in a fixed order).
"""
import ctypes

import numpy as np
import pytest
import torch

import kv_cache_decode_append_gb300 as kvd
from kv_cache_decode_append_gb300 import workloads as wl
from helpers import TOL, row_rel_err

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def c_entry():
    import __graft_entry__
    __graft_entry__.build()
    lib = ctypes.CDLL(kvd.library_path())
    f = lib.kvd_decode_attention_noalloc
    vp, ci = ctypes.c_void_p, ctypes.c_int
    f.restype = ci
    f.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, ctypes.c_float, ci, vp, vp]
    return f


def _case(w, past, seed):
    past = torch.as_tensor(past, dtype=torch.int32)
    t = wl.layer_inputs(w, 0, past, device="cpu", seed_base=seed)
    g = {k: v.to(DEV) for k, v in t.items()}
    past_d = past.to(DEV)
    max_past = int(past.max())
    kvd.kvd_append(g["k_cache"], g["v_cache"], g["k_new"], g["v_new"], past_d, max_past)
    return g, past_d, max_past


def _reference(w, g, past_d, max_past):
    ws = kvd.alloc_workspace(w.B, w.H_q, w.H_kv, w.D, w.N, max_past, w.torch_dtype, DEV)
    out = torch.empty_like(g["q"])
    kvd.kvd_decode_attention(g["q"], g["k_cache"], g["v_cache"], out, past_d, max_past, 0.0, ws)
    return out


def _noalloc(c_entry, w, g, past_d, max_past, err):
    out = torch.full_like(g["q"], float("nan"))
    st = c_entry(g["q"].data_ptr(), g["k_cache"].data_ptr(), g["v_cache"].data_ptr(), out.data_ptr(),
                 past_d.data_ptr(), w.B, w.H_q, w.H_kv, w.T_max, w.D, w.N, max_past, 0.0,
                 kvd.KVD_BF16 if w.dtype == "bf16" else kvd.KVD_F32, err.data_ptr(),
                 torch.cuda.current_stream().cuda_stream)
    assert st == kvd.KVD_OK, kvd.kvd_status_string(st)
    return out


def _same_bits(a, b):
    return np.array_equal(a.contiguous().cpu().view(torch.uint8).numpy(), b.contiguous().cpu().view(torch.uint8).numpy())


def test_noalloc_matches_workspace_entry_point_twice_in_a_row(c_entry):
    cases = [
        # 32 long GQA sequences: ranges long enough for the separate merge
        # pass, which reads the split heads' partials from the scratch
        (wl.Workload(0, "gqa", L=1, B=32, H_q=32, H_kv=8, D=128, N=1, dtype="bf16", T_max=4200, P=0),
         [4100 - 97 * i for i in range(32)], 8101, 2),
        # chunked fp32 decode with several row blocks per KV head: split heads
        # merged inside the kernel through counters in the scratch
        (wl.Workload(0, "chunk", L=1, B=2, H_q=12, H_kv=4, D=64, N=4, dtype="f32", T_max=1500, P=0),
         [1200, 513], 8102, 1),
    ]
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    for w, past, seed, launches in cases:
        assert kvd.kvd_decode_plan(w.B, w.H_q, w.H_kv, w.D, w.N, max(past), w.torch_dtype)["launches"] == launches
        g, past_d, max_past = _case(w, past, seed)
        got = _noalloc(c_entry, w, g, past_d, max_past, err)
        ref = _reference(w, g, past_d, max_past)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        got_np, ref_np = got.double().cpu().numpy(), ref.double().cpu().numpy()
        assert np.isfinite(got_np).all()
        assert row_rel_err(got_np, ref_np) <= TOL[w.dtype]
        # the same plan and kernels on the same inputs: the same bits
        assert _same_bits(got, ref)


def test_noalloc_python_binding(c_entry):
    """The binding's wrapper calls the same entry point (bf16, split heads)."""
    w = wl.Workload(0, "py", L=1, B=4, H_q=16, H_kv=4, D=64, N=2, dtype="bf16", T_max=900, P=0)
    g, past_d, max_past = _case(w, [850, 3, 400, 777], 8103)
    out = torch.full_like(g["q"], float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvd.kvd_decode_attention_noalloc(g["q"], g["k_cache"], g["v_cache"], out, past_d, max_past, err_word=err)
    ref = _reference(w, g, past_d, max_past)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert _same_bits(out, ref)


def test_noalloc_rejects_shapes_beyond_its_scratch(c_entry):
    # 8192 sequences x 128 KV heads need more than the built-in 4 MiB.
    q = torch.zeros(64, dtype=torch.bfloat16, device=DEV)
    past = torch.zeros(8192, dtype=torch.int32, device=DEV)
    need = kvd.kvd_decode_workspace_bytes(8192, 128, 128, 128, 1, 10, "bf16")
    assert need > 4 << 20
    st = c_entry(q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), past.data_ptr(),
                 8192, 128, 128, 16, 128, 1, 10, 0.0, kvd.KVD_BF16, None, None)
    assert st == kvd.KVD_ERR_WORKSPACE
