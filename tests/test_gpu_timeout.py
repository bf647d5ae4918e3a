"""The device-side timeout path, run on purpose.

Every pipeline wait in the kernels is bounded; when one runs out the kernel
sets KVD_DEVERR_TIMEOUT in the error word, stops issuing work, waits (also
bounded) for what it already has in flight, and returns; the context stays
usable and the workspace must be zeroed again before its next use (kvd.h).
A healthy GPU never gets there.  These tests build a separate copy of the
library with KVD_TIMEOUT_TEST: its pipeline waits give up after 2 ms instead
of 2 s, and kvd_test_inject_stall(1) makes the first tile stage of every CTA
of the next launches expect 16 bytes more than its copies bring, so that
stage never completes (a wait on a flag nothing sets; no fault, nothing left
in flight).  For each kernel the tests check that the call returns with the bit
set, and that after zeroing the workspace a normal call of the same library
gives the oracle's results.
"""
import numpy as np
import pytest
import torch

import ctypes

import kv_cache_decode_append_gb300 as kvd
from kv_cache_decode_append_gb300 import build as kbuild
from kv_cache_decode_append_gb300 import kvd as binding
from kv_cache_decode_append_gb300 import workloads as wl
from helpers import TOL, row_rel_err, to_np

pytestmark = [pytest.mark.gpu, pytest.mark.timeout(900)]

DEV = "cuda"
DTYPE = {"f32": kvd.KVD_F32, "bf16": kvd.KVD_BF16}


@pytest.fixture(scope="module")
def tlib():
    import __graft_entry__
    __graft_entry__.build()
    path = kbuild.build(extra_flags=["-DKVD_TIMEOUT_TEST"], variant="timeout_test")
    lib = binding._Lib(path)
    lib.kvd_test_inject_stall.restype = None
    lib.kvd_test_inject_stall.argtypes = [ctypes.c_int]
    return lib


def _call(lib, w, g, out, past_d, max_past, ws, err, fused):
    stream = torch.cuda.current_stream().cuda_stream
    if fused:
        return lib.kvd_decode_step(g["q"].data_ptr(), g["k_cache"].data_ptr(), g["v_cache"].data_ptr(),
                                   g["k_new"].data_ptr(), g["v_new"].data_ptr(), out.data_ptr(), past_d.data_ptr(),
                                   w.B, w.H_q, w.H_kv, w.T_max, w.D, w.N, max_past, 0.0, DTYPE[w.dtype],
                                   ws.data_ptr(), ws.numel(), err.data_ptr(), stream)
    return lib.kvd_decode_attention(g["q"].data_ptr(), g["k_cache"].data_ptr(), g["v_cache"].data_ptr(),
                                    out.data_ptr(), past_d.data_ptr(), w.B, w.H_q, w.H_kv, w.T_max, w.D, w.N,
                                    max_past, 0.0, DTYPE[w.dtype], ws.data_ptr(), ws.numel(), err.data_ptr(), stream)


CASES = [  # (id, B, H_q, H_kv, D, N, T_max, past, dtype, fused, expected plan)
    ("cuda_cores_cluster", 2, 4, 4, 64, 1, 400, [300, 250], "bf16", True, {"tensor_cores": 0, "cluster": 2}),
    ("cuda_cores_small", 1, 2, 2, 64, 1, 2200, [2000], "f32", True, {"tensor_cores": 0, "cluster": 0, "early_start": 1}),
    ("cuda_cores_large", 4, 8, 8, 128, 1, 4100, [4000, 3100, 1, 2500], "f32", False, {"tensor_cores": 0, "early_start": 0}),
    ("mma_sync", 2, 8, 2, 128, 1, 800, [700, 300], "bf16", True, {"tensor_cores": 1}),
    ("tcgen05", 2, 8, 2, 128, 5, 700, [600, 130], "bf16", True, {"tensor_cores": 2}),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_timeout_returns_flagged_and_recovers(tlib, oracle_lib, case):
    name, B, H_q, H_kv, D, N, T_max, past, dtype, fused, expect = case
    w = wl.Workload(0, name, L=1, B=B, H_q=H_q, H_kv=H_kv, D=D, N=N, dtype=dtype, T_max=T_max, P=0)
    past = torch.tensor(past, dtype=torch.int32)
    max_past = int(past.max())
    plan = kvd.kvd_decode_plan(B, H_q, H_kv, D, N, max_past, w.torch_dtype)
    for k, v in expect.items():
        assert plan[k] == v, (k, plan)
    t = wl.layer_inputs(w, 0, past, device="cpu", seed_base=9900 + D + N)
    past_d = past.to(DEV)
    nbytes = tlib.kvd_decode_workspace_bytes(B, H_q, H_kv, D, N, max_past, DTYPE[dtype])
    ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)

    # 1. a stalled stage: the call returns, flagged
    g = {k: v.to(DEV) for k, v in t.items()}
    if not fused:
        kvd.kvd_append(g["k_cache"], g["v_cache"], g["k_new"], g["v_new"], past_d, max_past)
    out = torch.empty_like(g["q"])
    tlib.kvd_test_inject_stall(1)
    try:
        assert _call(tlib, w, g, out, past_d, max_past, ws, err, fused) == kvd.KVD_OK
        torch.cuda.synchronize()
    finally:
        tlib.kvd_test_inject_stall(0)
    assert int(err.item()) & kvd.KVD_DEVERR_TIMEOUT

    # 2. zero the workspace again; a normal call of the same library is exact
    assert tlib.kvd_workspace_init(ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream) == kvd.KVD_OK
    err.zero_()
    g = {k: v.to(DEV) for k, v in t.items()}
    if not fused:
        kvd.kvd_append(g["k_cache"], g["v_cache"], g["k_new"], g["v_new"], past_d, max_past)
    out = torch.full_like(g["q"], float("nan"))
    assert _call(tlib, w, g, out, past_d, max_past, ws, err, fused) == kvd.KVD_OK
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    h = {k: to_np(v) for k, v in t.items()}
    assert oracle_lib.append(h["k_cache"], h["v_cache"], h["k_new"], h["v_new"], past.numpy(), dtype) == 0
    assert np.array_equal(to_np(g["k_cache"]).view(np.uint8), h["k_cache"].view(np.uint8))
    assert np.array_equal(to_np(g["v_cache"]).view(np.uint8), h["v_cache"].view(np.uint8))
    ref, st = oracle_lib.decode_attention(h["q"], h["k_cache"], h["v_cache"], past.numpy(), dtype)
    assert st == 0
    assert row_rel_err(out.double().cpu().numpy(), ref) <= TOL[dtype]


def test_timeout_e4m3_eight_row_form(tlib, oracle_lib):
    """The same for the E4M3 fused step in the tensor-core kernel's 8-row (swapped-operand)
    form: 4 query rows per KV head, four ring stages."""
    import test_gpu_e4m3 as e8
    B, H_q, H_kv, D, N, T_max = 2, 16, 4, 128, 1, 900
    w = wl.Workload(0, "e4m3_timeout", L=1, B=B, H_q=H_q, H_kv=H_kv, D=D, N=N, dtype="bf16", T_max=T_max, P=0)
    past, t = e8._inputs(w, [850, 200], 9990)
    max_past = int(past.max())
    plan = kvd.kvd_decode_plan(B, H_q, H_kv, D, N, max_past, "e4m3")
    assert plan["tensor_cores"] == 1 and plan["rows_per_block"] == 8
    past_d = past.to(DEV)
    nbytes = tlib.kvd_decode_workspace_bytes(B, H_q, H_kv, D, N, max_past, kvd.KVD_E4M3)
    ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream

    def call(g, out):
        return tlib.kvd_decode_step_e4m3(g["q"].data_ptr(), g["k_cache"].data_ptr(), g["v_cache"].data_ptr(),
                                         g["k_new"].data_ptr(), g["v_new"].data_ptr(), out.data_ptr(),
                                         past_d.data_ptr(), B, H_q, H_kv, T_max, D, N, max_past, 0.0, e8.K_SCALE,
                                         e8.V_SCALE, ws.data_ptr(), ws.numel(), err.data_ptr(), stream)

    g = {k: v.to(DEV) for k, v in t.items()}
    out = torch.empty_like(g["q"])
    tlib.kvd_test_inject_stall(1)
    try:
        assert call(g, out) == kvd.KVD_OK
        torch.cuda.synchronize()
    finally:
        tlib.kvd_test_inject_stall(0)
    assert int(err.item()) & kvd.KVD_DEVERR_TIMEOUT

    assert tlib.kvd_workspace_init(ws.data_ptr(), ws.numel(), stream) == kvd.KVD_OK
    err.zero_()
    g = {k: v.to(DEV) for k, v in t.items()}
    out = torch.full_like(g["q"], float("nan"))
    assert call(g, out) == kvd.KVD_OK
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref, h = e8._oracle(oracle_lib, w, past, t)
    assert np.array_equal(g["k_cache"].cpu().numpy(), h["k_cache"])
    assert np.array_equal(g["v_cache"].cpu().numpy(), h["v_cache"])
    assert row_rel_err(out.double().cpu().numpy(), ref) <= TOL["bf16"]
