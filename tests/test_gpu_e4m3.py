"""E4M3 (8-bit) caches on the GPU: kvd_append_e4m3, kvd_decode_attention_e4m3 and
kvd_decode_step_e4m3 against the oracle (append bit for bit, attention within the
bf16 tolerance), the fused step bit-identical to append + attention."""
import numpy as np
import pytest
import torch

import kv_cache_decode_append_gb300 as kvd
from kv_cache_decode_append_gb300 import workloads as wl
from helpers import TOL, row_rel_err, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda"
K_SCALE, V_SCALE = 0.05, 0.02


@pytest.fixture(scope="module")
def orc():
    import __graft_entry__
    __graft_entry__.build()
    import oracle
    return oracle.load()


def _inputs(w, past, seed, device="cpu", new_dtype=torch.bfloat16):
    """bf16 q and new rows; E4M3 history codes (torch's float8 cast of N(0,1)/scale),
    NaN codes (0x7f) from slot P on."""
    past = torch.as_tensor(past, dtype=torch.int32)
    t = wl.layer_inputs(w, 0, past, device=device, seed_base=seed)
    codes = {}
    for key, sc in (("k_cache", K_SCALE), ("v_cache", V_SCALE)):
        c = (torch.nan_to_num(t.pop(key).float()) / sc).to(torch.float8_e4m3fn).view(torch.uint8)
        tail = torch.arange(w.T_max, device=device).view(1, 1, -1, 1) >= past.to(device).view(-1, 1, 1, 1)
        codes[key] = c.masked_fill(tail, 0x7F).contiguous()
    t.update(codes)
    for key in ("k_new", "v_new"):
        t[key] = t[key].to(new_dtype)
    return past, t


def _gpu(w, past, t, fused=False):
    max_past = int(past.max())
    g = {k: v.to(DEV).clone() for k, v in t.items()}
    past_d = past.to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = kvd.alloc_workspace(w.B, w.H_q, w.H_kv, w.D, w.N, max_past, "e4m3", DEV)
    out = torch.full_like(g["q"], float("nan"))
    if fused:
        kvd.kvd_decode_step_e4m3(g["q"], g["k_cache"], g["v_cache"], g["k_new"], g["v_new"], out, past_d, max_past,
                                 K_SCALE, V_SCALE, 0.0, ws, err)
    else:
        kvd.kvd_append_e4m3(g["k_cache"], g["v_cache"], g["k_new"], g["v_new"], past_d, max_past, K_SCALE, V_SCALE,
                            err)
        kvd.kvd_decode_attention_e4m3(g["q"], g["k_cache"], g["v_cache"], out, past_d, max_past, K_SCALE, V_SCALE,
                                      0.0, ws, err)
    torch.cuda.synchronize()
    return out, g, int(err.item())


def _same_bits(a, b):
    return np.array_equal(to_np(a).view(np.uint8), to_np(b).view(np.uint8))


def _oracle(orc, w, past, t):
    h = {k: (v.cpu().numpy().copy() if v.dtype == torch.uint8 else to_np(v)) for k, v in t.items()}
    nd = {torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "f32"}[t["k_new"].dtype]
    assert orc.append_e4m3(h["k_cache"], h["v_cache"], h["k_new"], h["v_new"], past.numpy(), nd, K_SCALE,
                           V_SCALE) == 0
    ref, st = orc.decode_attention_e4m3(h["q"], h["k_cache"], h["v_cache"], past.numpy(), "bf16", K_SCALE, V_SCALE)
    assert st == 0
    return ref, h


def _check(orc, w, past, seed, device="cpu", fused_too=True):
    past, t = _inputs(w, past, seed, device)
    out, g, err = _gpu(w, past, t)
    assert err == 0
    ref, h = _oracle(orc, w, past, t)
    assert np.array_equal(g["k_cache"].cpu().numpy(), h["k_cache"])
    assert np.array_equal(g["v_cache"].cpu().numpy(), h["v_cache"])
    assert row_rel_err(out.double().cpu().numpy(), ref) <= TOL["bf16"]
    if fused_too:
        out2, g2, err2 = _gpu(w, past, t, fused=True)
        assert err2 == 0
        assert _same_bits(g2["k_cache"], g["k_cache"]) and _same_bits(g2["v_cache"], g["v_cache"])
        assert _same_bits(out2, out)


# (B, H_q, H_kv, D, N, T_max, past)
E4M3_CASES = [
    (8, 12, 12, 64, 1, 1024, [1023, 0, 512, 1, 64, 900, 333, 1000]),  # GPT-2 shapes, batch 8
    (4, 32, 8, 128, 1, 3000, [2999, 17, 1500, 2048]),                 # GQA 4 rows, ragged
    (3, 16, 2, 128, 1, 900, [899, 450, 0]),                           # 8 rows: two row blocks of 4
    (2, 8, 2, 64, 5, 700, [63, 600]),                                 # chunk of 5 across a tile
    (1, 4, 4, 128, 3, 3, [0]),                                        # empty history, P + N = T_max
    (2, 14, 2, 128, 1, 1500, [1499, 700]),                            # 7 rows (8-row form, one padding row)
    (3, 8, 4, 128, 3, 700, [650, 64, 0]),                             # 6 rows: chunk of 3, per-row limits
    (2, 8, 8, 128, 1, 1000, [999, 500]),                              # 1 row per KV head
]


@pytest.mark.parametrize("case", E4M3_CASES, ids=[f"e4m3_{i}" for i in range(len(E4M3_CASES))])
def test_e4m3_parity(orc, case):
    B, H_q, H_kv, D, N, T_max, past = case
    w = wl.Workload(0, "e4m3", L=1, B=B, H_q=H_q, H_kv=H_kv, D=D, N=N, dtype="bf16", T_max=T_max, P=0)
    _check(orc, w, past, seed=9600 + D + N)


@pytest.mark.parametrize("new_dtype", [torch.float32, torch.float16], ids=["f32", "f16"])
def test_e4m3_append_other_input_types(orc, new_dtype):
    w = wl.Workload(0, "e4m3a", L=1, B=2, H_q=4, H_kv=2, D=128, N=3, dtype="bf16", T_max=300, P=0)
    past, t = _inputs(w, [17, 290], 9700, new_dtype=new_dtype)
    t["k_new"] = t["k_new"] * 40  # some quotients beyond 448: saturation
    _, g, err = _gpu(w, past, t)
    assert err == 0
    _, h = _oracle(orc, w, past, t)
    assert np.array_equal(g["k_cache"].cpu().numpy(), h["k_cache"])
    assert np.array_equal(g["v_cache"].cpu().numpy(), h["v_cache"])
    assert (h["k_cache"][:, :, 17:20] & 0x7F == 0x7E).any()  # saturated codes were exercised


# (4 and 8 rows per KV head: the 8-row form)
@pytest.mark.parametrize("case", [(16, 32, 8, 128, 12300, 12200, 2), (16, 32, 8, 128, 1100, 1000, 1),
                                  (16, 64, 8, 128, 12300, 12200, 2)],
                         ids=["merge_pass", "in_kernel", "merge_pass_8rows"])
def test_e4m3_merge_modes(orc, case):
    B, H_q, H_kv, D, T_max, max_past, launches = case
    plan = kvd.kvd_decode_plan(B, H_q, H_kv, D, 1, max_past, "e4m3")
    assert plan["launches"] == launches and plan["rows_per_block"] == 8
    gen = torch.Generator().manual_seed(9800 + launches)
    past = torch.randint(0, max_past + 1, (B,), generator=gen, dtype=torch.int32)
    past[2] = max_past
    w = wl.Workload(0, "e4m3m", L=1, B=B, H_q=H_q, H_kv=H_kv, D=D, N=1, dtype="bf16", T_max=T_max, P=0)
    _check(orc, w, past, seed=9810 + launches)


# More than 16 query rows per KV head: several 16-row tensor-core blocks per head.
# (B, H_q, H_kv, D, N, T_max, past)
E4M3_MANY_ROWS_CASES = [
    (2, 32, 8, 128, 8, 1100, [1000, 63]),                             # 32 rows, ragged tails
    (3, 32, 2, 128, 10, 800, [700, 0, 129]),                          # 160 rows: two row blocks
    (1, 32, 8, 128, 32, 300, [200]),                                  # 128 rows, a chunk of 32 across tiles
]


@pytest.mark.parametrize("case", E4M3_MANY_ROWS_CASES, ids=[f"e4m3_rows_{i}" for i in range(len(E4M3_MANY_ROWS_CASES))])
def test_e4m3_many_rows_parity(orc, case):
    B, H_q, H_kv, D, N, T_max, past = case
    assert kvd.kvd_decode_plan(B, H_q, H_kv, D, N, max(past), "e4m3")["tensor_cores"] == 1
    w = wl.Workload(0, "e4m3t", L=1, B=B, H_q=H_q, H_kv=H_kv, D=D, N=N, dtype="bf16", T_max=T_max, P=0)
    _check(orc, w, past, seed=9650 + N)


@pytest.mark.parametrize("case", [(16, 32, 8, 128, 9300, 9200, 2), (16, 32, 8, 128, 1100, 1000, 1)],
                         ids=["merge_pass", "in_kernel"])
def test_e4m3_many_rows_merge_modes(orc, case):
    B, H_q, H_kv, D, T_max, max_past, launches = case
    plan = kvd.kvd_decode_plan(B, H_q, H_kv, D, 8, max_past, "e4m3")
    assert plan["tensor_cores"] == 1 and plan["launches"] == launches
    gen = torch.Generator().manual_seed(9830 + launches)
    past = torch.randint(0, max_past + 1, (B,), generator=gen, dtype=torch.int32)
    past[5] = max_past
    w = wl.Workload(0, "e4m3tm", L=1, B=B, H_q=H_q, H_kv=H_kv, D=D, N=8, dtype="bf16", T_max=T_max, P=0)
    _check(orc, w, past, seed=9840 + launches)


def _gpu_attention(w, past, t):
    """kvd_decode_attention_e4m3 alone over the given caches (no append)."""
    g = {k: v.to(DEV) for k, v in t.items()}
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = kvd.alloc_workspace(w.B, w.H_q, w.H_kv, w.D, w.N, int(past.max()), "e4m3", DEV)
    out = torch.full_like(g["q"], float("nan"))
    kvd.kvd_decode_attention_e4m3(g["q"], g["k_cache"], g["v_cache"], out, past.to(DEV), int(past.max()), K_SCALE,
                                  V_SCALE, 0.0, ws, err)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), int(err.item())


def _oracle_attention(orc, t, past):
    h = {k: (v.cpu().numpy().copy() if v.dtype == torch.uint8 else to_np(v)) for k, v in t.items()}
    ref, st = orc.decode_attention_e4m3(h["q"], h["k_cache"], h["v_cache"], past.numpy(), "bf16", K_SCALE, V_SCALE)
    assert st == 0
    return ref


# (H_q, N): 32 rows per KV head (16-row blocks), 8 rows (the 8-row form)
TWO_FORMS = [(32, 8), (16, 4)]


@pytest.mark.parametrize("hq_n", TWO_FORMS, ids=["rows32", "rows8"])
def test_e4m3_subnormal_codes(orc, hq_n):
    """Caches of zero and subnormal codes only (|x| = m * 2^-9): the widening keeps them
    exactly (a flush to zero would zero the output)."""
    H_q, N = hq_n
    w = wl.Workload(0, "e4m3s", L=1, B=2, H_q=H_q, H_kv=8, D=128, N=N, dtype="bf16", T_max=400, P=0)
    past = torch.tensor([300, 57], dtype=torch.int32)
    t = wl.layer_inputs(w, 0, past, device="cpu", seed_base=9870)
    gen = torch.Generator().manual_seed(9871)
    for key in ("k_cache", "v_cache"):
        mag = torch.randint(0, 8, t[key].shape, generator=gen, dtype=torch.int32)
        sign = torch.randint(0, 2, t[key].shape, generator=gen, dtype=torch.int32) * 0x80
        t[key] = (mag | sign).to(torch.uint8)
    # (every slot holds a code: the chunk's rows P .. P+N-1 included)
    out, err = _gpu_attention(w, past, t)
    assert err == 0
    ref = _oracle_attention(orc, t, past)
    assert np.abs(ref).max() > 0
    assert row_rel_err(out, ref) <= TOL["bf16"]


@pytest.mark.parametrize("hq_n", TWO_FORMS, ids=["rows32", "rows8"])
def test_e4m3_nan_codes(orc, hq_n):
    """A NaN code among the keys makes exactly the rows that see it NaN, as in the oracle (a
    masked key's score is replaced, not multiplied); a NaN value code seen by every row of its
    head makes that column NaN.  (A non-finite value at a key masked for some rows of the
    chunk reaches them too: the zero weight times NaN in the P . V product is NaN.)"""
    H_q, N = hq_n
    g = H_q // 8
    w = wl.Workload(0, "e4m3n", L=1, B=2, H_q=H_q, H_kv=8, D=128, N=N, dtype="bf16", T_max=400, P=0)
    past = torch.tensor([300, 120], dtype=torch.int32)
    _, t = _inputs(w, past + w.N, 9880)      # valid codes up to P + N (the chunk's rows), NaN codes after
    t["k_cache"][0, 1, 200, 5] = 0x7F        # every row of (b 0, h 1) sees key 200
    t["k_cache"][1, 5, 121, 7] = 0xFF        # rows of (b 1, h 5) from the second new token on see key P + 1
    t["v_cache"][1, 3, 100, 64] = 0x7F       # every row of (b 1, h 3) sees value row 100
    out, err = _gpu_attention(w, past, t)
    assert err == 0
    ref = _oracle_attention(orc, t, past)
    assert np.array_equal(np.isnan(out), np.isnan(ref))
    rows = np.isnan(ref).any(axis=-1)
    assert rows[0, g:2 * g].all() and rows[1, 3 * g:4 * g].all()
    # (row i of the chunk sees key P + i)
    assert rows[1, 5 * g:6 * g].sum() == g * (N - 1) and not rows[1, 5 * g:6 * g, 0].any()
    fin = ~np.isnan(ref).any(axis=-1)
    assert row_rel_err(out[fin], ref[fin]) <= TOL["bf16"]


def test_e4m3_kernel_choice():
    """E4M3 caches stay on mma.sync at every row count (D = 128), CUDA cores at D = 64; heads
    of at most 8 rows in the 8-row (swapped) form."""
    def plan(*a):
        p = kvd.kvd_decode_plan(*a, 1000, "e4m3")
        return p["tensor_cores"], p["rows_per_block"]
    assert plan(4, 32, 8, 128, 4) == (1, 16)   # 16 rows
    assert plan(4, 17, 1, 128, 1) == (1, 16)   # 17 rows
    assert plan(4, 9, 1, 128, 1) == (1, 16)    # 9 rows
    assert plan(4, 32, 8, 128, 2) == (1, 8)    # 8 rows
    assert plan(4, 32, 8, 128, 1) == (1, 8)    # 4 rows
    assert plan(4, 8, 8, 128, 1) == (1, 8)     # 1 row
    assert plan(4, 32, 1, 64, 1)[0] == 0       # D = 64


def test_e4m3_gqa_longctx_chunk8_full_size(orc):
    """The long-context workload at full size with an E4M3 cache and 8 new tokens (32 rows per
    KV head), in the launch configuration bench.py --cache e4m3 --n-new 8 times."""
    w = wl.with_n(wl.WORKLOADS["gqa_longctx_b32_bf16"], 8)
    assert kvd.kvd_decode_plan(w.B, w.H_q, w.H_kv, w.D, w.N, max(wl.past_lens(w).tolist()), "e4m3")["tensor_cores"] == 1
    _check(orc, w, wl.past_lens(w), seed=9910, device=DEV)


def test_e4m3_gqa_longctx_full_size(orc):
    """The long-context workload's shapes and lengths at full size with an E4M3 cache."""
    w = wl.WORKLOADS["gqa_longctx_b32_bf16"]
    _check(orc, w, wl.past_lens(w), seed=9900, device=DEV)


def test_e4m3_rejects_misuse():
    q = torch.zeros((1, 4, 1, 64), dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros((1, 2, 16, 64), dtype=torch.uint8, device=DEV)
    past = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = kvd.alloc_workspace(1, 4, 2, 64, 1, 8, "e4m3", DEV)
    with pytest.raises(kvd.KvdError) as e:  # a scale must be positive
        kvd.kvd_decode_attention_e4m3(q, kc, kc, torch.empty_like(q), past, 8, 0.0, 1.0, 0.0, ws)
    assert e.value.status == kvd.KVD_ERR_INVALID_ARG
    assert kvd.raw.kvd_decode_attention(q.data_ptr(), kc.data_ptr(), kc.data_ptr(), q.data_ptr(), past.data_ptr(),
                                        1, 4, 2, 16, 64, 1, 8, 0.0, kvd.KVD_E4M3, ws.data_ptr(), ws.numel(), None,
                                        None) == kvd.KVD_ERR_UNSUPPORTED
