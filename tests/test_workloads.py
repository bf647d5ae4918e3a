"""The seeded synthetic workloads (CPU): reproducible draws, the recipe's rounding and
tail fill, and room in every cache for the history plus the new rows at each swept N."""
import pytest
import torch

from kv_cache_decode_append_gb300 import workloads as wl

# N values the measurements sweep: the workload's own, the chunked-decode sweep, and the
# long-context runs with 8 / 16 / 32 new tokens (32 / 64 / 128 query rows per KV head).
SWEEP = {name: sorted({w.N, *(wl.CHUNKED_N if w.name.startswith("gpt2s_chunked") else ()),
                       *((4, 8, 16, 32) if w.name.startswith("gqa") else ())})
         for name, w in wl.WORKLOADS.items()}


@pytest.mark.parametrize("name", sorted(wl.WORKLOADS))
def test_history_and_new_rows_fit(name):
    w = wl.WORKLOADS[name]
    past = wl.past_lens(w)
    assert past.dtype == torch.int32 and past.shape == (w.B,)
    if w.P is not None:
        assert (past == w.P).all()
    else:
        lo, hi = w.P_range
        assert int(past.min()) >= lo and int(past.max()) <= hi
    for N in SWEEP[name]:
        assert int(past.max()) + N <= w.T_max, (name, N)
        assert w.group * N <= 1024  # query rows per KV head the library accepts


def test_long_context_lengths_are_spread_and_reproducible():
    w = wl.WORKLOADS["gqa_longctx_b32_bf16"]
    a, b = wl.past_lens(w), wl.past_lens(w)
    assert torch.equal(a, b)
    assert len(set(a.tolist())) > w.B // 2            # distinct per-sequence lengths, not one value
    assert int(a.max()) - int(a.min()) > 2048


def test_draws_follow_the_recipe():
    """bf16 inputs are the fp32 N(0,1) draws rounded to nearest even; same seed, same bits;
    another layer, other bits; slots at or past P_b hold the tail fill."""
    w32 = wl.WORKLOADS["gpt2s_chunked_p512_f32"]
    w16 = wl.Workload(w32.wid, "bf16 twin", L=w32.L, B=w32.B, H_q=w32.H_q, H_kv=w32.H_kv, D=w32.D, N=w32.N,
                      dtype="bf16", T_max=w32.T_max, P=w32.P)
    past = wl.past_lens(w32)
    f = wl.layer_inputs(w32, 3, past)
    h = wl.layer_inputs(w16, 3, past)
    for key in ("q", "k_new", "v_new"):
        assert torch.equal(h[key], f[key].to(torch.bfloat16))
    assert torch.equal(wl.layer_inputs(w32, 3, past)["q"], f["q"])
    assert not torch.equal(wl.layer_inputs(w32, 4, past)["q"], f["q"])
    P = w32.P
    for key in ("k_cache", "v_cache"):
        assert torch.isfinite(f[key][:, :, :P]).all()
        assert torch.isnan(f[key][:, :, P:]).all()
    z = wl.layer_inputs(w32, 3, past, tail_fill="zero")
    assert (z["k_cache"][:, :, P:] == 0).all() and torch.equal(z["k_cache"][:, :, :P], f["k_cache"][:, :, :P])
    # the five streams of a layer are distinct draws
    assert not torch.equal(f["k_cache"][:, :, :P], f["v_cache"][:, :, :P])
    # N(0, 1): loose moments over the 393,216 cached K values of one layer
    x = f["k_cache"][:, :, :P].double()
    assert abs(float(x.mean())) < 0.01 and abs(float(x.std()) - 1.0) < 0.01
