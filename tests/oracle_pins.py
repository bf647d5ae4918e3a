"""Pins for the CPU oracle: facts fixed by the pages and by mathematics.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises ``AssertionError`` when the
oracle disagrees with something other than itself:

* printed values   -- the KV-cache size table (golden file);
* library routines -- ``torch.cat`` for the cache update, and
  ``torch.nn.functional.scaled_dot_product_attention`` (float64, square causal
  mask, ``enable_gqa``) for the uncached full-recompute route;
* closed forms     -- one visible key gives exactly its value row; identical
  keys give the mean of the visible value rows; a dominant key gives its value
  row;
* invariants       -- the pages' trap: with one new token a joint permutation
  of cached (K, V) pairs leaves the output unchanged, with several new tokens a
  reversed old/new order changes it;
* paged cache      -- with pages laid out from a contiguous cache and the
  identity block table, paged append and paged attention give exactly the
  contiguous results (pinned above); renumbering the physical pages (and
  adding unused NaN pages) changes nothing; a needed page outside the pool is
  reported and only its sequence is affected.

``test_oracle_pins.py`` runs them on the real oracle and on mutants of it with
one planted mistake each, to show that every plausible mistake fails a pin.
"""
from __future__ import annotations

import os

import numpy as np
import torch
import torch.nn.functional as F

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
_UNITS = {"B": 1, "KiB": 1024, "MiB": 1024 ** 2}


# ---------------------------------------------------------------------------------
# helpers (no attention arithmetic here: inputs and conversions only)
_TORCH = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def _rand(shape, seed, dtype):
    g = torch.Generator("cpu").manual_seed(seed)
    t = torch.randn(shape, generator=g, dtype=torch.float32)
    return t.to(_TORCH[dtype])


def to_np(t: torch.Tensor) -> np.ndarray:
    """Oracle representation: float32, or uint16 raw bits for bf16."""
    t = t.contiguous()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def to_f64(t: torch.Tensor) -> torch.Tensor:
    return t.to(torch.float64)


def _appended(k_cache, v_cache, k_new, v_new, past_len):
    """Caches after the update, built with torch.cat on the sequence axis."""
    kc, vc = k_cache.clone(), v_cache.clone()
    N = k_new.shape[2]
    for b, P in enumerate(past_len.tolist()):
        kc[b, :, : P + N] = torch.cat([k_cache[b, :, :P], k_new[b]], dim=1)
        vc[b, :, : P + N] = torch.cat([v_cache[b, :, :P], v_new[b]], dim=1)
    return kc, vc


def _problem(B, H_q, H_kv, D, N, T_max, past, dtype, seed):
    q = _rand((B, H_q, N, D), seed, dtype)
    k_new = _rand((B, H_kv, N, D), seed + 1, dtype)
    v_new = _rand((B, H_kv, N, D), seed + 2, dtype)
    k_cache = _rand((B, H_kv, T_max, D), seed + 3, dtype)
    v_cache = _rand((B, H_kv, T_max, D), seed + 4, dtype)
    past_len = torch.tensor(past, dtype=torch.int32)
    for b, P in enumerate(past):  # slots past the history hold NaN
        k_cache[b, :, P:] = float("nan")
        v_cache[b, :, P:] = float("nan")
    return q, k_new, v_new, k_cache, v_cache, past_len


def _oracle_decode(orc, q, k_cache, v_cache, past_len, dtype, scale=None):
    out, st = orc.decode_attention(to_np(q), to_np(k_cache), to_np(v_cache),
                                   past_len.numpy(), dtype, scale)
    assert st == 0, f"oracle status {st}"
    return torch.from_numpy(out)


def _max_rel(a: torch.Tensor, b: torch.Tensor) -> float:
    """Row-normwise relative error of ``a`` against ``b`` over the last axis."""
    num = (a - b).abs().amax(dim=-1)
    den = b.abs().amax(dim=-1).clamp_min(1e-300)
    return float((num / den).max())


# ---------------------------------------------------------------------------------
def pin_cache_bytes(orc):
    """The size formula reproduces every value the page prints."""
    with open(os.path.join(GOLDEN, "kv_cache_bytes.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 9
    for L, B, H, D, T, s, expected, unit, match in rows:
        got = orc.cache_bytes(int(L), int(B), int(H), int(D), int(T), int(s)) / _UNITS[unit]
        if match == "exact":
            assert got == float(expected), (L, B, H, D, T, s, got, expected)
        else:
            decimals = len(expected.split(".")[1])
            assert round(got, decimals) == float(expected), (got, expected)


def pin_append_is_concat(orc):
    """Cache update = concat of history and new tokens on the sequence axis, in place."""
    for dtype in ("f32", "bf16"):
        B, H, T_max, D, N = 3, 2, 11, 8, 3
        past = [4, 0, T_max - N]
        _, k_new, v_new, k_cache, v_cache, past_len = _problem(B, H, H, D, N, T_max, past, dtype, 7)
        # sentinel: slots past P+N keep arbitrary recognisable values
        k_cache[:, :, :] = torch.where(torch.isnan(k_cache), torch.full_like(k_cache, -3.25), k_cache)
        v_cache[:, :, :] = torch.where(torch.isnan(v_cache), torch.full_like(v_cache, 5.5), v_cache)
        exp_k, exp_v = _appended(k_cache, v_cache, k_new, v_new, past_len)
        kc, vc = to_np(k_cache), to_np(v_cache)
        st = orc.append(kc, vc, to_np(k_new), to_np(v_new), past_len.numpy(), dtype)
        assert st == 0
        assert np.array_equal(kc.view(np.uint8), to_np(exp_k).view(np.uint8))
        assert np.array_equal(vc.view(np.uint8), to_np(exp_v).view(np.uint8))
        # capacity: P + N > T_max must leave that sequence untouched and report it
        bad = torch.tensor([T_max - N + 1, 0, 2], dtype=torch.int32)
        kc2, vc2 = to_np(k_cache), to_np(v_cache)
        st = orc.append(kc2, vc2, to_np(k_new), to_np(v_new), bad.numpy(), dtype)
        assert st == 2
        assert np.array_equal(kc2[0], to_np(k_cache)[0])
        assert np.array_equal(vc2[0], to_np(v_cache)[0])
        assert not np.array_equal(kc2[1], to_np(k_cache)[1])


def pin_single_visible_key(orc):
    """Empty history, one new token: the only visible key has weight 1, out = v_new.

    Runs over every bf16 bit pattern as a value, so the bf16 widening is pinned
    against torch's own conversion (NaN stays NaN, infinities stay infinite).
    """
    D = 1 << 16
    v_bits = torch.arange(D, dtype=torch.int32).to(torch.int16).view(1, 1, 1, D)
    v_new = v_bits.view(torch.bfloat16).clone()
    q = torch.zeros((1, 1, 1, D), dtype=torch.bfloat16)
    k_new = torch.zeros_like(q)
    k_cache = torch.zeros((1, 1, 2, D), dtype=torch.bfloat16)
    v_cache = torch.zeros_like(k_cache)
    past_len = torch.tensor([0], dtype=torch.int32)
    kc, vc = _appended(k_cache, v_cache, k_new, v_new, past_len)
    out = _oracle_decode(orc, q, kc, vc, past_len, "bf16")
    want = to_f64(v_new)
    assert torch.equal(torch.isnan(out), torch.isnan(want))
    fin = ~torch.isnan(want)
    assert torch.equal(out[fin], want[fin])
    for dtype in ("f32", "bf16", "f16"):
        q, k_new, v_new, k_cache, v_cache, past_len = _problem(2, 4, 2, 16, 1, 5, [0, 0], dtype, 11)
        kc, vc = _appended(k_cache, v_cache, k_new, v_new, past_len)
        out = _oracle_decode(orc, q, kc, vc, past_len, dtype)
        want = to_f64(v_new).repeat_interleave(2, dim=1)
        assert torch.equal(out, want)


def pin_widening_all_patterns(orc):
    """Every bf16 and fp16 bit pattern widens to the value torch's own conversion gives."""
    bits = torch.arange(1 << 16, dtype=torch.int32).to(torch.int16)
    for dtype, tdt in (("bf16", torch.bfloat16), ("f16", torch.float16)):
        vals = bits.view(tdt)
        got = orc.widen(to_np(vals), dtype)
        want = vals.to(torch.float64).numpy()
        assert np.array_equal(np.isnan(got), np.isnan(want))
        fin = ~np.isnan(want)
        assert np.array_equal(got[fin], want[fin])


def pin_identical_keys_mean(orc):
    """All keys equal: equal weights, so row i is the mean of the P+i+1 visible value rows."""
    for dtype in ("f32", "bf16", "f16"):
        B, H_q, H_kv, D, N, T_max = 2, 4, 2, 8, 4, 16
        past = [5, 9]
        q, k_new, v_new, k_cache, v_cache, past_len = _problem(B, H_q, H_kv, D, N, T_max, past, dtype, 21)
        key = _rand((D,), 99, dtype)
        k_cache[:] = key
        k_new[:] = key
        kc, vc = _appended(k_cache, v_cache, k_new, v_new, past_len)
        out = _oracle_decode(orc, q, kc, vc, past_len, dtype)
        vf = to_f64(vc)
        for b, P in enumerate(past):
            for hq in range(H_q):
                for i in range(N):
                    want = vf[b, hq // (H_q // H_kv), : P + i + 1].mean(dim=0)
                    assert _max_rel(out[b, hq, i], want) < 1e-13


def pin_dominant_key(orc):
    """One key aligned with q far above the rest: softmax puts all weight on it."""
    D, T_max = 16, 12
    for dtype in ("f32", "bf16", "f16"):
        q, k_new, v_new, k_cache, v_cache, past_len = _problem(1, 2, 1, D, 2, T_max, [7], dtype, 31)
        q[:] = _rand((D,), 5, dtype)
        for j in (0, 3, 6):  # history positions, visible to both new rows
            kc, vc = _appended(k_cache, v_cache, k_new, v_new, past_len)
            kc[0, 0, :9] = 0.01 * _rand((9, D), 40 + j, "f32").to(kc.dtype)
            kc[0, 0, j] = (q[0, 0, 0].float() * 64.0).to(kc.dtype)  # score ~ 64*|q|^2/4
            out = _oracle_decode(orc, q, kc, vc, past_len, dtype)
            want = to_f64(vc[0, 0, j])
            for hq in range(2):
                for i in range(2):
                    assert _max_rel(out[0, hq, i], want) < 1e-9, (dtype, j, hq, i)


def _route_b_sdpa(q, k_new, v_new, k_cache, v_cache, past_len, scale, seed):
    """Uncached route: full causal attention over the concatenated sequence, last N rows.

    The first P query rows are random and discarded; keys/values are
    ``torch.cat([history, new])``; the square causal mask comes from SDPA.
    """
    B, H_q, N, D = q.shape
    H_kv = k_new.shape[1]
    outs = []
    for b, P in enumerate(past_len.tolist()):
        qf = torch.cat([to_f64(_rand((H_q, P, D), seed + b, "f32")), to_f64(q[b])], dim=1)
        kf = torch.cat([to_f64(k_cache[b, :, :P]), to_f64(k_new[b])], dim=1)
        vf = torch.cat([to_f64(v_cache[b, :, :P]), to_f64(v_new[b])], dim=1)
        o = F.scaled_dot_product_attention(qf[None], kf[None], vf[None], is_causal=True,
                                           scale=scale, enable_gqa=H_q != H_kv)[0]
        outs.append(o[:, P:])
    return torch.stack(outs)


_ROUTE_CASES = [
    # B, H_q, H_kv, D, N, T_max, past, dtype, scale
    (1, 12, 12, 64, 1, 64, [16], "f32", None),
    (2, 4, 4, 64, 4, 40, [0, 13], "f32", None),
    (2, 8, 2, 128, 3, 33, [30, 7], "bf16", None),
    (3, 8, 1, 64, 16, 48, [32, 0, 5], "bf16", 0.3),
    (1, 6, 3, 128, 5, 21, [16], "f32", 1.7),
    (2, 8, 4, 64, 2, 24, [9, 21], "f16", None),
]


def pin_route_b_sdpa(orc):
    """Cached chunked decode = last N rows of uncached full causal attention (library SDPA)."""
    for n, (B, H_q, H_kv, D, N, T_max, past, dtype, scale) in enumerate(_ROUTE_CASES):
        q, k_new, v_new, k_cache, v_cache, past_len = _problem(B, H_q, H_kv, D, N, T_max, past, dtype, 100 + n)
        kc, vc = _appended(k_cache, v_cache, k_new, v_new, past_len)
        out = _oracle_decode(orc, q, kc, vc, past_len, dtype, scale)
        want = _route_b_sdpa(q, k_new, v_new, k_cache, v_cache, past_len,
                             scale if scale is not None else 1.0 / D ** 0.5, 500 + n)
        assert _max_rel(out, want) < 1e-12, (n, _max_rel(out, want))


def pin_full_causal_sdpa(orc):
    """The oracle's own uncached route agrees with library causal attention."""
    for T, D, scale in ((1, 8, 0.5), (17, 64, 0.125), (40, 128, 1.0 / 128 ** 0.5)):
        qf, kf, vf = (to_f64(_rand((T, D), 600 + s, "f32")) for s in range(3))
        got = torch.from_numpy(orc.full_causal_attention(qf.numpy(), kf.numpy(), vf.numpy(), scale))
        want = F.scaled_dot_product_attention(qf[None], kf[None], vf[None], is_causal=True, scale=scale)[0]
        assert _max_rel(got, want) < 1e-12


def pin_permutation_single_token(orc):
    """N = 1: jointly permuting the (K, V) pairs of all visible slots changes nothing."""
    for dtype in ("f32", "bf16"):
        P, D = 23, 64
        q, k_new, v_new, k_cache, v_cache, past_len = _problem(1, 4, 2, D, 1, 32, [P], dtype, 41)
        kc, vc = _appended(k_cache, v_cache, k_new, v_new, past_len)
        base = _oracle_decode(orc, q, kc, vc, past_len, dtype)
        perm = torch.randperm(P + 1, generator=torch.Generator().manual_seed(3))
        kp, vp = kc.clone(), vc.clone()
        kp[:, :, : P + 1] = kc[:, :, perm]
        vp[:, :, : P + 1] = vc[:, :, perm]
        out = _oracle_decode(orc, q, kp, vp, past_len, dtype)
        assert _max_rel(out, base) < 1e-13


def pin_reversed_order_trap(orc):
    """The concat-order trap: new||old hides for N = 1 and shows for N > 1."""
    for dtype in ("f32", "bf16"):
        for N, must_differ in ((1, False), (4, True)):
            P, D = 12, 64
            q, k_new, v_new, k_cache, v_cache, past_len = _problem(1, 2, 2, D, N, 24, [P], dtype, 51)
            kc, vc = _appended(k_cache, v_cache, k_new, v_new, past_len)
            good = _oracle_decode(orc, q, kc, vc, past_len, dtype)
            kr, vr = kc.clone(), vc.clone()
            kr[0, :, : P + N] = torch.cat([k_new[0], k_cache[0, :, :P]], dim=1)
            vr[0, :, : P + N] = torch.cat([v_new[0], v_cache[0, :, :P]], dim=1)
            rev = _oracle_decode(orc, q, kr, vr, past_len, dtype)
            err = _max_rel(rev, good)
            if must_differ:
                assert err > 1e-2, err
            else:
                assert err < 1e-13, err


# ---------------------------------------------------------------------------------
# paged cache: pages [num_pages, H_kv, page_size, D]; logical page j of sequence b
# is physical page block_table[b, j]
def _to_pages(cache: torch.Tensor, page_size: int) -> torch.Tensor:
    """Pages of a contiguous [B, H, T, D] cache, sequence b's page j at index b * (T / page_size) + j."""
    B, H, T, D = cache.shape
    assert T % page_size == 0
    return cache.reshape(B, H, T // page_size, page_size, D).permute(0, 2, 1, 3, 4).reshape(
        B * (T // page_size), H, page_size, D).contiguous()


def _identity_table(B: int, max_pages: int) -> np.ndarray:
    return np.arange(B * max_pages, dtype=np.int32).reshape(B, max_pages)


def pin_paged_identity_layout(orc):
    """Identity block table: paged append / attention = contiguous append / attention, bit for bit."""
    for dtype, ps in (("f32", 4), ("bf16", 8)):
        B, H_q, H_kv, D, N, T_max = 3, 4, 2, 16, 3, 32
        past = [5, 0, T_max - N]
        q, k_new, v_new, k_cache, v_cache, past_len = _problem(B, H_q, H_kv, D, N, T_max, past, dtype, 71)
        k_cache = torch.where(torch.isnan(k_cache), torch.full_like(k_cache, 1.75), k_cache)
        v_cache = torch.where(torch.isnan(v_cache), torch.full_like(v_cache, -0.5), v_cache)
        table = _identity_table(B, T_max // ps)
        kp, vp = to_np(_to_pages(k_cache, ps)), to_np(_to_pages(v_cache, ps))
        st = orc.paged_append(kp, vp, to_np(k_new), to_np(v_new), table, past_len.numpy(), dtype)
        assert st == 0
        exp_k, exp_v = _appended(k_cache, v_cache, k_new, v_new, past_len)
        assert np.array_equal(kp.view(np.uint8), to_np(_to_pages(exp_k, ps)).view(np.uint8))
        assert np.array_equal(vp.view(np.uint8), to_np(_to_pages(exp_v, ps)).view(np.uint8))
        paged, st = orc.paged_decode_attention(to_np(q), kp, vp, table, past_len.numpy(), dtype)
        assert st == 0
        flat = _oracle_decode(orc, q, exp_k, exp_v, past_len, dtype).numpy()
        assert np.array_equal(paged, flat)


def pin_paged_renumbered_pages(orc):
    """Renumbering the physical pages and adding unused NaN pages changes nothing."""
    for dtype, ps in (("f32", 8), ("bf16", 4)):
        B, H_q, H_kv, D, N, T_max = 2, 6, 3, 8, 2, 24
        q, k_new, v_new, k_cache, v_cache, past_len = _problem(B, H_q, H_kv, D, N, T_max, [9, 20], dtype, 81)
        kc, vc = _appended(k_cache, v_cache, k_new, v_new, past_len)
        kp, vp = _to_pages(kc, ps), _to_pages(vc, ps)
        table = _identity_table(B, T_max // ps)
        base, st = orc.paged_decode_attention(to_np(q), to_np(kp), to_np(vp), table, past_len.numpy(), dtype)
        assert st == 0
        n_used, n_pool = kp.shape[0], kp.shape[0] + 5
        perm = torch.randperm(n_pool, generator=torch.Generator().manual_seed(5))[:n_used]
        kp2 = torch.full((n_pool,) + tuple(kp.shape[1:]), float("nan"), dtype=kp.dtype)
        vp2 = torch.full_like(kp2, float("nan"))
        kp2[perm], vp2[perm] = kp, vp
        table2 = perm.numpy().astype(np.int32)[table]
        out, st = orc.paged_decode_attention(to_np(q), to_np(kp2), to_np(vp2), table2, past_len.numpy(), dtype)
        assert st == 0
        assert np.array_equal(out, base)


def pin_paged_bad_page(orc):
    """A needed block-table entry outside the pool is reported; other sequences are unaffected."""
    dtype, ps = "f32", 4
    B, H_q, H_kv, D, N, T_max = 2, 2, 2, 8, 1, 16
    q, k_new, v_new, k_cache, v_cache, past_len = _problem(B, H_q, H_kv, D, N, T_max, [6, 6], dtype, 91)
    kc, vc = _appended(k_cache, v_cache, k_new, v_new, past_len)
    kp, vp = to_np(_to_pages(kc, ps)), to_np(_to_pages(vc, ps))
    table = _identity_table(B, T_max // ps)
    table[0, 3] = -1                       # not needed (tokens 0..6 use pages 0, 1): fine
    good, st = orc.paged_decode_attention(to_np(q), kp, vp, table, past_len.numpy(), dtype)
    assert st == 0 and np.isfinite(good).all()
    table[1, 1] = kp.shape[0]              # needed by sequence 1: out of the pool
    out, st = orc.paged_decode_attention(to_np(q), kp, vp, table, past_len.numpy(), dtype)
    assert st == 3
    assert np.array_equal(out[0], good[0]) and np.isnan(out[1]).all()
    kp2 = kp.copy()
    st = orc.paged_append(kp2, vp.copy(), to_np(k_new), to_np(v_new), table, past_len.numpy(), dtype)
    assert st == 3
    assert np.array_equal(kp2[4:].view(np.uint8), kp[4:].view(np.uint8))  # sequence 1 untouched


# ---------------------------------------------------------------------------------
# E4M3 cache
def _e4m3_values() -> torch.Tensor:
    """All 256 E4M3 codes as torch float8_e4m3fn values."""
    return torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)


def pin_e4m3_decode_all_codes(orc):
    """Every E4M3 code decodes to the value torch's float8_e4m3fn conversion gives."""
    vals = _e4m3_values()
    got = orc.widen(vals.view(torch.uint8).numpy().copy(), "e4m3")
    want = vals.to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    fin = ~np.isnan(want)
    assert np.array_equal(got[fin], want[fin])
    assert np.nanmax(np.abs(got)) == 448.0


def pin_e4m3_quantize(orc):
    """Quantization = torch's round-to-nearest-even float8_e4m3fn cast inside +-448
    (random values, every exact midpoint between neighbouring codes and its two
    float32 neighbours, subnormals, signed zeros); saturation to +-448 beyond."""
    vals = _e4m3_values().to(torch.float64)
    fin = vals[~torch.isnan(vals)]
    pos = torch.sort(torch.unique(fin[fin >= 0])).values
    mids = ((pos[1:] + pos[:-1]) / 2).to(torch.float32)
    up = torch.nextafter(mids, torch.full_like(mids, float("inf")))
    dn = torch.nextafter(mids, torch.full_like(mids, -float("inf")))
    g = torch.Generator().manual_seed(17)
    rnd = torch.cat([torch.randn(20000, generator=g) * 50, torch.rand(5000, generator=g) * 0.03])
    x = torch.cat([mids, up, dn, -mids, -up, -dn, rnd.clamp(-448, 448), torch.tensor([0.0, -0.0, 448.0, -448.0])])
    got = orc.quantize_e4m3(x.numpy())
    want = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want)
    big = np.array([448.5, 464.0, 1e6, np.inf, -500.0, -np.inf], dtype=np.float32)
    assert np.array_equal(orc.quantize_e4m3(big), np.array([126, 126, 126, 126, 254, 254], dtype=np.uint8))
    assert orc.quantize_e4m3(np.array([np.nan], dtype=np.float32))[0] & 0x7f == 0x7f


def pin_e4m3_append(orc):
    """The E4M3 append stores the quantized fp32 quotient new / scale in the new slots only."""
    for new_dtype in ("bf16", "f32"):
        B, H, T_max, D, N = 2, 3, 9, 16, 2
        past = torch.tensor([3, 7], dtype=torch.int32)
        k_new = _rand((B, H, N, D), 61, new_dtype) * 7
        v_new = _rand((B, H, N, D), 62, new_dtype) * 0.02
        k_scale, v_scale = 0.75, 3.0e-4
        kc = np.full((B, H, T_max, D), 0xA5, dtype=np.uint8)
        vc = kc.copy()
        st = orc.append_e4m3(kc, vc, to_np(k_new), to_np(v_new), past.numpy(), new_dtype, k_scale, v_scale)
        assert st == 0
        kq = (k_new.float() / torch.tensor(k_scale, dtype=torch.float32)).to(torch.float8_e4m3fn)
        vq = (v_new.float() / torch.tensor(v_scale, dtype=torch.float32)).to(torch.float8_e4m3fn)
        exp_k = np.full_like(kc, 0xA5)
        exp_v = exp_k.copy()
        for b, P in enumerate(past.tolist()):
            exp_k[b, :, P:P + N] = kq[b].view(torch.uint8).numpy()
            exp_v[b, :, P:P + N] = vq[b].view(torch.uint8).numpy()
        assert np.array_equal(kc, exp_k) and np.array_equal(vc, exp_v)


def pin_e4m3_attention(orc):
    """E4M3 attention = attention over the exactly dequantized cache: bit for bit the
    fp32 oracle when the scales are powers of two (the products are exact), and
    library SDPA in float64 for general scales."""
    B, H_q, H_kv, D, N, T_max = 2, 8, 2, 32, 3, 20
    past = torch.tensor([6, 17], dtype=torch.int32)
    g = torch.Generator().manual_seed(23)
    k8 = torch.randint(0, 256, (B, H_kv, T_max, D), generator=g, dtype=torch.int32).to(torch.uint8)
    v8 = torch.randint(0, 256, (B, H_kv, T_max, D), generator=g, dtype=torch.int32).to(torch.uint8)
    for c in (k8, v8):  # no NaN codes in the visible slots
        c[(c & 0x7f) == 0x7f] = 0x3c
    q = _rand((B, H_q, N, D), 24, "bf16")
    for k_scale, v_scale in ((0.25, 8.0), (0.0173, 3.7)):
        out, st = orc.decode_attention_e4m3(to_np(q), k8.numpy(), v8.numpy(), past.numpy(), "bf16", k_scale, v_scale)
        assert st == 0
        kd = k8.view(torch.float8_e4m3fn).to(torch.float64) * k_scale
        vd = v8.view(torch.float8_e4m3fn).to(torch.float64) * v_scale
        if k_scale == 0.25:
            flat, st = orc.decode_attention(to_np(q.float()), kd.float().numpy(), vd.float().numpy(),
                                            past.numpy(), "f32")
            assert st == 0 and np.array_equal(out, flat)
        want = torch.stack([
            F.scaled_dot_product_attention(
                to_f64(q[b])[None], kd[b, :, : int(P) + N][None], vd[b, :, : int(P) + N][None],
                attn_mask=(torch.arange(int(P) + N)[None, :] <= (int(P) + torch.arange(N))[:, None]),
                scale=1.0 / D ** 0.5, enable_gqa=True)[0]
            for b, P in enumerate(past)])
        assert _max_rel(torch.from_numpy(out), want) < 1e-12


ALL_PINS = [
    pin_cache_bytes,
    pin_append_is_concat,
    pin_single_visible_key,
    pin_widening_all_patterns,
    pin_identical_keys_mean,
    pin_dominant_key,
    pin_route_b_sdpa,
    pin_full_causal_sdpa,
    pin_permutation_single_token,
    pin_reversed_order_trap,
    pin_paged_identity_layout,
    pin_paged_renumbered_pages,
    pin_paged_bad_page,
    pin_e4m3_decode_all_codes,
    pin_e4m3_quantize,
    pin_e4m3_append,
    pin_e4m3_attention,
]
