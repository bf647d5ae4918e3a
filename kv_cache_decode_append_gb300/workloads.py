"""Seeded synthetic workloads for the KV-cache decode step.

This module only describes shapes and draws random inputs; it performs none of
the method's arithmetic.  Tests feed the same tensors to the CUDA path and to
the CPU oracle, and the benchmark draws its inputs here.

The five workloads follow the shapes of the pages' GPT-2 Small experiment
(openai-hub.com/news/2435 "GPT-2缓存实测：千倍计算只快6倍", section
"实验到底测了什么": 12 layers, 12 heads, hidden 768 so head dim 64, context
limit 1024, batch 1, fp32) plus a grouped-query long-context case (query
heads share fewer KV heads, section "GPT-2缓存要占多少显存", last paragraphs).

Recipe (all workloads): Q, new K/V and cached history ~ N(0, 1) drawn in fp32
by ``torch.randn`` from a seeded generator, then rounded to bf16 (round to
nearest even, ``Tensor.to``) where the workload is bf16.  Seeds: workload id
``c`` and layer ``l`` give ``1000*c + l``; Q, K_new, V_new, the K cache and the V cache use
``10*that + {0, 1, 2, 3, 4}``; per-sequence history lengths use ``1000*c + 999``.
Cache slots at or past ``P_b`` hold a tail fill: NaN for correctness runs (a
masked slot that leaked into the arithmetic would poison the output) or 0 for
timing runs.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Optional, Tuple

import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@dataclass(frozen=True)
class Workload:
    wid: int                 # workload id (1..5), part of the seed
    name: str
    L: int                   # layers
    B: int                   # sequences
    H_q: int                 # query heads
    H_kv: int                # KV heads
    D: int                   # head dim
    N: int                   # new tokens per sequence
    dtype: str               # "f32" | "bf16" | "f16" (cache, q, new K/V and output)
    T_max: int               # preallocated slots per cache row
    P: Optional[int] = None                  # history length (same for every sequence)
    P_range: Optional[Tuple[int, int]] = None  # inclusive range, drawn per sequence

    @property
    def group(self) -> int:
        return self.H_q // self.H_kv

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def describe(self) -> str:
        p = f"P={self.P}" if self.P is not None else f"P~U[{self.P_range[0]},{self.P_range[1]}]"
        return (f"{self.name}: L={self.L} B={self.B} H_q={self.H_q} H_kv={self.H_kv} "
                f"D={self.D} {p} N={self.N} {self.dtype} T_max={self.T_max}")


WORKLOADS = {
    # GPT-2 Small, one layer, short history.
    "gpt2s_1layer_p16_f32": Workload(1, "gpt2s_1layer_p16_f32", L=1, B=1, H_q=12, H_kv=12, D=64,
                                     N=1, dtype="f32", T_max=1024, P=16),
    # GPT-2 Small, full stack, at the pages' measured context of 1000.
    "gpt2s_12layer_p1000_f32": Workload(2, "gpt2s_12layer_p1000_f32", L=12, B=1, H_q=12, H_kv=12,
                                        D=64, N=1, dtype="f32", T_max=1024, P=1000),
    # GPT-2 Small chunked decode (N new tokens, row i sees keys 0..P+i); N is swept.
    "gpt2s_chunked_p512_f32": Workload(3, "gpt2s_chunked_p512_f32", L=12, B=1, H_q=12, H_kv=12,
                                       D=64, N=16, dtype="f32", T_max=1024, P=512),
    # GPT-2 Small, batch 8 at the context limit, bf16 cache.
    "gpt2s_b8_p1023_bf16": Workload(4, "gpt2s_b8_p1023_bf16", L=12, B=8, H_q=12, H_kv=12, D=64,
                                    N=1, dtype="bf16", T_max=1024, P=1023),
    # Grouped-query long context: 32 layers, 32 sequences, 32 query / 8 KV heads.
    "gqa_longctx_b32_bf16": Workload(5, "gqa_longctx_b32_bf16", L=32, B=32, H_q=32, H_kv=8,
                                     D=128, N=1, dtype="bf16", T_max=8320, P_range=(1024, 8192)),
}

CHUNKED_N = (2, 4, 8, 16)


def with_n(w: Workload, N: int) -> Workload:
    return replace(w, N=N)


def past_lens(w: Workload) -> torch.Tensor:
    """History length per sequence (int32, CPU), before the append."""
    if w.P is not None:
        return torch.full((w.B,), w.P, dtype=torch.int32)
    g = torch.Generator("cpu").manual_seed(1000 * w.wid + 999)
    lo, hi = w.P_range
    return torch.randint(lo, hi + 1, (w.B,), generator=g, dtype=torch.int64).to(torch.int32)


def _randn(shape, seed: int, device, dtype: torch.dtype) -> torch.Tensor:
    g = torch.Generator(device).manual_seed(seed)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(dtype)


def layer_inputs(w: Workload, layer: int, past_len: torch.Tensor, device="cpu",
                 tail_fill: str = "nan", seed_base: Optional[int] = None) -> dict:
    """Q [B,H_q,N,D], K_new/V_new [B,H_kv,N,D] and caches [B,H_kv,T_max,D] of one layer.

    Cache slots ``t < past_len[b]`` are N(0,1); slots ``t >= past_len[b]`` hold
    ``tail_fill`` ("nan" or "zero").
    """
    dt = w.torch_dtype
    base = 10 * (1000 * w.wid + layer) if seed_base is None else 10 * seed_base
    q = _randn((w.B, w.H_q, w.N, w.D), base + 0, device, dt)
    k_new = _randn((w.B, w.H_kv, w.N, w.D), base + 1, device, dt)
    v_new = _randn((w.B, w.H_kv, w.N, w.D), base + 2, device, dt)
    shape = (w.B, w.H_kv, w.T_max, w.D)
    k_cache = _randn(shape, base + 3, device, dt)
    v_cache = _randn(shape, base + 4, device, dt)
    fill = float("nan") if tail_fill == "nan" else 0.0
    t = torch.arange(w.T_max, device=device).view(1, 1, w.T_max, 1)
    tail = t >= past_len.to(device=device, dtype=torch.int64).view(w.B, 1, 1, 1)
    k_cache.masked_fill_(tail, fill)
    v_cache.masked_fill_(tail, fill)
    return {"q": q, "k_new": k_new, "v_new": v_new, "k_cache": k_cache, "v_cache": v_cache}


def to_paged(k_cache: torch.Tensor, v_cache: torch.Tensor, page_size: int, extra_pages: int = 0,
             seed: int = 0, fill: float = float("nan"), shuffle: bool = True):
    """Lay contiguous [B,H_kv,T_max,D] caches out as a shuffled page pool.

    Returns ``(k_pages, v_pages, block_table)``: pages [num_pages, H_kv, page_size, D]
    with ``num_pages = B * max_pages + extra_pages`` (``max_pages = ceil(T_max /
    page_size)``), logical page j of sequence b stored at the seeded random physical
    page ``block_table[b, j]`` (or, without ``shuffle``, at page ``b * max_pages + j``);
    unused pages and the padding past T_max hold ``fill``.
    """
    B, H, T, D = k_cache.shape
    max_pages = -(-T // page_size)
    pad = max_pages * page_size - T
    dev = k_cache.device

    def logical(c):
        if pad:
            c = torch.cat([c, torch.full((B, H, pad, D), fill, dtype=c.dtype, device=dev)], dim=2)
        return c.reshape(B, H, max_pages, page_size, D).permute(0, 2, 1, 3, 4).reshape(
            B * max_pages, H, page_size, D)

    n_used = B * max_pages
    num_pages = n_used + extra_pages
    g = torch.Generator("cpu").manual_seed(seed)
    perm = torch.randperm(num_pages, generator=g)[:n_used] if shuffle else torch.arange(n_used)
    out = []
    for c in (k_cache, v_cache):
        pages = torch.full((num_pages, H, page_size, D), fill, dtype=c.dtype, device=dev)
        pages[perm.to(dev)] = logical(c)
        out.append(pages)
    table = perm.to(torch.int32).view(B, max_pages).to(dev)
    return out[0], out[1], table


def new_rows(w: Workload, layer: int, device="cpu") -> dict:
    """Q, K_new and V_new of one layer, drawn exactly as ``layer_inputs`` draws them
    (for a chunk size N set on an existing cache)."""
    dt = w.torch_dtype
    base = 10 * (1000 * w.wid + layer)
    return {"q": _randn((w.B, w.H_q, w.N, w.D), base + 0, device, dt),
            "k_new": _randn((w.B, w.H_kv, w.N, w.D), base + 1, device, dt),
            "v_new": _randn((w.B, w.H_kv, w.N, w.D), base + 2, device, dt)}
