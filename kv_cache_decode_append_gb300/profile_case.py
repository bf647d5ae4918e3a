"""Run a few decode steps of ONE layer of a workload, for kernel profilers.

    python -m kv_cache_decode_append_gb300.profile_case --workload gqa_longctx_b32_bf16 --launches 3

Each launch is one kvd_append + kvd_decode_attention (or, with --fused, one
kvd_decode_step; with --layout paged, their paged forms on a shuffled page
pool) on the same layer, so a
profiler filtered on a kernel name sees ``--launches`` identical launches with
the full-size per-layer working set (for the default workload 2 x 545 MB of
cache, larger than L2) and nothing else on the device.
"""
from __future__ import annotations

import argparse

import torch

from . import kvd
from . import workloads as wl


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="gqa_longctx_b32_bf16", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--n-new", type=int, default=None)
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--fused", action="store_true", help="kvd_decode_step instead of append + attention")
    ap.add_argument("--layout", default="contiguous", choices=["contiguous", "paged"])
    ap.add_argument("--cache", default="same", choices=["same", "e4m3"],
                    help="E4M3 cache codes (k_scale 0.05, v_scale 0.02) for a bf16 workload")
    ap.add_argument("--page-size", type=int, default=64)
    args = ap.parse_args()
    w = wl.WORKLOADS[args.workload]
    if args.n_new is not None:
        w = wl.with_n(w, args.n_new)
    dev = torch.device("cuda")
    past = wl.past_lens(w)
    max_past = int(past.max())
    x = wl.layer_inputs(w, 0, past, device=dev, tail_fill="zero")
    out = torch.empty_like(x["q"])
    past_d = past.to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = kvd.alloc_workspace(w.B, w.H_q, w.H_kv, w.D, w.N, max_past, w.torch_dtype, dev)
    if args.layout == "paged":
        kp, vp, table = wl.to_paged(x.pop("k_cache"), x.pop("v_cache"), args.page_size, fill=0.0)
    e4m3 = args.cache == "e4m3"
    if e4m3:
        for key, sc in (("k_cache", 0.05), ("v_cache", 0.02)):
            x[key] = (x[key].float() / sc).to(torch.float8_e4m3fn).view(torch.uint8)
        ws = kvd.alloc_workspace(w.B, w.H_q, w.H_kv, w.D, w.N, max_past, "e4m3", dev)
    for _ in range(args.launches):
        if e4m3 and args.fused:
            kvd.kvd_decode_step_e4m3(x["q"], x["k_cache"], x["v_cache"], x["k_new"], x["v_new"], out, past_d,
                                     max_past, 0.05, 0.02, 0.0, ws, err)
        elif e4m3:
            kvd.kvd_append_e4m3(x["k_cache"], x["v_cache"], x["k_new"], x["v_new"], past_d, max_past, 0.05, 0.02, err)
            kvd.kvd_decode_attention_e4m3(x["q"], x["k_cache"], x["v_cache"], out, past_d, max_past, 0.05, 0.02, 0.0,
                                          ws, err)
        elif args.layout == "paged" and args.fused:
            kvd.kvd_paged_decode_step(x["q"], kp, vp, x["k_new"], x["v_new"], out, table, past_d, max_past, 0.0,
                                      ws, err)
        elif args.layout == "paged":
            kvd.kvd_paged_append(kp, vp, x["k_new"], x["v_new"], table, past_d, max_past, err)
            kvd.kvd_paged_decode_attention(x["q"], kp, vp, out, table, past_d, max_past, 0.0, ws, err)
        elif args.fused:
            kvd.kvd_decode_step(x["q"], x["k_cache"], x["v_cache"], x["k_new"], x["v_new"], out, past_d,
                                max_past, 0.0, ws, err)
        else:
            kvd.kvd_append(x["k_cache"], x["v_cache"], x["k_new"], x["v_new"], past_d, max_past, err)
            kvd.kvd_decode_attention(x["q"], x["k_cache"], x["v_cache"], out, past_d, max_past, 0.0, ws, err)
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise SystemExit(f"device error word {int(err.item())}")
    print(f"{w.describe()}: {args.launches} launches ok")


if __name__ == "__main__":
    main()
