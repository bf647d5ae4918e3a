"""Benchmark of the KV-cache decode step on GB300.

One step = one decode step of the whole layer stack: for every layer,
kvd_decode_step (new K/V into the preallocated cache and split-T attention in
one launch, then the log-sum-exp merge), on one stream; ``--path separate``
times kvd_append + kvd_decode_attention instead.  The default workload is the
grouped-query long-context case (32 layers, B=32, 32 query / 8 KV heads,
D=128, per-sequence history U[1024, 8192], N=1, bf16); the K/V read per step
(21.8 GB) is far larger than L2, so no flush is needed between steps.  A
workload whose step reads less than twice the L2 gets a write of twice the
L2 size between timed steps, outside the per-step events.

Metric: achieved HBM GB/s of algorithmic bytes (K/V read over P+N keys, Q
read, O written, append read+write; workspace traffic excluded) and
microseconds per layer-step.  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

``--impl reference`` times the CPU oracle (double precision, all host cores)
on the same workload, one layer-step per step.  Under torchrun with N > 1 each
rank runs an independent replica (the path shards by sequence and head with no
exchange): weak scaling, the max time over ranks, no data-path collective.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from kv_cache_decode_append_gb300 import workloads as wl  # noqa: E402

METRIC = "decode attention: achieved HBM GB/s (% of GB300 peak) and μs per layer-step"
DEFAULT_WORKLOAD = "gqa_longctx_b32_bf16"
FALLBACK_HBM_GBS = 6800.0
L2_FALLBACK_BYTES = 132 * 10**6  # GB300 L2, when torch does not report it
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "decode_step_gqa_longctx_b32.md")


# ---------------------------------------------------------------------------------
# algorithmic bytes (the roofline's per-unit figures)
def attn_bytes(w: wl.Workload, past, cache_elem: int = 0) -> int:
    """K/V read over P_b + N keys of every (b, h_kv), plus Q read and O written
    (cache_elem: bytes per cache element when the cache type differs, E4M3: 1)."""
    s = w.elem_bytes
    c = cache_elem or s
    keys = sum(int(p) + w.N for p in past)
    return 2 * w.H_kv * w.D * c * keys + 2 * w.B * w.H_q * w.N * w.D * s


def append_bytes(w: wl.Workload, cache_elem: int = 0) -> int:
    """New K and V read, and written into the cache (in the cache's element size)."""
    return 2 * w.B * w.H_kv * w.N * w.D * (w.elem_bytes + (cache_elem or w.elem_bytes))


def layer_bytes(w, past, cache_elem: int = 0) -> int:
    return attn_bytes(w, past, cache_elem) + append_bytes(w, cache_elem)


# ---------------------------------------------------------------------------------
def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """C++/CUDA source without its comments and with whitespace runs collapsed:
    a comment edit does not change what the counters were taken on."""
    out, i, n = [], 0, len(text)
    while i < n:
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif text[i] == '"':  # string literal (asm text, messages): kept verbatim
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(text[i])
            i += 1
    return " ".join("".join(out).split())


# Device sources the dominant kernel of the default workload (the bf16 mma.sync
# decode step and its merge pass, described by PROFILE_SUMMARY) is compiled from.
PROFILED_KERNEL_SOURCES = ("kvd_device.cuh", "kvd_attention.cuh", "kvd_attention_mma.cuh", "kvd_mma_bf16.cu",
                           "kvd_mma_bf16_tk.cu")


def kernel_source_hash() -> str:
    """Hash of the profiled kernel's sources (code only, see _code_only)."""
    h = hashlib.sha256()
    for name in PROFILED_KERNEL_SOURCES:
        with open(os.path.join(ROOT, "kv_cache_decode_append_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it matches this source."""
    try:
        with open(PROFILE_SUMMARY) as f:
            text = f.read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("kernel_source_sha256") != kernel_source_hash():
        return None
    try:
        return float(fields["dram_bytes_per_full_launch"])
    except (KeyError, ValueError):
        return None


def gpu_smi_id(dev) -> str:
    """An nvidia-smi --id for this torch device (PCI bus id, else UUID, else index)."""
    props = torch.cuda.get_device_properties(dev)
    try:
        return f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
    except AttributeError:
        pass
    try:
        u = str(props.uuid)
        return u if u.startswith("GPU-") else f"GPU-{u}"
    except AttributeError:
        return str(dev.index or 0)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms in the background."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: str):
        self.index = index
        self.samples = []  # (time, sm_mhz, max_mhz, reasons)
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            reasons = [n for n, v in zip(names, parts[5:9]) if v.lower() == "active"]
            self.samples.append((time.time(), sm, mx, reasons))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        used = inside if inside else [s for s in self.samples if t0 - 0.5 <= s[0] <= t1 + 0.5]
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({r for s in used for r in s[3]})
        return {"sm_mhz": statistics.median(s[1] for s in used), "sm_max_mhz": max(s[2] for s in used),
                "reasons": reasons, "samples": len(used),
                "window": "timed region" if inside else "timed region +-0.5 s"}


# ---------------------------------------------------------------------------------
def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Host-side aggregation of the timed region (not part of the data path)."""
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda") if torch.cuda.is_available() and dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step_per_rank: int, steps: int, elapsed_max_s: float, world: int) -> float:
    """Weak scaling: every rank processes the same step; the job moves world x
    the bytes of one rank in the slowest rank's time."""
    return world * bytes_per_step_per_rank * steps / elapsed_max_s / 1e9


E4M3_SCALES = (0.05, 0.02)  # k_scale, v_scale of the E4M3 cache runs (N(0,1) data)


def oracle_layer_step(orc, host, past_np, dtype):
    if host["k_cache" if "k_cache" in host else "k_pages"].dtype == "uint8":  # E4M3 cache
        st = orc.append_e4m3(host["k_cache"], host["v_cache"], host["k_new"], host["v_new"], past_np, dtype,
                             *E4M3_SCALES)
        out, st2 = orc.decode_attention_e4m3(host["q"], host["k_cache"], host["v_cache"], past_np, dtype,
                                             *E4M3_SCALES)
    elif "k_pages" in host:  # paged layout
        st = orc.paged_append(host["k_pages"], host["v_pages"], host["k_new"], host["v_new"], host["table"],
                              past_np, dtype)
        out, st2 = orc.paged_decode_attention(host["q"], host["k_pages"], host["v_pages"], host["table"],
                                              past_np, dtype)
    else:
        st = orc.append(host["k_cache"], host["v_cache"], host["k_new"], host["v_new"], past_np, dtype)
        out, st2 = orc.decode_attention(host["q"], host["k_cache"], host["v_cache"], past_np, dtype)
    if st != 0 or st2 != 0:
        raise RuntimeError("oracle rejected the workload")
    return out


def to_host_np(t: torch.Tensor):
    import numpy as np
    t = t.detach().contiguous().cpu()
    if t.dtype in (torch.int32, torch.uint8):
        return t.numpy().copy()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def time_oracle(w, host, past, budget_s: float = 10.0, max_reps: int = 64):
    """Repeat the oracle's layer-step on one layer's host data for about budget_s."""
    import oracle
    orc = oracle.load()
    past_np = past.numpy()
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle_layer_step(orc, host, past_np, w.dtype)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= max_reps:
            break
    return reps, el, orc.max_threads()


# ---------------------------------------------------------------------------------
def run_reference(args, w, rank, world):
    """The reference arm: the CPU oracle, as it stands, one layer-step per step."""
    if rank != 0:
        return
    import oracle
    orc = oracle.load()
    past = wl.past_lens(w)
    t = wl.layer_inputs(w, 0, past, device="cpu", tail_fill="zero")
    host = {k: to_host_np(v) for k, v in t.items()}
    past_np = past.numpy()
    for _ in range(args.warmup):
        oracle_layer_step(orc, host, past_np, w.dtype)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_layer_step(orc, host, past_np, w.dtype)
    el = time.perf_counter() - t0
    per_step = el / args.steps
    gbs = layer_bytes(w, past.tolist()) / per_step / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(per_step * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "describe": w.describe(),
                   "step": "one layer-step (append + decode attention) of the workload"},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": orc.max_threads(),
                         "kind": "oracle",
                         "sample": f"one layer of {w.name} (all {w.B} sequences) per step"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_gpu(args, w, rank, world, local):
    import kv_cache_decode_append_gb300 as kvd

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    past = wl.past_lens(w)
    max_past = int(past.max())
    past_d = past.to(dev)
    paged = args.layout == "paged"
    e4m3 = args.cache == "e4m3"
    if e4m3 and (paged or w.dtype != "bf16"):
        raise SystemExit("--cache e4m3 needs a bf16 workload and the contiguous layout")
    cache_elem = 1 if e4m3 else 0
    layers = []
    for l in range(w.L):
        x = wl.layer_inputs(w, l, past, device=dev, tail_fill="zero")
        if e4m3:  # the same data as E4M3 codes (torch's float8 cast of value / scale)
            for key, sc in zip(("k_cache", "v_cache"), E4M3_SCALES):
                x[key] = (x[key].float() / sc).to(torch.float8_e4m3fn).view(torch.uint8)
        if paged:  # the same data as a shuffled page pool with a block table
            x["k_pages"], x["v_pages"], x["table"] = wl.to_paged(
                x.pop("k_cache"), x.pop("v_cache"), args.page_size, seed=l, fill=0.0,
                shuffle=args.page_order == "shuffled")
        layers.append(x)
    outs = [torch.empty_like(x["q"]) for x in layers]
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    plan_dtype = "e4m3" if e4m3 else w.torch_dtype
    ws = kvd.alloc_workspace(w.B, w.H_q, w.H_kv, w.D, w.N, max_past, plan_dtype, dev)
    plan = kvd.kvd_decode_plan(w.B, w.H_q, w.H_kv, w.D, w.N, max_past, plan_dtype)
    merge = plan["launches"] == 2
    launches_per_layer = plan["launches"] + (0 if args.path == "fused" else 1)

    fused = args.path == "fused"

    def layer_step(l):
        x = layers[l]
        # the current stream: the capture stream inside torch.cuda.graph
        if e4m3 and fused:
            kvd.kvd_decode_step_e4m3(x["q"], x["k_cache"], x["v_cache"], x["k_new"], x["v_new"], outs[l], past_d,
                                     max_past, *E4M3_SCALES, 0.0, ws, err)
        elif e4m3:
            kvd.kvd_append_e4m3(x["k_cache"], x["v_cache"], x["k_new"], x["v_new"], past_d, max_past,
                                *E4M3_SCALES, err)
            kvd.kvd_decode_attention_e4m3(x["q"], x["k_cache"], x["v_cache"], outs[l], past_d, max_past,
                                          *E4M3_SCALES, 0.0, ws, err)
        elif paged and fused:
            kvd.kvd_paged_decode_step(x["q"], x["k_pages"], x["v_pages"], x["k_new"], x["v_new"], outs[l],
                                      x["table"], past_d, max_past, 0.0, ws, err)
        elif paged:
            kvd.kvd_paged_append(x["k_pages"], x["v_pages"], x["k_new"], x["v_new"], x["table"], past_d,
                                 max_past, err)
            kvd.kvd_paged_decode_attention(x["q"], x["k_pages"], x["v_pages"], outs[l], x["table"], past_d,
                                           max_past, 0.0, ws, err)
        elif fused:
            kvd.kvd_decode_step(x["q"], x["k_cache"], x["v_cache"], x["k_new"], x["v_new"], outs[l], past_d,
                                max_past, 0.0, ws, err)
        else:
            kvd.kvd_append(x["k_cache"], x["v_cache"], x["k_new"], x["v_new"], past_d, max_past, err)
            kvd.kvd_decode_attention(x["q"], x["k_cache"], x["v_cache"], outs[l], past_d, max_past, 0.0, ws,
                                     err)

    def step():
        for l in range(w.L):
            layer_step(l)

    # warm-up (also builds nothing: the library is loaded on the first call)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())}")

    sampler = ClockSampler(gpu_smi_id(dev))
    if rank == 0:
        sampler.start()
        time.sleep(0.2)

    # The step is captured once as a CUDA graph (launch overhead off the
    # critical path); a second graph holds only the L attention calls, for
    # the roofline of the attention kernel.
    step_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(step_graph):
        step()
    attn_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(attn_graph):
        for l in range(w.L):
            x = layers[l]
            if e4m3 and fused:
                kvd.kvd_decode_step_e4m3(x["q"], x["k_cache"], x["v_cache"], x["k_new"], x["v_new"], outs[l],
                                         past_d, max_past, *E4M3_SCALES, 0.0, ws, err)
            elif e4m3:
                kvd.kvd_decode_attention_e4m3(x["q"], x["k_cache"], x["v_cache"], outs[l], past_d, max_past,
                                              *E4M3_SCALES, 0.0, ws, err)
            elif paged and fused:
                kvd.kvd_paged_decode_step(x["q"], x["k_pages"], x["v_pages"], x["k_new"], x["v_new"], outs[l],
                                          x["table"], past_d, max_past, 0.0, ws, err)
            elif paged:
                kvd.kvd_paged_decode_attention(x["q"], x["k_pages"], x["v_pages"], outs[l], x["table"], past_d,
                                               max_past, 0.0, ws, err)
            elif fused:  # the dominant kernel is the fused step itself
                kvd.kvd_decode_step(x["q"], x["k_cache"], x["v_cache"], x["k_new"], x["v_new"], outs[l],
                                    past_d, max_past, 0.0, ws, err)
            else:
                kvd.kvd_decode_attention(x["q"], x["k_cache"], x["v_cache"], outs[l], past_d, max_past, 0.0,
                                         ws, err)
    graph_stream = torch.cuda.current_stream()
    for _ in range(2):
        step_graph.replay()
        attn_graph.replay()
    torch.cuda.synchronize()

    # A step that reads less than twice the L2 would find its inputs there on
    # the next step: then every timed step gets its own events, with a write
    # of twice the L2 size between steps (outside the events).
    step_bytes = w.L * layer_bytes(w, past.tolist(), cache_elem)
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or L2_FALLBACK_BYTES)
    flush = step_bytes <= 2 * l2_bytes
    scratch = torch.empty(2 * l2_bytes // 4, dtype=torch.int32, device=dev) if flush else None

    def replay_timed(graph) -> float:
        """Seconds of args.steps replays of graph, on its stream."""
        if not flush:
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(graph_stream)
            for _ in range(args.steps):
                graph.replay()
            t1.record(graph_stream)
            torch.cuda.synchronize()
            return t0.elapsed_time(t1) / 1e3
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for i, (t0, t1) in enumerate(evs):
            scratch.fill_(i)
            t0.record(graph_stream)
            graph.replay()
            t1.record(graph_stream)
        torch.cuda.synchronize()
        return sum(t0.elapsed_time(t1) for t0, t1 in evs) / 1e3

    # timed region: K steps
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    elapsed = replay_timed(step_graph)
    t_wall1 = time.time()
    barrier(world)
    elapsed_max = max_over_ranks(elapsed, world)

    # attention kernel alone, same number of launches
    attn_per_launch = replay_timed(attn_graph) / (args.steps * w.L)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())}")

    # end to end: inputs from pinned host memory each step, result read back each step
    host_in = [{k: layers[l][k].cpu().pin_memory() for k in ("q", "k_new", "v_new")} for l in range(w.L)]
    host_out = [torch.empty(outs[l].shape, dtype=outs[l].dtype).pin_memory() for l in range(w.L)]
    past_h = past.pin_memory()
    h2d = sum(t.numel() * t.element_size() for d in host_in for t in d.values()) + past_h.numel() * 4
    d2h = sum(t.numel() * t.element_size() for t in host_out)

    def e2e_step():
        past_d.copy_(past_h, non_blocking=True)
        for l in range(w.L):
            for key in ("q", "k_new", "v_new"):
                layers[l][key].copy_(host_in[l][key], non_blocking=True)
            layer_step(l)
            host_out[l].copy_(outs[l], non_blocking=True)
        stream.synchronize()

    for _ in range(max(1, args.warmup // 2)):
        e2e_step()
    barrier(world)
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_steps = max(1, args.steps // 2)
    e_start.record(stream)
    for _ in range(e_steps):
        e2e_step()
    e_end.record(stream)
    torch.cuda.synchronize()
    e2e_el = max_over_ranks(e_start.elapsed_time(e_end) / 1e3, world)
    if rank == 0:
        sampler.stop()

    if rank != 0:
        return
    bytes_step = w.L * layer_bytes(w, past.tolist(), cache_elem)
    gbs = whole_job_gbs(bytes_step, args.steps, elapsed_max, world)
    ms_step = elapsed_max / args.steps * 1e3
    peak, peak_kind = measured_peak()
    a_bytes = layer_bytes(w, past.tolist(), cache_elem) if fused else attn_bytes(w, past.tolist(), cache_elem)
    achieved = a_bytes / attn_per_launch / 1e9

    # CPU baseline: the oracle on layer 0's data, all host cores, ~10 s
    host = {k: to_host_np(v) for k, v in layers[0].items()}
    reps, cpu_el, cores = time_oracle(w, host, past, budget_s=args.cpu_seconds)
    cpu_gbs = reps * layer_bytes(w, past.tolist(), cache_elem) / cpu_el / 1e9

    line = {
        "metric": METRIC,
        "value": round(gbs, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic",
        "config": {
            "workload": w.name, "describe": w.describe(), "layers": w.L, "B": w.B, "H_q": w.H_q,
            "H_kv": w.H_kv, "D": w.D, "N": w.N, "T_max": w.T_max,
            "P": (w.P if w.P is not None else f"U[{w.P_range[0]},{w.P_range[1]}] seeded, sum {int(past.sum())}"),
            "step": (f"{w.L} x kvd_decode_step (append + attention in one launch)" if fused else
                     f"{w.L} x (kvd_append + kvd_decode_attention)") + " on one stream, one CUDA graph per step",
            "l2": (f"flushed: {2 * l2_bytes / 1e6:.0f} MB written between timed steps, outside their events "
                   f"({bytes_step / 1e6:.1f} MB per step; e2e not flushed)") if flush else
                  f"no flush: inputs larger than L2 ({bytes_step / 1e9:.1f} GB per step)",
            "parallelism": f"replicas x{world}",
            "cache_layout": (f"paged: {args.page_size}-token pages, {args.page_order} pool, block table"
                             if paged else "contiguous [B, H_kv, T_max, D]"),
            "cache_dtype": (f"e4m3 (k_scale {E4M3_SCALES[0]}, v_scale {E4M3_SCALES[1]}; q, new K/V, out bf16)"
                            if e4m3 else w.dtype),
        },
        "us_per_layer_step": round(ms_step * 1e3 / w.L, 3),
        "frac_of_peak": round(gbs / world / peak, 4),
        "attn_us_per_layer": round(attn_per_launch * 1e6, 3),
        "path": args.path,
        "roofline": {
            "bound": "hbm",
            "kernel": ("kvd_decode_step (fused append + split-T attention" if fused else
                       "kvd_decode_attention (split-T attention") + (" + LSE merge)" if merge else ")"),
            "timing": "graph of the L calls replayed K times, CUDA events on its stream",
            "achieved": round(achieved, 2),
            "peak": peak,
            "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, copy burst)" if peak_kind == "measured" else "fallback",
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "algorithmic_bytes_per_launch": a_bytes,
            "plan": plan,
            "traffic": None if (paged or e4m3) else profiled_traffic(),
        },
        "cpu_baseline": {
            "value": round(cpu_gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"layer 0 of {w.name} (all {w.B} sequences, append + attention, fp64), "
                      f"repeated {reps}x in {cpu_el:.1f} s",
        },
        "e2e": {
            "value": round(whole_job_gbs(bytes_step, e_steps, e2e_el, world), 2), "unit": "GB/s",
            "ms_per_step": round(e2e_el / e_steps * 1e3, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
        },
        "gpu_launches": args.steps * w.L * launches_per_layer,
        "clocks": sampler.summary(t_wall0, t_wall1),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--n-new", type=int, default=None, help="override N (chunked decode sweep)")
    ap.add_argument("--impl", default="kvd", choices=["kvd", "reference"])
    ap.add_argument("--path", default="fused", choices=["fused", "separate"],
                    help="fused: kvd_decode_step per layer; separate: kvd_append + kvd_decode_attention")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--layout", default="contiguous", choices=["contiguous", "paged"],
                    help="KV cache layout (paged: kvd_paged_* on a shuffled page pool)")
    ap.add_argument("--page-size", type=int, default=64, help="tokens per page for --layout paged")
    ap.add_argument("--cache", default="same", choices=["same", "e4m3"],
                    help="cache element type: the workload's, or E4M3 codes (bf16 workloads)")
    ap.add_argument("--page-order", default="shuffled", choices=["shuffled", "sequential"],
                    help="physical page order of the pool for --layout paged")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = wl.WORKLOADS[args.workload]
    if args.n_new is not None:
        w = wl.with_n(w, args.n_new)
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, w, rank, world)
    else:
        run_gpu(args, w, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
