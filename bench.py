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
microseconds per layer-step.  Prints ONE JSON line on rank 0.  Each timed step
replays the step graph R times, R chosen so that the timed region spans at
least --min-seconds (R = 1 when the L2 is flushed between steps), which gives
the clock sampler tens of samples.  A single-GPU default run also times the
other workloads (``per_config``: the GPT-2 Small cases, the chunked sweep
N = 2, 4, 8, 16, the long-context caches with N = 8 and with an E4M3 cache),
each with its own end-to-end time and the oracle's time on all host cores and
on one; ``memory`` puts the allocator's counters next to the cache size
formula.

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
def config_block(w: wl.Workload, past, world: int, layout: str = "contiguous", page_size: int = 64,
                 page_order: str = "shuffled", cache: str = "same") -> dict:
    """The workload keys shared by both arms' ``config`` (shapes, layout, cache type)."""
    return {
        "workload": w.name, "describe": w.describe(), "layers": w.L, "B": w.B, "H_q": w.H_q,
        "H_kv": w.H_kv, "D": w.D, "N": w.N, "T_max": w.T_max,
        "P": (w.P if w.P is not None else f"U[{w.P_range[0]},{w.P_range[1]}] seeded, sum {int(sum(past))}"),
        "parallelism": f"replicas x{world}",
        "cache_layout": (f"paged: {page_size}-token pages, {page_order} pool, block table"
                         if layout == "paged" else "contiguous [B, H_kv, T_max, D]"),
        "cache_dtype": (f"e4m3 (k_scale {E4M3_SCALES[0]}, v_scale {E4M3_SCALES[1]}; q, new K/V, out bf16)"
                        if cache == "e4m3" else w.dtype),
    }


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
    config = config_block(w, past.tolist(), world)
    config["step"] = (f"one layer-step (append + decode attention, fp64) of the {w.L}-layer workload per "
                      f"step, as a bounded sample; GB/s (algorithmic bytes / time) is the unit comparable "
                      f"with the GPU arm, whose step is the whole layer stack")
    config["l2"] = "host memory (CPU oracle)"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(per_step * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config,
        "us_per_layer_step": round(per_step * 1e6, 1),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": orc.max_threads(),
                         "kind": "oracle",
                         "sample": f"one layer of {w.name} (all {w.B} sequences) per step"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------
class Case:
    """One workload on the device: every layer's inputs, caches, outputs and the
    calls of one decode step, as the library's public API takes them."""

    def __init__(self, w, dev, *, path="fused", layout="contiguous", cache="same", page_size=64,
                 page_order="shuffled", reuse=None, flags=None):
        import kv_cache_decode_append_gb300 as kvd
        self.kvd = kvd
        self.w, self.dev = w, dev
        self.fused = path == "fused"
        self.paged = layout == "paged"
        self.e4m3 = cache == "e4m3"
        self.flags = flags  # kvd_decode_step_flags (contiguous fused step): the caller's guarantees
        if self.e4m3 and (self.paged or w.dtype != "bf16"):
            raise SystemExit("an E4M3 cache needs a bf16 workload and the contiguous layout")
        self.cache_elem = 1 if self.e4m3 else 0
        self.past = wl.past_lens(w)
        self.max_past = int(self.past.max())
        self.past_d = self.past.to(dev)
        self.layers = []
        for l in range(w.L):
            if reuse is not None:  # another chunk size N over the same caches
                x = wl.new_rows(w, l, device=dev)
                for key in ("k_cache", "v_cache", "k_pages", "v_pages", "table"):
                    if key in reuse.layers[l]:
                        x[key] = reuse.layers[l][key]
            else:
                x = wl.layer_inputs(w, l, self.past, device=dev, tail_fill="zero")
                if self.e4m3:  # the same data as E4M3 codes (torch's float8 cast of value / scale)
                    for key, sc in zip(("k_cache", "v_cache"), E4M3_SCALES):
                        x[key] = (x[key].float() / sc).to(torch.float8_e4m3fn).view(torch.uint8)
                if self.paged:  # the same data as a page pool with a block table
                    x["k_pages"], x["v_pages"], x["table"] = wl.to_paged(
                        x.pop("k_cache"), x.pop("v_cache"), page_size, seed=l, fill=0.0,
                        shuffle=page_order == "shuffled")
            self.layers.append(x)
        self.outs = [torch.empty_like(x["q"]) for x in self.layers]
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        plan_dtype = "e4m3" if self.e4m3 else w.torch_dtype
        self.ws = kvd.alloc_workspace(w.B, w.H_q, w.H_kv, w.D, w.N, self.max_past, plan_dtype, dev)
        self.plan = kvd.kvd_decode_plan(w.B, w.H_q, w.H_kv, w.D, w.N, self.max_past, plan_dtype)
        self.launches_per_layer = self.plan["launches"] + (0 if self.fused else 1)
        self.step_bytes = w.L * layer_bytes(w, self.past.tolist(), self.cache_elem)

    def layer_call(self, l, attention_only=False):
        kvd, x, out, past_d, mp = self.kvd, self.layers[l], self.outs[l], self.past_d, self.max_past
        ws, err = self.ws, self.err
        if self.e4m3 and self.fused:
            kvd.kvd_decode_step_e4m3(x["q"], x["k_cache"], x["v_cache"], x["k_new"], x["v_new"], out, past_d,
                                     mp, *E4M3_SCALES, 0.0, ws, err)
        elif self.e4m3:
            if not attention_only:
                kvd.kvd_append_e4m3(x["k_cache"], x["v_cache"], x["k_new"], x["v_new"], past_d, mp,
                                    *E4M3_SCALES, err)
            kvd.kvd_decode_attention_e4m3(x["q"], x["k_cache"], x["v_cache"], out, past_d, mp, *E4M3_SCALES,
                                          0.0, ws, err)
        elif self.paged and self.fused:
            kvd.kvd_paged_decode_step(x["q"], x["k_pages"], x["v_pages"], x["k_new"], x["v_new"], out,
                                      x["table"], past_d, mp, 0.0, ws, err)
        elif self.paged:
            if not attention_only:
                kvd.kvd_paged_append(x["k_pages"], x["v_pages"], x["k_new"], x["v_new"], x["table"], past_d,
                                     mp, err)
            kvd.kvd_paged_decode_attention(x["q"], x["k_pages"], x["v_pages"], out, x["table"], past_d, mp,
                                           0.0, ws, err)
        elif self.fused:
            kvd.kvd_decode_step(x["q"], x["k_cache"], x["v_cache"], x["k_new"], x["v_new"], out, past_d, mp,
                                0.0, ws, err, flags=self.flags)
        else:
            if not attention_only:
                kvd.kvd_append(x["k_cache"], x["v_cache"], x["k_new"], x["v_new"], past_d, mp, err)
            kvd.kvd_decode_attention(x["q"], x["k_cache"], x["v_cache"], out, past_d, mp, 0.0, ws, err)

    def step(self, attention_only=False):
        for l in range(self.w.L):
            self.layer_call(l, attention_only)

    def check_err(self):
        torch.cuda.synchronize()
        if int(self.err.item()) != 0:
            raise RuntimeError(f"{self.w.name}: device error word {int(self.err.item())}")

    def graph(self, attention_only=False):
        """The L calls of one step captured as one CUDA graph (launch overhead off the
        critical path; programmatic launches keep their early start inside it)."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step(attention_only)
        return g

    def e2e(self, steps, warmup, world):
        """The same step through the public API with its inputs in page-locked host
        memory and every layer's output read back, every step (eager calls).  A
        contiguous fused step goes through kvd_decode_step_host_packed (the library copies
        q, k_new, v_new and past_len in and out back, on the stream); the other
        paths copy with torch around their device-pointer calls."""
        w, stream = self.w, torch.cuda.current_stream()
        host_in = [{k: self.layers[l][k].cpu().pin_memory() for k in ("q", "k_new", "v_new")}
                   for l in range(w.L)]
        host_out = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in self.outs]
        past_h = self.past.pin_memory()
        in_bytes = sum(t.numel() * t.element_size() for d in host_in for t in d.values())
        d2h = sum(t.numel() * t.element_size() for t in host_out)
        host_call = self.fused and not self.paged and not self.e4m3 and not self.flags
        if host_call:
            # each layer's inputs in one page-locked block laid out as the
            # staging buffer's inputs: one host-to-device copy per call
            kvd = self.kvd
            staging = kvd.alloc_host_staging(w.B, w.H_q, w.H_kv, w.D, w.N, w.torch_dtype, self.dev)
            packed = []
            for l in range(w.L):
                hp = kvd.alloc_host_inputs(w.B, w.H_q, w.H_kv, w.D, w.N, w.torch_dtype)
                for key in ("q", "k_new", "v_new"):
                    hp[key].copy_(host_in[l][key])
                hp["past_len"].copy_(self.past)
                packed.append(hp)
            h2d = in_bytes + w.L * past_h.numel() * 4

            def one():
                for l in range(w.L):
                    x, hp = self.layers[l], packed[l]
                    kvd.kvd_decode_step_host_packed(hp, x["k_cache"], x["v_cache"], host_out[l], self.max_past,
                                                    staging, 0.0, self.ws, self.err)
                stream.synchronize()
        else:
            h2d = in_bytes + past_h.numel() * 4

            def one():
                self.past_d.copy_(past_h, non_blocking=True)
                for l in range(w.L):
                    for key in ("q", "k_new", "v_new"):
                        self.layers[l][key].copy_(host_in[l][key], non_blocking=True)
                    self.layer_call(l)
                    host_out[l].copy_(self.outs[l], non_blocking=True)
                stream.synchronize()

        for _ in range(max(1, warmup)):
            one()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            one()
        e1.record(stream)
        torch.cuda.synchronize()
        el = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
        return {"value": round(whole_job_gbs(self.step_bytes, steps, el, world), 2), "unit": "GB/s",
                "ms_per_step": round(el / steps * 1e3, 4), "us_per_layer_step": round(el / steps / w.L * 1e6, 3),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": "kvd_decode_step_host_packed (host buffers, one copy in and one out per call)" if host_call else
                       "device-pointer calls, torch copies from / to page-locked host memory",
                "timing": f"{steps} eager steps, CUDA events on the stream"}


class Timer:
    """CUDA-event timing of graph replays on the capturing stream.  A workload whose
    step reads less than twice the L2 gets a write of twice the L2 size before each
    timed step, outside its events, so every step starts from a cold L2."""

    def __init__(self, dev):
        self.stream = torch.cuda.current_stream()
        self.l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or L2_FALLBACK_BYTES)
        self.scratch = torch.empty(2 * self.l2_bytes // 4, dtype=torch.int32, device=dev)

    def needs_flush(self, step_bytes):
        return step_bytes <= 2 * self.l2_bytes

    def time(self, graph, steps, replays, flush):
        """Seconds of steps x replays graph replays (the sum over per-step windows
        when flushing; then replays is 1)."""
        if not flush:
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(self.stream)
            for _ in range(steps * replays):
                graph.replay()
            t1.record(self.stream)
            torch.cuda.synchronize()
            return t0.elapsed_time(t1) / 1e3
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for i, (t0, t1) in enumerate(evs):
            self.scratch.fill_(i)
            t0.record(self.stream)
            graph.replay()
            t1.record(self.stream)
        torch.cuda.synchronize()
        return sum(t0.elapsed_time(t1) for t0, t1 in evs) / 1e3


def oracle_times(case, cores_all: int, reps_all: int = 1, reps_one: int = 1):
    """The oracle on layer 0 of a case: ms per layer-step on all host cores and on one."""
    import oracle
    orc = oracle.load()
    host = {k: to_host_np(v) for k, v in case.layers[0].items()}
    past_np = case.past.numpy()
    out = {}
    for label, cores, reps in (("all_cores", cores_all, reps_all), ("one_core", 1, reps_one)):
        if reps < 1:
            continue
        orc.set_threads(cores)
        t0 = time.perf_counter()
        for _ in range(reps):
            oracle_layer_step(orc, host, past_np, case.w.dtype)
        out[label] = {"ms_per_layer_step": round((time.perf_counter() - t0) / reps * 1e3, 3), "cores": cores,
                      "reps": reps}
    orc.set_threads(cores_all)
    return out


def per_config_line(case, timer, steps, world, label, cores_all, with_oracle=True):
    """Throughput of one more workload (a graph of its L-layer step, timed like the
    headline), its end-to-end time and the oracle's time on its layer 0."""
    w = case.w
    for _ in range(3):
        case.step()
    case.check_err()
    g = case.graph()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    flush = timer.needs_flush(case.step_bytes)
    n = max(steps, 20)
    el = max_over_ranks(timer.time(g, n, 1, flush), world)
    case.check_err()
    peak, _ = measured_peak()
    gbs = whole_job_gbs(case.step_bytes, n, el, world)
    line = {
        "workload": w.name, "N": w.N, "label": label, "path": "fused" if case.fused else "separate",
        "flags": case.flags or 0,
        "us_per_layer_step": round(el / n / w.L * 1e6, 3), "gbs": round(gbs, 2),
        "frac": round(gbs / world / peak, 4), "step_bytes": case.step_bytes,
        "l2": "flushed before each step" if flush else "not flushed (step larger than twice the L2)",
        "steps": n,
        "plan": {k: case.plan[k] for k in ("grid", "tensor_cores", "launches", "early_start", "cluster", "rows_per_block")},
        "e2e": case.e2e(max(3, steps // 4), 2, world),
    }
    if with_oracle:
        line["oracle"] = oracle_times(case, cores_all)
    del g
    return line


def kvd_stable_flag() -> int:
    import kv_cache_decode_append_gb300 as kvd
    return kvd.KVD_STEP_HISTORY_STABLE


def memory_report(case, ws_bytes):
    w = case.w
    s = 1 if case.e4m3 else w.elem_bytes
    return {
        "kv_cache_bytes_preallocated": case.kvd.kvd_cache_bytes(w.L, w.B, w.H_kv, w.D, w.T_max,
                                                                 "e4m3" if case.e4m3 else w.torch_dtype),
        "kv_cache_bytes_in_use": 2 * w.L * w.H_kv * w.D * s * sum(int(p) + w.N for p in case.past.tolist()),
        "workspace_bytes": ws_bytes,
        "torch_memory_allocated": torch.cuda.memory_allocated(),
        "torch_memory_reserved": torch.cuda.memory_reserved(),
        "torch_max_memory_allocated": torch.cuda.max_memory_allocated(),
        "note": "torch counters taken after the timed region (peak since the caches were allocated)",
    }


def run_gpu(args, w, rank, world, local):
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    case = Case(w, dev, path=args.path, layout=args.layout, cache=args.cache, page_size=args.page_size,
                page_order=args.page_order)
    for _ in range(args.warmup):
        case.step()
    case.check_err()

    sampler = ClockSampler(gpu_smi_id(dev))
    if rank == 0:
        sampler.start()
        time.sleep(0.2)

    # The step is captured once as a CUDA graph; a second graph holds only the
    # attention calls (the fused step itself when fused), for the roofline.
    step_graph = case.graph()
    attn_graph = case.graph(attention_only=True)
    for _ in range(2):
        step_graph.replay()
        attn_graph.replay()
    torch.cuda.synchronize()
    timer = Timer(dev)
    flush = timer.needs_flush(case.step_bytes)

    # Each timed step replays the step graph R times (R = 1 with an L2 flush), R
    # chosen so that the timed region spans at least --min-seconds.
    replays = 1
    if not flush:
        probe = timer.time(step_graph, 3, 1, False) / 3
        replays = max(1, int(-(-args.min_seconds // max(probe * args.steps, 1e-9))))

    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    elapsed = timer.time(step_graph, args.steps, replays, flush)
    t_wall1 = time.time()
    barrier(world)
    elapsed_max = max_over_ranks(elapsed, world)
    passes = args.steps * replays
    attn_per_launch = timer.time(attn_graph, args.steps, replays, flush) / (passes * w.L)
    case.check_err()
    mem = memory_report(case, case.ws.numel() if case.ws is not None else 0)
    e2e = case.e2e(max(1, args.steps // 2), max(1, args.warmup // 2), world)
    clocks = sampler.summary(t_wall0, t_wall1)

    # More workloads on the same device: the other configurations, the chunked
    # sweep and the long-context variants (rank 0 of a single-GPU run only).
    per_config = []
    cores_all = None
    if rank == 0:
        import oracle
        cores_all = oracle.load().max_threads()
    if args.per_config == "on" or (args.per_config == "auto" and world == 1 and w.name == DEFAULT_WORKLOAD
                                   and args.n_new is None and args.layout == "contiguous" and args.cache == "same"):
        del step_graph, attn_graph
        torch.cuda.synchronize()
        specs = [("gpt2s_1layer_p16_f32", None, {}), ("gpt2s_12layer_p1000_f32", None, {})]
        specs += [("gpt2s_chunked_p512_f32", n, {}) for n in wl.CHUNKED_N]
        specs += [("gpt2s_b8_p1023_bf16", None, {}), ("gpt2s_b8_p1023_bf16", None, {"layout": "paged"})]
        # The same steps through kvd_decode_step_flags(KVD_STEP_HISTORY_STABLE): in this
        # step nothing writes past_len or a layer's history between the layers' calls.
        stable = {"flags": kvd_stable_flag()}
        specs += [("gpt2s_12layer_p1000_f32", None, stable), ("gpt2s_chunked_p512_f32", 16, stable),
                  ("gpt2s_b8_p1023_bf16", None, stable)]
        for name, n, opts in specs:
            wc = wl.WORKLOADS[name] if n is None else wl.with_n(wl.WORKLOADS[name], n)
            c = Case(wc, dev, **opts)
            label = wc.describe() + (" (paged)" if "layout" in opts else "") + \
                (" (kvd_decode_step_flags: history stable)" if "flags" in opts else "")
            per_config.append(per_config_line(c, timer, args.steps, world, label, cores_all,
                                              with_oracle=rank == 0 and not opts))
            del c
            torch.cuda.empty_cache()
        for n in (8,):  # the chunked decode over the long-context caches: tcgen05, 32 rows per KV head
            c = Case(wl.with_n(w, n), dev, reuse=case)
            per_config.append(per_config_line(c, timer, args.steps, world, f"{w.name} N={n} (same caches)",
                                              cores_all, with_oracle=False))
            del c
        c = Case(w, dev, cache="e4m3")
        per_config.append(per_config_line(c, timer, args.steps, world, f"{w.name} with an E4M3 cache",
                                          cores_all, with_oracle=False))
        del c
        torch.cuda.empty_cache()
    t_wall2 = time.time()
    if rank == 0:
        sampler.stop()
    if rank != 0:
        return

    peak, peak_kind = measured_peak()
    gbs = whole_job_gbs(case.step_bytes, passes, elapsed_max, world)
    ms_step = elapsed_max / args.steps * 1e3
    lb = layer_bytes(w, case.past.tolist(), case.cache_elem)
    a_bytes = lb if case.fused else attn_bytes(w, case.past.tolist(), case.cache_elem)
    achieved = a_bytes / attn_per_launch / 1e9

    # CPU baseline: the oracle on layer 0's data, all host cores (~cpu_seconds), and once on one core
    host = {k: to_host_np(v) for k, v in case.layers[0].items()}
    reps, cpu_el, cores = time_oracle(w, host, case.past, budget_s=args.cpu_seconds)
    cpu_gbs = reps * lb / cpu_el / 1e9
    one = oracle_times(case, cores, reps_all=0, reps_one=1)["one_core"] if args.cpu_one_core else None

    config = config_block(w, case.past.tolist(), world, args.layout, args.page_size, args.page_order, args.cache)
    config["step"] = ((f"{replays} replay(s) of one CUDA graph of " if replays > 1 else "one CUDA graph of ") +
                      (f"{w.L} x kvd_decode_step (append + attention in one launch)" if case.fused else
                       f"{w.L} x (kvd_append + kvd_decode_attention)") + " on one stream")
    config["l2"] = ((f"flushed: {2 * timer.l2_bytes / 1e6:.0f} MB written before each timed step, outside its "
                     f"events ({case.step_bytes / 1e6:.1f} MB per step; e2e not flushed)") if flush else
                    f"no flush: inputs larger than L2 ({case.step_bytes / 1e9:.1f} GB per pass of the layers)")
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
        "config": config,
        "replays_per_step": replays,
        "timed_seconds": round(elapsed_max, 3),
        "us_per_layer_step": round(elapsed_max / passes / w.L * 1e6, 3),
        "frac_of_peak": round(gbs / world / peak, 4),
        "attn_us_per_layer": round(attn_per_launch * 1e6, 3),
        "path": args.path,
        "roofline": {
            "bound": "hbm",
            "kernel": ("kvd_decode_step (fused append + split-T attention" if case.fused else
                       "kvd_decode_attention (split-T attention") + (" + LSE merge)" if case.plan["launches"] == 2 else ")"),
            "timing": "graph of the L calls replayed, CUDA events on its stream",
            "achieved": round(achieved, 2),
            "peak": peak,
            "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, copy burst)" if peak_kind == "measured" else "fallback",
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "algorithmic_bytes_per_launch": a_bytes,
            "plan": case.plan,
            "traffic": None if (case.paged or case.e4m3) else profiled_traffic(),
        },
        "cpu_baseline": {
            "value": round(cpu_gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"layer 0 of {w.name} (all {w.B} sequences, append + attention, fp64), "
                      f"repeated {reps}x in {cpu_el:.1f} s",
            "ms_per_layer_step": round(cpu_el / reps * 1e3, 3),
            "one_core": one,
        },
        "e2e": e2e,
        "memory": mem,
        "gpu_launches": passes * w.L * case.launches_per_layer,
        "clocks": clocks,
        "clocks_whole_run": sampler.summary(t_wall0, t_wall2),
        "per_config": per_config,
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
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="each timed step replays the step graph often enough that the timed region "
                         "spans at least this long (workloads larger than twice the L2)")
    ap.add_argument("--per-config", default="auto", choices=["auto", "on", "off"],
                    help="also time the other workloads (auto: single-GPU default runs)")
    ap.add_argument("--no-cpu-one-core", dest="cpu_one_core", action="store_false",
                    help="skip the one-core oracle time")
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
