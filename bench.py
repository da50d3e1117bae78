#!/usr/bin/env python
"""Benchmark of ragged paged attention on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl reference] [--no-cpu-baseline] [--no-configs]

One step = one rpa_forward over one synthetic batch (planner, decode kernel,
prefill kernel; the page write is fused into the two attention kernels).
Inputs are resident in HBM when the timed region starts; L2 is flushed (a 512 MB
write) before every timed step, outside its events.  Each step is timed
with two CUDA events on the launching stream (the attention kernels are
programmatic dependents of the kernel before them, so no event sits between
them); each kernel's own time comes from a second set of steps run through
rpa_forward_timed, whose events sit between the kernels.  With N > 1 (torchrun) every rank runs an
independent replica ("replicas only": the op has no exchange step), the time
is the max over ranks, and value counts the tokens of all ranks.

The default run times the decode workload (the headline: value, e2e,
roofline) and then, under "configs", the mixed, long, long_w4096, fp8,
fp8_w8a8, decode_d256 and long_d256 workloads, each with its own step time,
kernel times, clocks and per-kernel rooflines.

Prints ONE JSON line (rank 0).  --impl reference times the CPU oracle instead
(on the host cores, a bounded sample of the same workload per step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "RPA tokens/s; decode KV HBM GB/s & prefill TFLOP/s vs GB300 peak"
L2_FLUSH_BYTES = 512 << 20

DESCRIPTIONS = {
    "decode": "decode-heavy, Llama-3-8B attention shape: 256 seqs q_len=1, kv_len~U[512,4096]; "
              "Hq32/Hkv8/D128, bf16 cache, page_size 16, 80000-page pool",
    "mixed": "chunked-prefill mixed batch: 128 decode (kv~U[1024,8192]) + 8x512-token chunks "
             "(prior kv~U[0,4096]) + 2x1536 fresh; Hq64/Hkv8/D128, bf16, page_size 32",
    "long": "long-context prefill: 2 seqs q=kv=32768 causal; Hq32/Hkv8/D128, bf16, page_size 64",
    "long_w4096": "long-context prefill: 2 seqs q=kv=32768, sliding_window 4096; "
                  "Hq32/Hkv8/D128, bf16, page_size 64",
    "fp8": "fp8 e4m3 cache (k/v scale 0.05), soft cap 30, sinks, window 128: 512 decode "
           "(kv~U[256,16384]) + 8x256 chunks (prior kv~U[0,8192]); Hq64/Hkv8/D64, page_size 16",
    "fp8_w8a8": "the fp8 batch with quantised queries (q_scale 0.02, w8a8): Q K^T of the "
                "prefill on the e4m3 codes",
    "decode_small": "decode shape at 64 seqs (profiling size): q_len=1, kv_len~U[512,4096]; "
                    "Hq32/Hkv8/D128, bf16, page_size 16, pool = pages used + 10%",
    "long_small": "long-context shape at profiling size: 1 seq q=kv=8192 causal; Hq32/Hkv8/D128, "
                  "bf16, page_size 64",
    "long_small_fp8": "long_small with an e4m3 cache (k/v scale 0.05): 1 seq q=kv=8192 causal; "
                      "Hq32/Hkv8/D128, page_size 64 (profiling size)",
    "long_small_fp8_w8a8": "long_small_fp8 with quantised queries (q_scale 0.02): Q K^T of the "
                           "prefill on e4m3 codes (profiling size)",
    "fp8_small": "fp8 shape at profiling size: 64 decode + 8x256 chunks; e4m3 cache, cap 30, "
                 "sinks, window 128; Hq64/Hkv8/D64, page_size 16",
    "tiny": "tiny mixed batch: 3 seqs (1,17),(24,24),(5,40); Hq4/Hkv2/D64/P16",
    "decode_d256": "decode, Gemma-2-9B attention shape (head_dim 256): 256 seqs q_len=1, "
                   "kv_len~U[512,4096]; Hq16/Hkv8/D256, window 4096, soft cap 50, scale 1/16, "
                   "bf16 cache, page_size 16, pool = pages used + 10%",
    "decode_d256_small": "decode_d256 shape at 64 seqs (profiling size)",
    "long_d256": "long causal prefill at head_dim 256: 2 seqs q=kv=8192; Hq16/Hkv8/D256, "
                 "scale 1/16, bf16 cache, page_size 64",
}


# ------------------------------------------------------------ work counting
def classify(w):
    """Per sequence: True where the planner takes the decode path."""
    d0 = int(w.distribution[0])
    return np.array([s < d0 and int(w.q_lens[s]) == 1 for s in range(w.num_seqs)])


def algorithmic_work(w):
    """Algorithmic HBM bytes and flops of the decode and prefill kernels.

    bytes: every key/value inside the causal/window band read once (cache
    rows 2*Hkv*D*elem per cached key; new tokens read from the bf16 inputs),
    the new tokens' page write, the queries read and the outputs written.
    flops: 4*D*Hq per unmasked (query token, key) pair."""
    H, Hq, D, e = w.num_kv_heads, w.num_q_heads, w.head_dim, w.elem_bytes
    W = w.sliding_window
    dec = classify(w)
    out = {"decode": {"bytes": 0, "flops": 0, "tokens": 0},
           "prefill": {"bytes": 0, "flops": 0, "tokens": 0}}
    for s in range(w.num_seqs):
        q, kv = int(w.q_lens[s]), int(w.kv_lens_valid[s])
        if q == 0:
            continue
        ctx = kv - q
        first = ctx  # position of the first new token
        lo_first = max(0, first - W + 1) if W else 0
        cached_needed = max(0, ctx - lo_first)  # cached keys any token of the seq needs
        pos = np.arange(ctx, kv, dtype=np.int64)
        keys_per_tok = np.minimum(pos + 1, W) if W else pos + 1
        k = out["decode" if dec[s] else "prefill"]
        k["bytes"] += cached_needed * 2 * H * D * e + q * 2 * H * D * (2 + e) + 2 * q * Hq * D * 2
        k["flops"] += int(keys_per_tok.sum()) * 4 * D * Hq
        k["tokens"] += q
    return out


# ------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.path = tempfile.mktemp(prefix="rpa_clocks_", suffix=".csv")
        self.proc = None
        self.dev = device_index
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.4)

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[3], parts[4:]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        # samples under load: the upper half of the SM clock distribution
        sm = [r[0] for r in rows]
        reasons = set()
        names = ("active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap")
        for r in rows:
            for n, v in zip(names[1:], r[3][1:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(r[1] for r in rows),
                "samples": len(rows), "reasons": sorted(reasons)}


# -------------------------------------------------------------------- peaks
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "bf16_tflops": float(pk["bf16_tflops"]),
                "bf16_tflops_sustained": float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def kernel_source_sha(kernel_file: str) -> str:
    """Hash of a kernel's translation unit and every shared header."""
    import glob
    csrc = os.path.join(ROOT, "ragged_paged_attention_kv_gb300", "csrc")
    h = hashlib.sha256()
    for f in [os.path.join(csrc, kernel_file)] + sorted(glob.glob(os.path.join(csrc, "*.cuh"))) + \
            sorted(glob.glob(os.path.join(csrc, "*.h"))) + [os.path.join(ROOT, "include", "rpa.h")]:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_for(kernel_file: str, workload: str):
    """DRAM bytes per launch from a committed ncu capture, if the kernel's
    source is unchanged since the capture; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            table = json.load(f)
        ent = table[workload]
        if ent["source"] != kernel_file or kernel_source_sha(kernel_file) != ent["source_sha"]:
            return None
        return float(ent["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


# --------------------------------------------------------------- GPU arm
def setup_dist(backend: str = "nccl"):
    """(world, rank, local rank) from the torchrun environment; joins the
    process group when there is more than one rank (one GPU per rank with
    NCCL; the host-logic tests use gloo on the CPU)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(x: float, world: int, device: str = "cuda") -> float:
    """The largest x over all ranks (the job's time is its slowest rank's)."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world, cuda: bool = True):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    if cuda:
        torch.cuda.synchronize()


def job_throughput(tokens_per_step: int, world: int, steps: int, seconds: float) -> float:
    """Whole-job tokens/s: every rank runs `steps` steps of `tokens_per_step`
    tokens (weak scaling, replicas), in `seconds` = the max over ranks."""
    return tokens_per_step * world * steps / seconds


def prefill_kernel_name(w):
    """The prefill kernel the library runs for this workload's shape: the
    tcgen05 kernels for pages of at least 8 rows (two query tiles per unit at
    head_dim 64/128, one at 192/256), else the warp-level MMA kernel."""
    if w.page_size >= 8 and w.head_dim in (64, 128):
        return "prefill_tc_kernel", "prefill_tc.cu"
    if w.page_size >= 8 and w.head_dim in (192, 256):
        return "prefill_tc_wide_kernel", "prefill_tc_wide.cu"
    return "prefill_kernel", "prefill.cu"


def launches_per_step(w):
    """The library's kernels one rpa_forward launches: planner, decode and
    prefill kernels, and with an e4m3 cache and a tcgen05 prefill the page
    write of the prefill sequences' new tokens."""
    name, _ = prefill_kernel_name(w)
    return 3 + (1 if w.kv_dtype == "fp8" and name != "prefill_kernel" else 0)


# How each workload is bounded (the roofline each of its kernels is held to).
BOUNDS = {
    "decode": "hbm",
    "decode_d256": "hbm",
    "mixed": "hbm (decode share) + tensor (prefill share); the decode kernel runs on 80 of 152 "
             "the SMs while the prefill kernel starts on the rest, so its time alone (kernel "
             "events) is longer than its share of the overlapped step",
    "long": "tensor",
    "long_w4096": "tensor",
    "long_d256": "tensor",
    "fp8": "hbm, window-limited (67 MB of keys/values in the window): latency-dominated",
    "fp8_w8a8": "as fp8; Q K^T of the prefill on e4m3 codes",
}


def rooflines(w, work, dec_avg, pf_avg, peaks, name=None):
    """Per kernel: achieved vs peak.  The decode kernel is HBM-bound (its
    algorithmic bytes over its event time, against the measured copy
    bandwidth); the prefill kernel is a bf16 contraction (its flops over its
    event time, against the measured burst bf16 GEMM rate: each launch is
    timed alone, after an L2 flush)."""
    r = {}
    if work["decode"]["tokens"]:
        a = work["decode"]["bytes"] / (dec_avg * 1e-3) / 1e9
        r["decode"] = {"bound": "hbm", "kernel": "decode_kernel", "achieved": round(a, 1),
                       "peak": peaks["hbm_gbs"], "unit": "GB/s",
                       "frac": round(a / peaks["hbm_gbs"], 4),
                       "algorithmic_bytes": int(work["decode"]["bytes"]),
                       "ms": round(dec_avg, 4),
                       "traffic": traffic_for("decode.cu", name) if name else None}
    if work["prefill"]["tokens"]:
        a = work["prefill"]["flops"] / (pf_avg * 1e-3) / 1e12
        r["prefill"] = {"bound": "tensor", "kernel": prefill_kernel_name(w)[0],
                        "achieved": round(a, 1), "peak": peaks["bf16_tflops"],
                        "unit": "TFLOP/s", "frac": round(a / peaks["bf16_tflops"], 4),
                        "algorithmic_flops": int(work["prefill"]["flops"]),
                        "ms": round(pf_avg, 4),
                        "traffic": traffic_for(prefill_kernel_name(w)[1], name) if name else None}
    return r


def prepare(w, dev):
    """Device copies of a workload's inputs, its pool, output and workspace."""
    import ragged_paged_attention_kv_gb300 as rpa
    fp8 = w.kv_dtype == "fp8"
    q, k, v = w.make_qkv()
    sink = w.make_sink()
    meta_host = {"kv_lens": torch.from_numpy(w.kv_lens),
                 "block_tables": torch.from_numpy(w.block_tables),
                 "qsl": torch.from_numpy(w.query_start_loc),
                 "dist": torch.from_numpy(w.distribution)}
    ctx = {
        "w": w, "host": (q, k, v, meta_host, sink),
        "dev": (q.to(dev), k.to(dev), v.to(dev), {n: t.to(dev) for n, t in meta_host.items()},
                sink.to(dev) if sink is not None else None),
        "pool": w.make_pool(dev),
        "kw": dict(softmax_scale=w.softmax_scale, sliding_window=w.sliding_window,
                   logits_soft_cap=w.logits_soft_cap, k_scale=w.k_scale if fp8 else None,
                   v_scale=w.v_scale if fp8 else None, q_scale=w.q_scale or None),
    }
    ctx["out"] = torch.empty_like(ctx["dev"][0])
    ctx["ws"] = rpa.alloc_workspace(rpa.make_params(**w.params()), dev)
    return ctx


def step(ctx, events=None, src=None):
    import ragged_paged_attention_kv_gb300 as rpa
    a = src or ctx["dev"]
    rpa.forward(a[0], a[1], a[2], ctx["pool"], a[3]["kv_lens"], a[3]["block_tables"],
                a[3]["qsl"], a[3]["dist"], a[4], out=ctx["out"], workspace=ctx["ws"],
                events=events, **ctx["kw"])


def time_steps(ctx, steps, warmup, flush, stream, world, rank, dev):
    """W warm-up steps, then two sets of K timed steps, each after an L2
    flush.  The step time comes from the first set, bracketed by two events
    on the launching stream only: the decode and prefill kernels are launched
    as programmatic dependents of the kernel before them, and an event
    between two kernels would serialise them.  The second set runs
    rpa_forward_timed, whose four events around the planner, decode and
    prefill kernels give each kernel's time (its sum is a little longer than
    the first set's step).  Returns per-step ms lists and the clocks sampled
    during both sets."""
    import ragged_paged_attention_kv_gb300 as rpa
    for _ in range(warmup):
        flush.zero_()
        step(ctx)
    if rpa.get_status(ctx["ws"]) != 0:
        raise RuntimeError(f"{ctx['w'].name}: device status nonzero after warm-up")

    def events(n, k):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(k)] for _ in range(n)]
        for ev in evs:  # record once so each CUDA event exists before its handle is passed on
            for e in ev:
                e.record(stream)
        return evs

    outer, inner = events(steps, 2), events(steps, 4)
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    if rank == 0:
        clocks.start()
    barrier(world)
    for i in range(steps):
        flush.zero_()
        outer[i][0].record(stream)
        step(ctx)
        outer[i][1].record(stream)
    for i in range(steps):
        flush.zero_()
        step(ctx, events=inner[i])
    barrier(world)
    clk = clocks.stop() if rank == 0 else None
    ms = {"step": [e[0].elapsed_time(e[1]) for e in outer],
          "plan": [e[0].elapsed_time(e[1]) for e in inner],
          "decode": [e[1].elapsed_time(e[2]) for e in inner],
          "prefill": [e[2].elapsed_time(e[3]) for e in inner],
          "step_serialised": [e[0].elapsed_time(e[3]) for e in inner]}
    return ms, clk


def e2e_steps(ctx, steps, flush, stream, world, dev):
    """The same step through the public call from pinned host buffers: every
    step's inputs are packed into one pinned host buffer (each tensor at a
    256-byte aligned offset) and copied with one host-to-device copy, as a
    serving loop stages a step; the output comes back with one device-to-host
    copy.  Both copies are inside the timed region.  Returns (ms per step
    list, h2d bytes, d2h bytes)."""
    q, k, v, meta_host, sink = ctx["host"]
    host_in = [q, k, v, *meta_host.values()] + ([sink] if sink is not None else [])
    offs, total = [], 0
    for t in host_in:
        offs.append(total)
        total += -(-(t.numel() * t.element_size()) // 256) * 256
    hbuf = torch.empty(total, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(total, dtype=torch.uint8, device=dev)

    def view(buf, t, off):
        n = t.numel() * t.element_size()
        return buf[off:off + n].view(t.dtype).view(t.shape)

    for t, off in zip(host_in, offs):
        view(hbuf, t, off).copy_(t)
    dviews = [view(dbuf, t, off) for t, off in zip(host_in, offs)]
    src = (dviews[0], dviews[1], dviews[2],
           dict(zip(meta_host.keys(), dviews[3:3 + len(meta_host)])),
           dviews[-1] if sink is not None else None)
    out = ctx["out"]
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = hout.numel() * hout.element_size()
    ms = []
    barrier(world)
    for _ in range(steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dbuf.copy_(hbuf, non_blocking=True)
        step(ctx, src=src)
        hout.copy_(out, non_blocking=True)
        e1.record(stream)
        e0.synchronize()
        e1.synchronize()
        ms.append(e0.elapsed_time(e1))
    barrier(world)
    return ms, h2d, d2h


def measure(name, args, world, rank, dev, flush, stream, with_e2e):
    """One workload: timed steps, per-kernel rooflines, clocks (and the
    end-to-end leg when asked).  Returns (result dict, workload)."""
    w = wl.get(name)
    work = algorithmic_work(w)
    ctx = prepare(w, dev)
    ms, clk = time_steps(ctx, args.steps, args.warmup, flush, stream, world, rank, dev)
    total_s = max_over_ranks(sum(ms["step"]) / 1e3, world)
    tokens = w.num_query_tokens
    dec_avg, pf_avg = statistics.mean(ms["decode"]), statistics.mean(ms["prefill"])
    peaks = load_peaks()
    res = {
        "workload": f"{name}: {DESCRIPTIONS[name]}",
        "value": round(job_throughput(tokens, world, args.steps, total_s), 1),
        "unit": "tokens/s", "tokens_per_step": tokens,
        "ms_per_step": round(total_s * 1e3 / args.steps, 4),
        "kernels_ms": {"plan": round(statistics.mean(ms["plan"]), 4),
                       "decode": round(dec_avg, 4), "prefill": round(pf_avg, 4),
                       "step_with_kernel_events": round(statistics.mean(ms["step_serialised"]), 4)},
        "bound": BOUNDS.get(name, "hbm" if not work["prefill"]["tokens"] else "tensor"),
        "rooflines": rooflines(w, work, dec_avg, pf_avg, peaks, name),
        "decode_kv_gbs": round(work["decode"]["bytes"] / (dec_avg * 1e-3) / 1e9, 1)
        if work["decode"]["tokens"] else None,
        "prefill_tflops": round(work["prefill"]["flops"] / (pf_avg * 1e-3) / 1e12, 2)
        if work["prefill"]["tokens"] else None,
        "kv_dtype": w.kv_dtype, "clocks": clk, "peak_source": peaks["source"],
    }
    if with_e2e:
        e2e_ms, h2d, d2h = e2e_steps(ctx, args.steps, flush, stream, world, dev)
        e2e_s = max_over_ranks(sum(e2e_ms) / 1e3, world)
        res["e2e"] = {"value": round(job_throughput(tokens, world, args.steps, e2e_s), 1),
                      "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
                      "d2h_bytes_per_step": int(d2h),
                      "ms_per_step": round(e2e_s * 1e3 / args.steps, 4)}
    del ctx
    torch.cuda.empty_cache()
    return res, w


# The configurations timed after the headline in the default run: the other
# single-GPU configurations the metric is quoted on, plus head_dim 256.
EXTRA_CONFIGS = ("mixed", "long", "long_w4096", "fp8", "fp8_w8a8", "decode_d256", "long_d256")


def gpu_arm(args, world, rank, local):
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    head, w = measure(args.workload, args, world, rank, dev, flush, stream, with_e2e=True)

    # ---- roofline of the headline's dominant kernel
    rl = head["rooflines"]
    dominant = "decode" if "decode" in rl and (
        "prefill" not in rl or rl["decode"]["ms"] >= rl["prefill"]["ms"]) else "prefill"
    roof = {k_: rl[dominant][k_] for k_ in ("bound", "achieved", "peak", "unit", "frac")}
    kfile = "decode.cu" if dominant == "decode" else prefill_kernel_name(w)[1]
    roof["traffic"] = traffic_for(kfile, args.workload)
    roof["kernel"] = rl[dominant]["kernel"]
    roof["peak_source"] = head["peak_source"]
    roof["peak_kind"] = "measured copy bandwidth" if dominant == "decode" else \
        "measured bf16 GEMM, burst (kernel timed alone)"

    configs = {}
    if args.workload == "decode" and not args.no_configs:
        for name in EXTRA_CONFIGS:
            configs[name], _ = measure(name, args, world, rank, dev, flush, stream,
                                       with_e2e=False)

    res = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": head["workload"], "tokens_per_step": head["tokens_per_step"],
                   "l2": "flushed before every timed step (512 MB write, outside the events; "
                         "it also lets the host queue the step)",
                   "parallelism": f"replicas x{world}", "kv_dtype": head["kv_dtype"]},
        "roofline": roof,
        "kernels_ms": head["kernels_ms"],
        "decode_kv_gbs": head["decode_kv_gbs"],
        "prefill_tflops": head["prefill_tflops"],
        "e2e": head["e2e"],
        "gpu_launches": launches_per_step(w) * args.steps,
        "clocks": head["clocks"],
    }
    if configs:
        res["configs"] = configs
    return res, w


# --------------------------------------------------------------- CPU oracle
def oracle_sample(w, budget_s: float, seed: int = 0, nthreads: int = 0):
    """Times the oracle on a seeded sample of the workload's sequences: the
    page write plus the attention of every new token of each sampled
    sequence (a seeded sample of rows for long prefills), adding sequences
    until about budget_s of CPU time has been spent.  Returns (tokens/s,
    threads used, description of the sample)."""
    import oracle
    rng = np.random.default_rng(seed)
    order = rng.permutation(w.num_seqs)
    q_all, k_all, v_all = _qkv(w)
    sink = w.make_sink()
    done_tokens, spent, n_seqs, passes = 0, 0.0, 0, 0
    rows_note = "all new tokens of each"
    prepared = _PREPARED.setdefault(w.name, {})
    # Sequences are taken in a seeded order; when every sequence has been
    # visited before the budget is spent, the order is walked again so that
    # the sample always holds about budget_s of oracle work.
    while spent < budget_s:
        visited = 0
        for s in order:
            if spent >= budget_s:
                break
            s = int(s)
            if int(w.q_lens[s]) == 0:
                continue
            entry = prepared.get(s)
            if entry is None:
                sub, sub_pool, tmap = w.subset([s], None)
                idx = torch.as_tensor(tmap)
                q_len = int(w.q_lens[s])
                keys = (min(int(w.kv_lens_valid[s]), w.sliding_window) if w.sliding_window
                        else int(w.kv_lens_valid[s]))
                rows = np.arange(q_len)
                if q_len * keys > 4_000_000:  # long prefill: a seeded sample of its rows
                    n = max(1, 4_000_000 // max(1, keys))
                    rows = np.unique(rng.integers(0, q_len, size=n))
                    rows_note = "all new tokens of each (a seeded row sample for long prefills)"
                cache = sub_pool.contiguous().view(torch.uint8).numpy().reshape(-1).copy()
                entry = (sub, oracle.make_params(**sub.params()), q_all[idx], k_all[idx],
                         v_all[idx], cache, rows)
                # compact pools are kept across calls (every step of the
                # reference arm samples the same workload), up to 4 GiB
                if _PREPARED_BYTES[0] + cache.nbytes <= 4 << 30:
                    prepared[s] = entry
                    _PREPARED_BYTES[0] += cache.nbytes
            # Writing a sequence's new tokens again stores the same bytes, so a
            # held pool serves every later pass unchanged.
            sub, p, q, k, v, cache, rows = entry
            t0 = time.perf_counter()
            cache = oracle.update_cache(p, k, v, cache, sub.kv_lens, sub.block_tables,
                                        sub.query_start_loc, sub.num_seqs)
            oracle.attention_rows(p, q, cache, sub.kv_lens, sub.block_tables, sub.query_start_loc,
                                  sub.num_seqs, rows, None if sink is None else sink.numpy(), nthreads)
            spent += time.perf_counter() - t0
            done_tokens += len(rows)
            n_seqs += 1
            visited += 1
        passes += 1
        if visited == 0:
            break
    value = done_tokens / spent if spent > 0 else 0.0
    desc = (f"{n_seqs} sequence passes over {min(n_seqs, w.num_seqs)} of {w.num_seqs} "
            f"sequences (seeded order, {passes} walk(s) of the order), {rows_note}: "
            f"{done_tokens} tokens in {spent:.1f} s")
    return value, oracle.max_threads(), desc


_QKV_CACHE = {}
_PREPARED = {}          # workload name -> {sequence: prepared oracle inputs}
_PREPARED_BYTES = [0]   # bytes of compact pools held in _PREPARED


def _qkv(w):
    if w.name not in _QKV_CACHE:
        _QKV_CACHE[w.name] = w.make_qkv()
    return _QKV_CACHE[w.name]


def reference_arm(args, world, rank):
    """The oracle as the reference arm: each step is a bounded sample."""
    if rank != 0:
        return None
    w = wl.get(args.workload)
    per_step = max(0.2, min(6.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(w, per_step, seed=0)
    vals = []
    t0 = time.perf_counter()
    for i in range(args.steps):
        val, cores, desc = oracle_sample(w, per_step, seed=1 + i)
        vals.append(val)
    wall = time.perf_counter() - t0
    value = statistics.mean(vals)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(wall * 1e3 / max(1, args.steps), 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {DESCRIPTIONS[args.workload]}",
                   "parallelism": "host cores (OpenMP)"},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores,
                         "kind": "oracle", "sample": f"per step ~{per_step:.1f} s: {desc}"},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="decode", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="time only the headline workload (skip the other configurations)")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        res = reference_arm(args, world, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return 0

    world, rank, local = setup_dist()
    if world != args.gpus and rank == 0:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    res, w = gpu_arm(args, world, rank, local)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            val, cores, desc = oracle_sample(w, args.cpu_budget)
            res["cpu_baseline"] = {"value": round(val, 3), "unit": "tokens/s", "cores": cores,
                                   "kind": "oracle", "sample": desc}
        else:
            res["cpu_baseline"] = None
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
