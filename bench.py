#!/usr/bin/env python3
"""Benchmark of the fused attention forward on the headline workload.

One step = one attn_fwd call over the whole workload (B=2, H=32, Hkv=8, N=8192, d=128, causal,
bf16 by default). Prints ONE JSON line on rank 0:
  value      device-timed TFLOP/s (4*B*H*N^2*d, halved for causal), summed over ranks, with
             inputs resident in HBM; CUDA events around each launch on the launching stream,
             L2 flushed (256 MiB write, then a 256 MiB read that drains the dirty lines) before
             every step, outside the events. The timed region is --repeats (default 5) repeats
             of exactly --steps steps, each bracketed by a barrier and a synchronize; value,
             ms_per_step and the roofline come from the median repeat, and every repeat's
             ms per step is listed;
  e2e        the same metric through attn_fwd_host (pinned host buffers, H2D of q/k/v and D2H
             of o/lse inside the timed region), the median of --repeats repeats of --steps calls;
  roofline   tensor-core bound: achieved TFLOP/s of the attention kernel against the measured
             dense bf16 peak (e4m3: x2 nominal ratio). A non-causal call whose last wave is halved
             along the keys runs the kernel as two launches; the step time covers both;
  cpu_baseline  the fp64 oracle on a bounded sample, on this host's cores (rank 0, N=1 only);
  clocks     nvidia-smi SM clock samples taken during the timed region.
--impl reference times the oracle itself (CPU) on bounded samples of the same workload.
Multi-GPU (torchrun): every rank runs its own replica of the workload (weak scaling); time is
the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attn fwd TFLOP/s (bf16, causal, N=8192, d=128) and % of GB300 dense peak"
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20
DECODE_NAMES = {"decode_gqa_bf16_nq1_nk16384_d128", "decode_gqa_bf16_nq16_nk8192_d128"}


class L2Flush:
    """Evicts the step's inputs from L2 before a timed step: writes a buffer larger than L2, then
    reads a second one. The read makes the write's dirty lines drain to DRAM here, outside the
    timed events, instead of during the next step's kernel."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def __call__(self, i: int):
        self.w.fill_(i & 0xFF)
        self.r.max()


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--repeats", type=int, default=5,
                    help="timed repeats of --steps steps each; the reported figures are the median repeat's")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None, help="name from exact_attention_72_gb300.inputs.WORKLOADS")
    ap.add_argument("--batch", type=int, default=None, help="override B (smaller cases for profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU-baseline time box")
    ap.add_argument("--oracle-full", action="store_true",
                    help="with --impl reference: run the oracle once over the whole workload (every head, every "
                         "row) and report its wall time, not the bounded per-step samples")
    return ap.parse_args(argv)


# ------------------------------------------------------------------------------------------ ranks
def rank_info():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def init_dist(world):
    if world <= 1:
        return None
    import torch.distributed as dist
    dist.init_process_group("gloo")
    return dist


def max_over_ranks(dist, value: float) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ------------------------------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples SM clock and throttle reasons with nvidia-smi while the timed region runs."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.samples = []   # (host time, [fields])
        self.error = None
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError as e:
            self.error = str(e)
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.samples.append((time.time(), parts))

    def wait_first(self, timeout=5.0):
        t0 = time.time()
        while not self.samples and self.proc is not None and time.time() - t0 < timeout:
            time.sleep(0.02)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if self.error or not self.samples:
            return {"error": self.error or "no nvidia-smi samples"}
        inside = [s for (t, s) in self.samples if t0 <= t <= t1 + 0.06]
        note = None
        if not inside:
            after = [s for (t, s) in self.samples if t >= t0]
            inside = after[:3]
            note = "timed region shorter than the sampling interval; nearest samples after its start"
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[0]) for s in inside if num(s[0]) is not None]
        mx = [num(s[1]) for s in inside if num(s[1]) is not None]
        reasons = sorted({self.REASONS[i] for s in inside for i in range(4) if s[3 + i].lower() == "active"})
        out = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
               "reasons": reasons, "samples": len(inside)}
        if note:
            out["note"] = note
        return out


# ------------------------------------------------------------------------------------------ helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback (1.9 PFLOP/s bf16 burst, earlier GB300 measurement)"


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy)"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback (6.8 TB/s, earlier GB300 measurement)"


# Sources the forward kernel's device code is built from: a change to any of them voids the
# committed DRAM-traffic figures (host-side files and other kernels do not).
FWD_KERNEL_SOURCES = ("attn_fwd_kernel.cuh", "ptx.cuh", "varlen.cuh", "launch_impl.cuh", "attn_fwd_bf16_d128.cu",
                      "attn_fwd_bf16_d64.cu", "attn_fwd_bf16_d256.cu", "attn_fwd_fp8_d128.cu", "attn_fwd_fp8_d64.cu")


def _code_only(text: str) -> str:
    """The source without comments, blank lines or trailing blanks: edits to comments alone leave
    the hash, and so the committed traffic figures, in force."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in FWD_KERNEL_SOURCES:
        with open(os.path.join(ROOT, "exact_attention_72_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(name.encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def measured_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this source."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("kernel_source_sha") != kernel_source_hash():
        return None
    return t.get("bytes_per_launch", {}).get(workload)


def credited_flops(w, rows, N):
    """Metric FLOPs for the given query rows (causal rows see i+1 keys, else N)."""
    if w.causal:
        return 4.0 * w.d * sum(int(r) + 1 for r in rows)
    return 4.0 * w.d * N * len(rows)


def timed_repeats(args, dist, stream, flush, step, with_mid=False):
    """args.repeats repeats of exactly args.steps timed steps. Each repeat is bracketed by a
    barrier and a synchronize on both sides; every step is preceded by an L2 flush outside its
    CUDA events. step(i, mid) runs step i and, when with_mid is set, records the event `mid`
    inside it. Returns (durations [R][K] in ms, start-to-mid durations or None, per-repeat
    totals taken as the max over ranks, index of the median repeat, host start, host end)."""
    import torch
    R, K = max(1, args.repeats), args.steps
    reps = []
    t_host0 = None
    for r in range(R):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3 if with_mid else 2)] for _ in range(K)]
        barrier(dist)
        torch.cuda.synchronize()
        if t_host0 is None:
            t_host0 = time.time()
        for i in range(K):
            flush(i)
            ev[i][0].record(stream)
            step(i, ev[i][2] if with_mid else None)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        barrier(dist)
        reps.append(ev)
    t_host1 = time.time()
    durs = [[e[0].elapsed_time(e[1]) for e in ev] for ev in reps]
    mids = [[e[0].elapsed_time(e[2]) for e in ev] for ev in reps] if with_mid else None
    totals = [max_over_ranks(dist, sum(d)) for d in durs]
    med = sorted(range(R), key=lambda r: totals[r])[R // 2]
    return durs, mids, totals, med, t_host0, t_host1


def timed_e2e(args, dist, stream, step):
    """End-to-end timing: args.repeats repeats of args.steps calls of step(), each repeat
    bracketed by a barrier and a synchronize and timed with CUDA events on `stream`; the repeat
    totals are maxed over ranks. Returns (ms per step of the median repeat, ms per step of every
    repeat), so a stall of the host in one repeat does not set the figure."""
    import torch
    per = []
    for _ in range(max(1, args.repeats)):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(dist)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(dist)
        per.append(max_over_ranks(dist, e0.elapsed_time(e1)) / args.steps)
    return sorted(per)[len(per) // 2], per


def cpu_oracle_sample(w, x, seconds: float, block_rows=512, max_steps=None):
    """Runs the oracle on row blocks of successive heads until the time box is used up.

    Returns (TFLOP/s credited by the metric's convention, description, seconds, steps)."""
    import numpy as np
    import oracle
    g = w.H // w.Hkv
    flops = 0.0
    elapsed = 0.0
    steps = 0
    n_blocks = max(1, w.N // block_rows)
    blocks_done = []
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    i = 0
    cache = {}
    while (elapsed < seconds) and (max_steps is None or steps < max_steps):
        b, h = heads[i % len(heads)]
        blk = (i * 7) % n_blocks
        i += 1
        r0 = blk * block_rows
        rows = np.arange(r0, min(w.N, r0 + block_rows))
        key = (b, h)
        if key not in cache:
            cache.clear()
            if w.dtype == "fp8_block":
                # the oracle's own block quantisation of this head (q, k rotated), then attention of
                # the dequantised values: the rotated q' k'^T equals the scores of the rotation's inputs
                from oracle import fp8_quant as fq
                signs = fp8_block_signs(w).double().numpy()

                def blocks(t, hh, rows, sg):
                    a = t[b:b + 1, :, hh:hh + 1, :].float().double().numpy()
                    c, ds = fq.quantize_blocks(a, rows, sg)
                    return fq.dequantize_blocks(c, ds, rows)[0, :, 0, :]
                cache[key] = (blocks(x.q, h, 128, signs), blocks(x.k, h // g, 64, signs),
                              blocks(x.v, h // g, w.n_keys, None))
            else:
                def f64(t, hh, s):
                    a = t[b, :, hh, :].float().double().numpy()
                    return a * np.float64(np.float32(s)) if t.element_size() == 1 else a
                cache[key] = (f64(x.q, h, x.descale_q), f64(x.k, h // g, x.descale_k),
                              f64(x.v, h // g, x.descale_v))
        q, k, v = cache[key]
        t0 = time.perf_counter()
        oracle.attention_head(q, k, v, w.scale, w.causal, rows=rows)
        elapsed += time.perf_counter() - t0
        flops += credited_flops(w, rows, w.n_keys)
        blocks_done.append((b, h, int(r0)))
        steps += 1
    desc = (f"{steps} blocks of {block_rows} query rows (full score rows, fp64) from heads of the "
            f"{w.name} workload; FLOPs credited by the metric's convention")
    return (flops / elapsed / 1e12 if elapsed > 0 else 0.0), desc, elapsed, steps


def fp8_block_signs(w):
    """Random signs of the Hadamard rotation of the block-scaled e4m3 workload."""
    from exact_attention_72_gb300 import inputs
    return inputs.hadamard_signs(w.d, w.seed + 7)


def cpu_model() -> str:
    """CPU model of this host (lscpu's model name, else /proc/cpuinfo's)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def run_reference_full(args, w, x):
    """The oracle over the whole workload, timed once on this host's cores (rank 0 only)."""
    import numpy as np
    import torch
    import oracle
    rank, _, _ = rank_info()
    if rank != 0:
        return
    torch.set_num_threads(cores_used())
    g = w.H // w.Hkv
    t_all = 0.0
    for b in range(w.B):
        for h in range(w.H):
            def f64(t, hh, sc):
                a = t[b, :, hh, :].float().double().numpy()
                return a * np.float64(np.float32(sc)) if t.element_size() == 1 else a
            q, k, v = f64(x.q, h, x.descale_q), f64(x.k, h // g, x.descale_k), f64(x.v, h // g, x.descale_v)
            t0 = time.perf_counter()
            oracle.attention_head(q, k, v, w.scale, w.causal)
            t_all += time.perf_counter() - t0
    line = {"impl": "reference", "metric": METRIC, "value": w.flops / t_all / 1e12, "unit": "TFLOP/s",
            "oracle_full": {"wall_s": t_all, "gflops": w.flops / t_all / 1e9, "cores": cores_used(),
                            "cpu_model": cpu_model(), "flops_credited": w.flops,
                            "what": "oracle.attention_head over every (batch, head) and every query row, fp64"},
            "config": config_of(w)}
    print(json.dumps(line), flush=True)


def cores_used() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------------------------------------ arms
def run_reference(args, w, x):
    rank, world, _ = rank_info()
    if rank != 0:
        return
    block = 256
    # warm-up steps (untimed), then K timed steps, each one oracle row block
    if args.warmup > 0:
        cpu_oracle_sample(w, x, seconds=1e9, block_rows=block, max_steps=args.warmup)
    tflops, desc, secs, steps = cpu_oracle_sample(w, x, seconds=1e9, block_rows=block, max_steps=args.steps)
    line = {
        "impl": "reference", "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / max(1, steps) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w),
        "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
                         "sample": "each step: " + desc},
        "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def config_of(w):
    extra = {"Nk": w.n_keys, "splits": w.splits} if w.name in DECODE_NAMES else {}
    if w.dtype == "fp8_block":
        extra = {"quantisation": "per step on the GPU: q e4m3 blocks of 128 rows and k of 64 rows after a "
                                 "random Hadamard rotation, v one descale per head"}
    return {"workload": w.name, "B": w.B, "H": w.H, "Hkv": w.Hkv, "N": w.N, "d": w.d, "causal": w.causal, **extra,
            "qkv_dtype": w.dtype, "k_outliers": w.k_outlier_frac,
            "l2": "flushed before every step (256 MiB write, then a 256 MiB read that drains its dirty lines; outside the timed events)",
            "parallelism": "replicas (one full workload per GPU)"}


def run_ours(args, w, x):
    import torch
    from exact_attention_72_gb300 import binding, build
    rank, world, local = rank_info()
    dist = init_dist(world)
    build.build()
    binding.lib()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fp8 = w.dtype in ("fp8_e4m3", "fp8_block")
    block = w.dtype == "fp8_block"
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    kw = {}
    if w.dtype == "fp8_e4m3":
        kw = {n: torch.tensor([s], dtype=torch.float32, device=dev)
              for n, s in (("descale_q", x.descale_q), ("descale_k", x.descale_k), ("descale_v", x.descale_v))}
    o = torch.empty((w.B, w.N, w.H, w.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()
    decode = w.name in DECODE_NAMES
    if decode:
        if w.splits == 0:   # the library's split heuristic (about one wave of SMs)
            w = w.replace(splits=binding.attn_splitkv_num_splits(w.B, w.H, w.Hkv, w.N, w.n_keys, w.d))
        ws = torch.empty(binding.attn_fwd_splitkv_workspace_bytes(w.B, w.H, w.N, w.d, w.splits), dtype=torch.uint8,
                         device=dev)

    if block:
        signs = fp8_block_signs(w).to(dev)
        q8, k8, v8 = (torch.empty(t.shape, dtype=torch.float8_e4m3fn, device=dev) for t in (q, k, v))
        dq = torch.empty((w.B, w.H, -(-w.N // 128)), dtype=torch.float32, device=dev)
        dk = torch.empty((w.B, w.Hkv, -(-w.N // 64)), dtype=torch.float32, device=dev)
        dv = torch.empty((w.B, w.Hkv, 1), dtype=torch.float32, device=dev)
    def step(i=None, mid=None):
        if decode:
            binding.attn_fwd_splitkv(q, k, v, w.splits, scale=w.scale, workspace=ws, out=o, lse=lse, **kw)
        elif block:
            binding.quantize_e4m3(q, 128, signs, out=q8, descale=dq)
            binding.quantize_e4m3(k, 64, signs, out=k8, descale=dk)
            binding.quantize_e4m3(v, w.N, out=v8, descale=dv)
            if mid is not None:
                mid.record(stream)
            binding.attn_fwd_fp8_blockscaled(q8, k8, v8, w.causal, dq, dk, dv.view(w.B, w.Hkv), scale=w.scale,
                                             out=o, lse=lse)
        else:
            binding.attn_fwd(q, k, v, causal=w.causal, scale=w.scale, out=o, lse=lse, **kw)

    for i in range(max(args.warmup, 0)):
        flush(i)
        step()
    torch.cuda.synchronize()
    st, detail = binding.attn_get_status()
    if st != binding.ATTN_OK:
        raise RuntimeError(f"device status {st} ({detail:#x}) after warm-up")

    sampler = ClockSampler(local)
    sampler.wait_first()
    durs_all, mids_all, totals, med, t_host0, t_host1 = timed_repeats(args, dist, stream, flush, step,
                                                                     with_mid=block)
    time.sleep(0.12)
    sampler.stop()
    durs = durs_all[med]   # ms per step, median repeat
    prepass = None
    if block:
        # the attention launch alone (the roofline's kernel), and the quantisation before it
        pre = mids_all[med]
        durs_attn = [d_ - m_ for d_, m_ in zip(durs, pre)]
        pre_ms = statistics.fmean(pre)
        qkv_bytes = (w.B * w.N * (w.H + 2 * w.Hkv) * w.d) * 3 + 4 * (dq.numel() + dk.numel() + dv.numel())
        hbm, hbm_src = hbm_peak()
        prepass = {"kernel": "quantize_kernel (q, k rotated; v per head)", "ms": pre_ms,
                   "algorithmic_bytes": qkv_bytes, "GB/s": qkv_bytes / (pre_ms * 1e-3) / 1e9,
                   "frac_hbm": qkv_bytes / (pre_ms * 1e-3) / 1e9 / hbm, "peak_source": hbm_src}
    st, detail = binding.attn_get_status()
    if st != binding.ATTN_OK:
        raise RuntimeError(f"device status {st} ({detail:#x}) after the timed region")
    total_ms = totals[med]
    value = w.flops * args.steps * world / (total_ms * 1e-3) / 1e12
    kdurs = durs_attn if block else durs
    mean_ms = statistics.fmean(kdurs)
    achieved = w.flops / (mean_ms * 1e-3) / 1e12
    peak_bf16, peak_src = peaks()
    peak = peak_bf16 * (2.0 if fp8 else 1.0)
    if fp8:
        peak_src += " x2 (e4m3/bf16 nominal dense ratio)"
    if decode:
        # Few query rows against a long KV sequence: bound by reading K and V once from HBM.
        gbs = w.algorithmic_bytes / (mean_ms * 1e-3) / 1e9
        hbm, hbm_src = hbm_peak()
        roofline = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                    "traffic": None, "kernel": "attn_fwd_kernel (split-KV) + splitkv_combine_kernel",
                    "peak_source": hbm_src, "algorithmic_bytes": w.algorithmic_bytes,
                    "kernel_ms": {"mean": mean_ms, "min": min(durs), "max": max(durs)}}
    else:
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": measured_traffic(w.name),
                    "kernel": "attn_fwd_kernel", "peak_source": peak_src,
                    "kernel_ms": {"mean": mean_ms, "min": min(kdurs), "max": max(kdurs)}}
        if prepass is not None:
            roofline["prepass"] = prepass

    e2e = None
    if not args.no_e2e and not decode:
        e2e = (measure_e2e_block if block else measure_e2e)(args, w, x, dev, dist, world)

    clocks = sampler.summary(t_host0, t_host1)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tflops, desc, secs, steps = cpu_oracle_sample(w, x, args.cpu_seconds)
        cpu = {"value": tflops, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
               "sample": desc + f"; {secs:.1f} s of CPU work"}
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3" if fp8 else "bf16", "data": "synthetic",
            "repeats": len(totals), "repeat_ms_per_step": [t / args.steps for t in totals],
            "config": config_of(w),
            "roofline": roofline,
            "e2e": e2e, "cpu_baseline": cpu, "gpu_launches": args.steps * len(totals) * launches_per_step(w), "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def launches_per_step(w):
    """Kernels of this library launched by one step."""
    from exact_attention_72_gb300 import binding
    if w.name in DECODE_NAMES:
        return 2                                  # split-KV forward + combine
    # a non-causal forward that cuts some tiles' keys across two launches makes a second launch
    fwd = 2 if binding.attn_fwd_tail_units(w.B, w.H, w.N, w.d, w.causal, fp8=w.dtype != "bf16") else 1
    if w.dtype == "fp8_block":
        v_launches = 1 if w.N <= 128 else 3       # one block per head: maxima, codes, descales
        return 1 + 1 + v_launches + fwd           # quantise q, k, v; block-scaled forward
    return fwd


def measure_e2e_block(args, w, x, dev, dist, world):
    """Block-scaled e4m3 chain end to end: pinned bf16 q/k/v copied in, quantised and attended on
    the GPU through the public binding, o and lse copied back to pinned host memory."""
    import torch
    from exact_attention_72_gb300 import binding
    qh, kh, vh = x.q.pin_memory(), x.k.pin_memory(), x.v.pin_memory()
    oh = torch.empty((w.B, w.N, w.H, w.d), dtype=torch.bfloat16).pin_memory()
    lh = torch.empty((w.B, w.H, w.N), dtype=torch.float32).pin_memory()
    qd, kd, vd = (torch.empty(t.shape, dtype=t.dtype, device=dev) for t in (qh, kh, vh))
    signs = fp8_block_signs(w).to(dev)
    o = torch.empty(oh.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(lh.shape, dtype=torch.float32, device=dev)

    def step():
        for d_, h_ in ((qd, qh), (kd, kh), (vd, vh)):
            d_.copy_(h_, non_blocking=True)
        q8, dq = binding.quantize_e4m3(qd, 128, signs)
        k8, dk = binding.quantize_e4m3(kd, 64, signs)
        v8, dv = binding.quantize_e4m3(vd, w.N)
        binding.attn_fwd_fp8_blockscaled(q8, k8, v8, w.causal, dq, dk, dv.view(w.B, w.Hkv), scale=w.scale, out=o,
                                         lse=lse)
        oh.copy_(o, non_blocking=True)
        lh.copy_(lse, non_blocking=True)

    for _ in range(max(args.warmup, 0)):
        step()
    ms, per = timed_e2e(args, dist, torch.cuda.current_stream(), step)
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    d2h = oh.numel() * oh.element_size() + lh.numel() * lh.element_size()
    return {"value": w.flops * world / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms, "repeat_ms_per_step": per,
            "entry_point": "quantize_e4m3 + attn_fwd_fp8_blockscaled on pinned host buffers"}


def measure_e2e(args, w, x, dev, dist, world):
    """Same metric through attn_fwd_host: pinned host q/k/v in, o/lse back to pinned host memory."""
    import torch
    from exact_attention_72_gb300 import binding
    code = binding.ATTN_DTYPE_FP8_E4M3 if w.dtype == "fp8_e4m3" else binding.ATTN_DTYPE_BF16
    ws = torch.empty(binding.attn_fwd_host_workspace_bytes(w.B, w.H, w.Hkv, w.N, w.d, code), dtype=torch.uint8,
                     device=dev)
    qh, kh, vh = x.q.pin_memory(), x.k.pin_memory(), x.v.pin_memory()
    oh = torch.empty((w.B, w.N, w.H, w.d), dtype=torch.bfloat16).pin_memory()
    lh = torch.empty((w.B, w.H, w.N), dtype=torch.float32).pin_memory()

    def step():
        binding.attn_fwd_host(qh, kh, vh, oh, lh, w.causal, ws, scale=w.scale, descale_q=x.descale_q,
                              descale_k=x.descale_k, descale_v=x.descale_v)

    for _ in range(max(args.warmup, 0)):
        step()
    ms, per = timed_e2e(args, dist, torch.cuda.current_stream(), step)
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh)) + (12 if code else 0)
    d2h = oh.numel() * oh.element_size() + lh.numel() * lh.element_size()
    return {"value": w.flops * world / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms, "repeat_ms_per_step": per,
            "entry_point": "attn_fwd_host"}


# ------------------------------------------------------------------------------------ backward
BWD_FLOP_FACTOR = 2.5   # five tile GEMMs against the forward's two (the usual backward convention)


def bwd_config(w):
    c = config_of(w)
    c["pass"] = "backward (dQ, dK, dV; O and LSE from one untimed forward)"
    return c


def bwd_cpu_sample(w, x, do, seconds: float, rows=1024, max_steps=None):
    """The backward oracle on causal prefixes of `rows` rows of successive heads (a valid
    sub-problem: a prefix of a causal sequence does not see later keys)."""
    import numpy as np
    import oracle
    g = w.H // w.Hkv
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    n = min(rows, w.N)
    flops = elapsed = 0.0
    steps = 0
    while elapsed < seconds and (max_steps is None or steps < max_steps):
        b, h = heads[steps % len(heads)]
        f = lambda t, hh: t[b, :n, hh, :].float().double().numpy()
        q, k, v, dd = f(x.q, h), f(x.k, h // g), f(x.v, h // g), f(do, h)
        t0 = time.perf_counter()
        oracle.attention_backward_head(q, k, v, dd, w.scale, w.causal)
        elapsed += time.perf_counter() - t0
        flops += BWD_FLOP_FACTOR * 4.0 * w.d * n * n / (2.0 if w.causal else 1.0)
        steps += 1
    desc = (f"{steps} backward sub-problems of the first {n} rows and keys of a head (fp64, P materialised) "
            f"of the {w.name} workload; FLOPs credited by the metric's convention")
    return (flops / elapsed / 1e12 if elapsed > 0 else 0.0), desc, elapsed, steps


def run_bwd_reference(args, w, x):
    from exact_attention_72_gb300 import inputs
    rank, world, _ = rank_info()
    if rank != 0:
        return
    do = inputs.make_grad_output(w)
    if args.warmup > 0:
        bwd_cpu_sample(w, x, do, seconds=1e9, rows=512, max_steps=args.warmup)
    tflops, desc, secs, steps = bwd_cpu_sample(w, x, do, seconds=1e9, rows=512, max_steps=args.steps)
    line = {
        "impl": "reference", "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / max(1, steps) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bwd_config(w),
        "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
                         "sample": "each step: " + desc},
        "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def run_bwd_ours(args, w, x):
    import torch
    from exact_attention_72_gb300 import binding, build, inputs
    rank, world, local = rank_info()
    dist = init_dist(world)
    build.build()
    binding.lib()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    do_h = inputs.make_grad_output(w)
    q, k, v, do = x.q.to(dev), x.k.to(dev), x.v.to(dev), do_h.to(dev)
    o, lse = binding.attn_fwd(q, k, v, causal=w.causal, scale=w.scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(binding.attn_bwd_workspace_bytes(w.B, w.H, w.N), dtype=torch.uint8, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()
    flops = BWD_FLOP_FACTOR * w.flops

    def step(i=None, mid=None):
        binding.attn_bwd(q, k, v, o, lse, do, w.causal, scale=w.scale, dq=dq, dk=dk, dv=dv, workspace=ws)

    for i in range(max(args.warmup, 0)):
        flush(i)
        step()
    torch.cuda.synchronize()
    st, detail = binding.attn_get_status()
    if st != binding.ATTN_OK:
        raise RuntimeError(f"device status {st} ({detail:#x}) after warm-up")
    sampler = ClockSampler(local)
    sampler.wait_first()
    durs_all, _, totals, med, t_host0, t_host1 = timed_repeats(args, dist, stream, flush, step)
    time.sleep(0.12)
    sampler.stop()
    durs = durs_all[med]
    st, detail = binding.attn_get_status()
    if st != binding.ATTN_OK:
        raise RuntimeError(f"device status {st} ({detail:#x}) after the timed region")
    total_ms = totals[med]
    value = flops * args.steps * world / (total_ms * 1e-3) / 1e12
    mean_ms = statistics.fmean(durs)
    achieved = flops / (mean_ms * 1e-3) / 1e12
    peak, peak_src = peaks()
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": None, "peak_source": peak_src,
                "kernel": "the backward pass as one unit: preprocess + attn_bwd_dkdv_kernel + attn_bwd_dq_kernel "
                          "(algorithmic FLOPs: five tile GEMMs; the kernels execute seven)",
                "kernel_ms": {"mean": mean_ms, "min": min(durs), "max": max(durs)}}
    e2e = None
    if not args.no_e2e:
        hs = [t.pin_memory() for t in (x.q, x.k, x.v)] + [do_h.pin_memory(), o.cpu().pin_memory(),
                                                           lse.cpu().pin_memory()]
        outs_h = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (dq, dk, dv)]
        devs = (q, k, v, do, o, lse)

        def e2e_step():
            for d_, h_ in zip(devs, hs):
                d_.copy_(h_, non_blocking=True)
            step()
            for h_, d_ in zip(outs_h, (dq, dk, dv)):
                h_.copy_(d_, non_blocking=True)

        for _ in range(max(args.warmup, 0)):
            e2e_step()
        ms, per = timed_e2e(args, dist, stream, e2e_step)
        e2e = {"value": flops * world / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in hs),
               "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in outs_h),
               "ms_per_step": ms, "repeat_ms_per_step": per, "entry_point": "attn_bwd on pinned host copies"}
    clocks = sampler.summary(t_host0, t_host1)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tflops, desc, secs, _ = bwd_cpu_sample(w, x, do_h, args.cpu_seconds)
        cpu = {"value": tflops, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
               "sample": desc + f"; {secs:.1f} s of CPU work"}
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "repeats": len(totals), "repeat_ms_per_step": [t / args.steps for t in totals],
            "config": bwd_config(w), "roofline": roofline, "e2e": e2e, "cpu_baseline": cpu,
            "gpu_launches": args.steps * len(totals) * 3, "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ------------------------------------------------------------------------------------ ragged batch
def varlen_config(w):
    return {"workload": w.name, "B": w.B, "H": w.H, "Hkv": w.Hkv, "d": w.d, "causal": w.causal,
            "lengths_q": list(w.lengths_q), "lengths_k": list(w.lk), "total_q": w.total_q, "qkv_dtype": w.dtype,
            "plan": "attn_varlen_plan built once before timing and reused by every step",
            "l2": "flushed before every step (256 MiB write, then a 256 MiB read that drains its dirty lines; outside the timed events)",
            "parallelism": "replicas (one full workload per GPU)"}


def varlen_cpu_sample(w, x, seconds: float, block_rows=512, max_steps=None):
    """The oracle on row blocks of successive (sequence, head) pairs of the ragged batch."""
    import numpy as np
    import oracle
    g = w.H // w.Hkv
    pairs = [(b, h) for b in range(w.B) if w.lengths_q[b] > 0 for h in range(w.H)]
    flops = elapsed = 0.0
    steps = i = 0
    cache = {}
    while elapsed < seconds and (max_steps is None or steps < max_steps):
        b, h = pairs[i % len(pairs)]
        nq, nk = w.lengths_q[b], w.lk[b]
        nblk = max(1, -(-nq // block_rows))
        blk = (i * 7) % nblk
        i += 1
        if (b, h) not in cache:
            cache.clear()
            q0, k0 = int(w.cu_q[b]), int(w.cu_k[b])

            def up(t, r0, n, hh, sc):
                a = t[r0:r0 + n, hh, :].float().double().numpy()
                return a * np.float64(np.float32(sc)) if t.element_size() == 1 else a
            cache[(b, h)] = (up(x.q, q0, nq, h, x.descale_q), up(x.k, k0, nk, h // g, x.descale_k),
                             up(x.v, k0, nk, h // g, x.descale_v))
        q, k, v = cache[(b, h)]
        rows = np.arange(blk * block_rows, min(nq, (blk + 1) * block_rows))
        t0 = time.perf_counter()
        oracle.attention_head(q, k, v, w.scale, w.causal, rows=rows, causal_offset=nk - nq)
        elapsed += time.perf_counter() - t0
        if w.causal:   # the metric's convention: half the rectangle for a causal sequence
            flops += 4.0 * w.d * nk * len(rows) / 2.0
        else:
            flops += 4.0 * w.d * nk * len(rows)
        steps += 1
    desc = (f"{steps} blocks of up to {block_rows} query rows (full score rows, fp64) from (sequence, head) "
            f"pairs of the {w.name} ragged batch; FLOPs credited by the metric's convention")
    return (flops / elapsed / 1e12 if elapsed > 0 else 0.0), desc, elapsed, steps


def run_varlen_reference(args, w, x):
    rank, world, _ = rank_info()
    if rank != 0:
        return
    if args.warmup > 0:
        varlen_cpu_sample(w, x, seconds=1e9, block_rows=256, max_steps=args.warmup)
    tflops, desc, secs, steps = varlen_cpu_sample(w, x, seconds=1e9, block_rows=256, max_steps=args.steps)
    line = {
        "impl": "reference", "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / max(1, steps) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": varlen_config(w),
        "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
                         "sample": "each step: " + desc},
        "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def run_varlen_ours(args, w, x):
    import torch
    from exact_attention_72_gb300 import binding, build
    rank, world, local = rank_info()
    dist = init_dist(world)
    build.build()
    binding.lib()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fp8 = w.dtype == "fp8_e4m3"
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    kw = {}
    if fp8:
        kw = {n: torch.tensor([s], dtype=torch.float32, device=dev)
              for n, s in (("descale_q", x.descale_q), ("descale_k", x.descale_k), ("descale_v", x.descale_v))}
    cu_q = torch.tensor(w.cu_q, dtype=torch.int32, device=dev)
    cu_k = torch.tensor(w.cu_k, dtype=torch.int32, device=dev)
    o = torch.empty((w.total_q, w.H, w.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.H, w.total_q), dtype=torch.float32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()
    # the plan: built once, like a serving loop reusing it across layers; its build time is reported
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    plan = binding.attn_varlen_plan(cu_q, cu_k, w.H, w.total_q, w.total_k, w.d, w.causal)
    p1.record(stream)

    def step(i=None, mid=None):
        binding.attn_fwd_varlen(q, k, v, cu_q, cu_k, plan, w.causal, scale=w.scale, out=o, lse=lse, **kw)

    for i in range(max(args.warmup, 0)):
        flush(i)
        step()
    torch.cuda.synchronize()
    plan_ms = p0.elapsed_time(p1)
    st, detail = binding.attn_get_status()
    if st != binding.ATTN_OK:
        raise RuntimeError(f"device status {st} ({detail:#x}) after warm-up")
    sampler = ClockSampler(local)
    sampler.wait_first()
    durs_all, _, totals, med, t_host0, t_host1 = timed_repeats(args, dist, stream, flush, step)
    time.sleep(0.12)
    sampler.stop()
    durs = durs_all[med]
    st, detail = binding.attn_get_status()
    if st != binding.ATTN_OK:
        raise RuntimeError(f"device status {st} ({detail:#x}) after the timed region")
    total_ms = totals[med]
    value = w.flops * args.steps * world / (total_ms * 1e-3) / 1e12
    mean_ms = statistics.fmean(durs)
    achieved = w.flops / (mean_ms * 1e-3) / 1e12
    peak_bf16, peak_src = peaks()
    peak = peak_bf16 * (2.0 if fp8 else 1.0)
    if fp8:
        peak_src += " x2 (e4m3/bf16 nominal dense ratio)"
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": measured_traffic(w.name), "kernel": "attn_fwd_kernel (varlen)", "peak_source": peak_src,
                "kernel_ms": {"mean": mean_ms, "min": min(durs), "max": max(durs)}, "plan_build_ms": plan_ms}
    e2e = None
    if not args.no_e2e:
        qh, kh, vh = x.q.pin_memory(), x.k.pin_memory(), x.v.pin_memory()
        oh = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        lh = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()

        def e2e_step():
            for d_, h_ in ((q, qh), (k, kh), (v, vh)):
                d_.copy_(h_, non_blocking=True)
            step()
            oh.copy_(o, non_blocking=True)
            lh.copy_(lse, non_blocking=True)

        for _ in range(max(args.warmup, 0)):
            e2e_step()
        ms, per = timed_e2e(args, dist, stream, e2e_step)
        e2e = {"value": w.flops * world / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in (qh, kh, vh)),
               "d2h_bytes_per_step": oh.numel() * oh.element_size() + lh.numel() * lh.element_size(),
               "ms_per_step": ms, "repeat_ms_per_step": per, "entry_point": "attn_fwd_varlen on pinned host copies"}
    clocks = sampler.summary(t_host0, t_host1)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tflops, desc, secs, _ = varlen_cpu_sample(w, x, args.cpu_seconds)
        cpu = {"value": tflops, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
               "sample": desc + f"; {secs:.1f} s of CPU work"}
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3" if fp8 else "bf16", "data": "synthetic",
            "repeats": len(totals), "repeat_ms_per_step": [t / args.steps for t in totals],
            "config": varlen_config(w), "roofline": roofline, "e2e": e2e, "cpu_baseline": cpu,
            "gpu_launches": args.steps * len(totals), "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main(argv=None):
    args = parse_args(argv)
    from exact_attention_72_gb300 import inputs
    name = args.workload or inputs.HEADLINE
    if name in inputs.VARLEN_WORKLOADS:
        w = inputs.VARLEN_WORKLOADS[name]
        rank, world, _ = rank_info()
        if args.impl == "reference" and rank != 0:
            return 0
        x = inputs.make_varlen_inputs(w)
        (run_varlen_reference if args.impl == "reference" else run_varlen_ours)(args, w, x)
        return 0
    if name in inputs.BWD_WORKLOADS:
        w = inputs.BWD_WORKLOADS[name]
        if args.batch is not None:
            w = w.replace(B=args.batch, name=f"{w.name}_b{args.batch}")
        rank, world, _ = rank_info()
        if args.impl == "reference" and rank != 0:
            return 0
        x = inputs.make_inputs(w)
        (run_bwd_reference if args.impl == "reference" else run_bwd_ours)(args, w, x)
        return 0
    table = {**inputs.WORKLOADS, **inputs.DECODE_WORKLOADS, **inputs.FP8_BLOCK_WORKLOADS,
             **inputs.EXTRA_FWD_WORKLOADS}
    w = table[name]
    if args.batch is not None:
        w = w.replace(B=args.batch, name=f"{w.name}_b{args.batch}")
    rank, world, _ = rank_info()
    if args.impl == "reference" and rank != 0:
        return 0
    x = inputs.make_inputs(w)
    if args.impl == "reference":
        (run_reference_full if args.oracle_full else run_reference)(args, w, x)
    else:
        run_ours(args, w, x)
    return 0


if __name__ == "__main__":
    sys.exit(main())
