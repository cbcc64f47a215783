#!/usr/bin/env python
"""Benchmark of the fused attention forward on GB300.

One step = one attn_fwd call (tcgen05 prefill kernel) on the long-prefill
causal workload: B=2, H=32, Nq=Nk=8192, d=128, bf16, K x4 on 1% of key rows,
inputs resident in device memory (Q+K+V = 403 MB, larger than the 129 MB L2,
so no flush is needed between steps).  The line also carries the split-KV
decode workload (B=16, H=32, Nq=1, Nk=32768, d=128) in GB/s, the other
prefill workloads, an end-to-end figure through the C ABI with pinned host
buffers, the roofline of the dominant kernel, and the CPU oracle timed on the
host's cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs N independent replicas (one per GPU, launched by torchrun); the
attention path needs no exchange between GPUs.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from attention_attn_fwd_07_gb300 import inputs as W  # noqa: E402

METRIC = "attention fwd TFLOPS (prefill) / HBM GB/s (decode) at 1 GB300, % of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PROFILE_TXT = os.path.join(ROOT, "profiles", "fwd_tcgen05_long_prefill_causal.md")
# Query heads per pipelined chunk of the end-to-end call (8: measured fastest
# of 1, 2, 4, 8, 16; smaller chunks make the host's per-chunk issue cost the
# bottleneck, larger ones leave more of the last compute and download
# exposed).
E2E_CHUNK_HEADS = 8
KERNEL_SOURCES = ["fwd_tcgen05.cu", "ptx.cuh", "internal.cuh"]
DECODE_PROFILE_TXT = os.path.join(ROOT, "profiles", "splitkv_decode.md")
DECODE_SOURCES = ["splitkv.cu", "splitkv_tc.cu", "ptx.cuh", "internal.cuh"]
BWD_PROFILE_TXT = os.path.join(ROOT, "profiles", "bwd_tcgen05_long_prefill_causal.md")
BWD_SOURCES = ["bwd_tcgen05.cu", "ptx.cuh", "internal.cuh"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true", help="main workload only (profiling runs)")
    ap.add_argument("--decode-profile-batch", type=int, default=0,
                    help="run only the split-KV decode workload with this batch size "
                         "(smaller cases for ncu captures) and print its GB/s")
    ap.add_argument("--decode-profile-gqa", action="store_true",
                    help="with --decode-profile-batch: the grouped-K/V-head decode workload")
    ap.add_argument("--decode-profile-gqa8", action="store_true",
                    help="with --decode-profile-batch: the decode with eight query heads per "
                         "K/V head (tensor-core partial kernel)")
    ap.add_argument("--prefill-profile", choices=["d64", "d96", "d256"], default=None,
                    help="run only this causal prefill workload (B4 H16 N2048 d64, or the "
                         "long prefill's bytes at d96 / d256; each small enough for ncu "
                         "captures) and print its TFLOPS")
    ap.add_argument("--seqlen-sweep", action="store_true",
                    help="latency and peak device memory of the forward and the backward as "
                         "the sequence length grows (B2 H32 d128 causal, N = 1k .. 32k)")
    ap.add_argument("--bwd-profile-batch", type=int, default=0,
                    help="run only the backward of the long causal prefill with this batch "
                         "size (smaller cases for ncu captures) and print its TFLOPS")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def prefill_flops(w: W.Workload) -> float:
    f = 4.0 * w.B * w.H * w.Nq * w.Nk * w.d
    return f / 2 if w.causal else f


def decode_bytes(w: W.Workload) -> int:
    kv = 2 * w.B * w.kv_heads * w.Nk * w.d * 2
    qo = 2 * w.B * w.H * w.Nq * w.d * 2
    return kv + qo + w.B * w.H * w.Nq * 4


def kernel_source_hash(sources=KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    for f in sources:
        with open(os.path.join(ROOT, "attention_attn_fwd_07_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(path=PROFILE_TXT, sources=KERNEL_SOURCES, key="traffic_bytes_per_launch"):
    """DRAM bytes per launch (full-size workload) from a committed ncu
    summary, if it was taken on the current kernel source (else None)."""
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    src = re.search(r"^kernel_source_sha256_16:\s*([0-9a-f]+)", txt, re.M)
    tb = re.search(r"^" + re.escape(key) + r":\s*([0-9]+)", txt, re.M)
    if not src or not tb or src.group(1) != kernel_source_hash(sources):
        return None
    return int(tb.group(1))


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while it runs."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self, t0: float, t1: float) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts + frac, float(parts[2]), float(parts[3]), parts[6:10]))
            except (ValueError, IndexError):
                continue
        os.unlink(self.path)
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        used = inside if len(inside) >= 3 else rows
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in used for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": float(np.median([r[1] for r in used])),
                "sm_max_mhz": float(max(r[2] for r in used)),
                "reasons": reasons, "samples": len(used),
                "window": "timed region" if used is inside else "whole run (timed region too short)"}


def event_time(fn, steps: int, stream) -> float:
    """Average ms per call of fn over `steps` calls, CUDA events on `stream`."""
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


def copy_only_step(stream, uploads, downloads, h2d: int, d2h: int, reps: int = 5) -> dict:
    """The end-to-end step's host<->device copies with no compute: uploads
    (device <- pinned host) alone, downloads (pinned host <- device) alone, and
    both at once on two streams.  `both_ms` is a floor for the end-to-end step
    (the copies have to happen; the forward can at best hide under them)."""
    side = torch.cuda.Stream()

    def up():
        for dst, src in uploads:
            dst.copy_(src, non_blocking=True)

    def down():
        for dst, src in downloads:
            dst.copy_(src, non_blocking=True)

    def both():
        side.wait_stream(torch.cuda.current_stream())
        up()
        with torch.cuda.stream(side):
            down()
        torch.cuda.current_stream().wait_stream(side)

    out = {}
    with torch.cuda.stream(stream):
        for name, fn in (("h2d", up), ("d2h", down), ("both", both)):
            fn()
            out[name + "_ms"] = event_time(fn, reps, stream)
    out["h2d_gbs"] = h2d / out["h2d_ms"] / 1e6
    out["d2h_gbs"] = d2h / out["d2h_ms"] / 1e6
    return out


def event_time_each(fn, steps: int, stream, scratch: torch.Tensor | None = None) -> list:
    """ms of each of `steps` calls, every call between its own CUDA events on
    `stream`; with `scratch` (a buffer larger than L2), L2 is flushed by
    rewriting it before each call, outside the events."""
    out = []
    for _ in range(steps):
        if scratch is not None:
            scratch.add_(1)
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        fn()
        end.record(stream)
        end.synchronize()
        out.append(start.elapsed_time(end))
    return out


def launch_stats(times_ms: list) -> dict:
    """Median, 10th and 90th percentile of per-call times (ms)."""
    a = np.asarray(times_ms, dtype=np.float64)
    return {"median": float(np.median(a)), "p10": float(np.percentile(a, 10)),
            "p90": float(np.percentile(a, 90)), "n": int(a.size)}


def graph_time(launch_on, calls: int, reps: int = 5) -> float | None:
    """ms per call of `calls` back-to-back calls captured in one CUDA graph
    and replayed `reps` times (launch overhead out of the picture);
    launch_on(stream) issues one call on that stream.  Capture and replay
    run on a stream of their own (the legacy default stream cannot be
    captured); None if the capture fails."""
    side = torch.cuda.Stream()
    fn = lambda: launch_on(side)  # noqa: E731
    try:
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            fn()  # warm: any one-time host work happens outside the capture
            torch.cuda.synchronize()
            with torch.cuda.graph(graph, stream=side):
                for _ in range(calls):
                    fn()
        with torch.cuda.stream(side):  # replay on the stream the events are on
            graph.replay()
            torch.cuda.synchronize()
            ms = event_time(graph.replay, reps, side) / calls
        del graph
        return ms
    except Exception:  # capture refused (a call not capturable here): no figure
        torch.cuda.synchronize()
        return None


def event_time_flushed(fn, steps: int, stream, scratch: torch.Tensor) -> tuple:
    """Average ms per call with L2 flushed before each call, and the per-call
    distribution."""
    t = event_time_each(fn, steps, stream, scratch)
    return sum(t) / len(t), launch_stats(t)


# ------------------------------------------------------------------ CPU oracle legs
def oracle_sample(w: W.Workload, q, k, v, target_s: float):
    """Time the oracle on a bounded sample of the workload's query rows.

    The sample is every query row of the first few (b, h) heads, as many
    heads as take about ``target_s`` seconds on all host threads (calibrated
    on a small sample first); FLOPs are counted per row (4*d*visible keys).
    """
    import oracle
    lib = oracle.load()
    threads = oracle.default_threads()
    BH = w.B * w.H

    def rows_flops(n_rows):
        flat = np.arange(n_rows, dtype=np.int64)
        i = flat % w.Nq
        keys = np.minimum(w.Nk, i + 1) if w.causal else np.full_like(i, w.Nk)
        return flat, float(4.0 * w.d * keys.sum())

    heads = 1
    while True:
        rows, fl = rows_flops(heads * w.Nq)
        t = time.perf_counter()
        oracle.attention(q, k, v, causal=w.causal, scale=w.scale, rows=rows, threads=threads,
                         lib=lib)
        dt = time.perf_counter() - t
        if dt >= 0.5 * target_s or heads == BH:
            break
        heads = int(min(BH, max(heads + 1, round(heads * target_s / max(dt, 1e-3)))))
    return {"value": fl / dt / 1e12, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
            "sample": f"all {w.Nq} query rows of the first {heads} of {BH} (b,h) heads of "
                      f"{w.name}; {fl / 1e9:.1f} GFLOP in {dt:.1f} s (fp64, all host threads)"}


def run_reference(args):
    """The oracle as the reference arm, on bounded samples of the same workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = W.LONG_PREFILL_CAUSAL
    q, k, v = W.make_qkv(w)
    import oracle
    threads = oracle.default_threads()

    def pick(n):
        r = np.linspace(0, w.Nq - 1, n).round().astype(np.int64)
        return r, sum(4.0 * w.d * (int(i) + 1) for i in r)

    # Size one step to about one second of host work (calibrated once).
    rows, fl = pick(4 * threads)
    t = time.perf_counter()
    oracle.attention(q, k, v, causal=True, scale=w.scale, rows=rows, threads=threads)
    dt = max(time.perf_counter() - t, 1e-3)
    rows, fl = pick(int(min(w.Nq, max(4 * threads, 4 * threads * 1.0 / dt))))
    times = []
    for step in range(args.warmup + args.steps):
        t = time.perf_counter()
        oracle.attention(q, k, v, causal=True, scale=w.scale, rows=rows, threads=threads)
        if step >= args.warmup:
            times.append(time.perf_counter() - t)
    ms = 1e3 * float(np.mean(times))
    value = fl / (ms / 1e3) / 1e12
    sample = (f"{len(rows)} evenly spaced query rows of head (0,0) per step "
              f"({fl / 1e9:.3f} GFLOP, fp64)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
                       "causal": True, "sample": sample},
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU leg
def init_ranks():
    """(world, rank, local_rank, dist) from the torchrun environment.  With
    more than one rank, gloo carries only the barrier around the timed region
    and the max over ranks of the timing: the ranks are independent replicas
    (no data-path collective)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group("gloo")
    return world, rank, local, dist


def barrier(dist) -> None:
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float) -> float:
    """The slowest rank's time: the job is done when every replica is."""
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def summary_of(line: dict) -> list:
    """[[workload, value, unit, roofline frac, ms], ...] for every line."""
    def one(name, r):
        if r is None:
            return None
        roof = r.get("roofline") or {}
        frac = roof.get("frac", r.get("frac_of_peak"))
        return [name, round(float(r["value"]), 1), r.get("unit") or r.get("metric"),
                None if frac is None else round(float(frac), 3),
                round(float(r["ms_per_step"]), 4)]

    out = [one(line["config"]["workload"], line)]
    out += [one(o["workload"], o) for o in line.get("other_workloads") or []]
    if line.get("decode_gqa"):
        out.append(one(line["decode_gqa"]["workload"], line["decode_gqa"]))
    if line.get("decode"):
        d = line["decode"]
        out.append(one(d["workload"] + f", S={d['splits']}", d))
    return [o for o in out if o is not None]


def run_seqlen_sweep(args, dev, stream, pk) -> list:
    """Forward and backward latency and peak device memory as N grows, at
    the long prefill's head shape (B2 H32 d128, causal).  Peak memory is
    torch's allocator high-water mark over the call (inputs, outputs and the
    backward's workspace: the library allocates nothing); the unfused score
    matrix a non-fused forward would hold (fp32 [B, H, N, N]) is listed
    beside it."""
    from attention_attn_fwd_07_gb300 import binding
    rows = []
    for N in (1024, 2048, 4096, 8192, 16384, 32768):
        w = W.Workload(f"B2 H32 N{N} d128 causal", 2, 32, N, N, 128, True, 1011)
        torch.cuda.empty_cache()
        torch.cuda.reset_peak_memory_stats(dev)
        base = torch.cuda.memory_allocated(dev)
        q, k, v = W.make_qkv(w, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, N), dtype=torch.float32, device=dev)

        def f():
            binding.attn_fwd(q, k, v, True, w.scale, o=o, lse=lse, stream=stream)

        for _ in range(args.warmup):
            f()
        fwd_ms = launch_stats(event_time_each(f, 10, stream))["median"]
        fwd_peak = torch.cuda.max_memory_allocated(dev) - base
        dout = W.make_dout(w, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty((binding.attn_bwd_workspace_bytes(w.B, w.H, N),), dtype=torch.uint8,
                         device=dev)

        def b():
            binding.attn_bwd(q, k, v, o, lse, dout, True, w.scale, workspace=ws, dq=dq, dk=dk,
                             dv=dv, stream=stream)

        for _ in range(args.warmup):
            b()
        bwd_ms = launch_stats(event_time_each(b, 10, stream))["median"]
        bwd_peak = torch.cuda.max_memory_allocated(dev) - base
        fl = prefill_flops(w)
        rows.append({"N": N, "fwd_ms": fwd_ms, "fwd_tflops": fl / (fwd_ms / 1e3) / 1e12,
                     "fwd_peak_bytes": int(fwd_peak), "bwd_ms": bwd_ms,
                     "bwd_tflops": 2.5 * fl / (bwd_ms / 1e3) / 1e12,
                     "bwd_peak_bytes": int(bwd_peak),
                     "unfused_scores_bytes": int(w.B * w.H * N * N * 4),
                     "fwd_frac": fl / (fwd_ms / 1e3) / 1e12 / pk["bf16_tflops"]})
        print(json.dumps(rows[-1]), flush=True)
        del q, k, v, o, lse, dout, dq, dk, dv, ws
    return rows


def run_backward(w, q, k, v, o, lse, dev, stream, args, pk, pk_src, world, max_over_ranks):
    """Time attn_bwd (three launches) on the workload's forward outputs."""
    from attention_attn_fwd_07_gb300 import binding
    dout = W.make_dout(w, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty((binding.attn_bwd_workspace_bytes(w.B, w.H, w.Nq),), dtype=torch.uint8,
                     device=dev)
    binding.attn_fwd(q, k, v, w.causal, w.scale, o=o, lse=lse, stream=stream)

    def sb():
        binding.attn_bwd(q, k, v, o, lse, dout, w.causal, w.scale, workspace=ws, dq=dq, dk=dk,
                         dv=dv, stream=stream)

    for _ in range(args.warmup):
        sb()
    m = max_over_ranks(event_time(sb, args.steps, stream))
    flops = 2.5 * prefill_flops(w)
    tf = flops / (m / 1e3) / 1e12
    del dout, dq, dk, dv, ws
    return {"workload": w.name + ", backward (dQ, dK, dV)", "metric": "TFLOPS",
            "value": world * tf, "ms_per_step": m, "launches_per_step": 3,
            "flops_convention": "2.5 x the forward's (five matmuls: S, dP, dV, dK, dQ); the "
                                "kernels execute seven (S and dP again in the dQ kernel)",
            "roofline": {"bound": "tensor", "achieved": tf, "peak": pk["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": tf / pk["bf16_tflops"],
                         "peak_source": f"{pk_src} bf16 dense (burst)",
                         "traffic": recorded_traffic(BWD_PROFILE_TXT, BWD_SOURCES)
                         if w is W.LONG_PREFILL_CAUSAL else None,
                         "traffic_kernel": "bwd_dkdv_kernel (dominant launch of the three)"},
            "l2": "inputs larger than L2; no flush"}


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    world, rank, local, dist = init_ranks()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from attention_attn_fwd_07_gb300 import binding, build
    build.build()
    binding.load_library()
    stream = torch.cuda.current_stream()
    pk, pk_src = peaks()

    def barrier_():
        barrier(dist)

    def max_over_ranks_(x: float) -> float:
        return max_over_ranks(dist, x)

    launches = 0

    if args.prefill_profile:
        # One prefill workload alone, L2 flushed before each timed launch as
        # in the full run.
        wp = {"d64": W.PREFILL, "d96": W.LONG_PREFILL_D96,
              "d256": W.LONG_PREFILL_D256}[args.prefill_profile]
        qp, kp, vp = W.make_qkv(wp, device=dev)
        op = torch.empty_like(qp)
        lp = torch.empty((wp.B, wp.H, wp.Nq), dtype=torch.float32, device=dev)

        def sp():
            binding.attn_fwd(qp, kp, vp, wp.causal, wp.scale, o=op, lse=lp, stream=stream)

        for _ in range(args.warmup):
            sp()
        scratch = torch.empty((256 << 20) // 4, dtype=torch.float32, device=dev)
        m, st = event_time_flushed(sp, args.steps, stream, scratch)
        print(json.dumps({"workload": wp.name, "ms_per_step": m, "launch_ms": st,
                          "TFLOPS": prefill_flops(wp) / (m / 1e3) / 1e12}), flush=True)
        return 0

    if args.seqlen_sweep:
        run_seqlen_sweep(args, dev, stream, pk)
        return 0

    if args.bwd_profile_batch > 0:
        # Backward only, smaller batch: the case the ncu captures run on.
        base = W.LONG_PREFILL_CAUSAL
        wb = W.Workload(base.name.replace("B2", f"B{args.bwd_profile_batch}"),
                        args.bwd_profile_batch, base.H, base.Nq, base.Nk, base.d, True,
                        base.seed)
        qb, kb, vb = W.make_qkv(wb, device=dev)
        ob = torch.empty_like(qb)
        lb = torch.empty((wb.B, wb.H, wb.Nq), dtype=torch.float32, device=dev)
        r = run_backward(wb, qb, kb, vb, ob, lb, dev, stream, args, pk, pk_src, 1,
                         lambda x: x)
        print(json.dumps(r), flush=True)
        return 0

    if args.decode_profile_batch > 0:
        # Decode only, smaller batch: the case the ncu captures run on.
        base = (W.DECODE_GQA8 if args.decode_profile_gqa8 else
                W.DECODE_GQA if args.decode_profile_gqa else W.DECODE)
        wd = W.Workload(base.name.replace("B16", f"B{args.decode_profile_batch}"),
                        args.decode_profile_batch, base.H, 1, base.Nk, base.d,
                        False, base.seed, Hkv=base.Hkv)
        qd, kd, vd = W.make_qkv(wd, device=dev)
        od = torch.empty_like(qd)
        ld = torch.empty((wd.B, wd.H, 1), dtype=torch.float32, device=dev)
        S = 16
        ws = torch.empty((binding.attn_splitkv_workspace_bytes(wd.B, wd.H, 1, wd.d, S),),
                         dtype=torch.uint8, device=dev)

        def sd():
            binding.attn_fwd_splitkv(qd, kd, vd, False, wd.scale, S, workspace=ws, o=od, lse=ld,
                                     stream=stream)

        for _ in range(args.warmup):
            sd()
        m = event_time(sd, args.steps, stream)
        print(json.dumps({"workload": wd.name, "splits": S, "ms_per_step": m,
                          "GB/s": decode_bytes(wd) / (m / 1e3) / 1e9}), flush=True)
        return 0

    # ---- main workload: long prefill, causal
    w = W.LONG_PREFILL_CAUSAL
    q_h, k_h, v_h = W.make_qkv(w)
    q, k, v = (t.to(dev) for t in (q_h, k_h, v_h))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)

    def step():
        binding.attn_fwd(q, k, v, True, w.scale, o=o, lse=lse, stream=stream)

    for _ in range(args.warmup):
        step()
    sampler = ClockSampler(local)
    sampler.start()
    barrier_()
    t0 = time.time()
    ms = event_time(step, args.steps, stream)
    t1 = time.time()
    barrier_()
    clocks = sampler.stop(t0, t1)
    launches += args.steps
    ms = max_over_ranks_(ms)
    # Per-launch distribution (this rank), taken after the timed region.
    main_dist = launch_stats(event_time_each(step, 50, stream))
    launches += 50
    flops = prefill_flops(w)
    value = world * flops / (ms / 1e3) / 1e12
    per_gpu = flops / (ms / 1e3) / 1e12
    roof = {"bound": "tensor", "achieved": per_gpu, "peak": pk["bf16_tflops"],
            "unit": "TFLOP/s", "frac": per_gpu / pk["bf16_tflops"],
            "peak_source": f"{pk_src} bf16 dense (burst: kernel timed back to back)",
            "traffic": recorded_traffic(),
            "algorithmic_flops_per_launch": flops}

    # ---- end to end through the C ABI with pinned host buffers
    q_p, k_p, v_p = (t.pin_memory() for t in (q_h, k_h, v_h))
    o_p = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    lse_p = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()

    def e2e_step():
        binding.fwd_from_host(q_p, k_p, v_p, True, w.scale, q, k, v, o, lse, o_p, lse_p,
                              stream=stream, chunk_heads=E2E_CHUNK_HEADS)

    e2e_steps = max(3, min(args.steps, 20))
    for _ in range(3):
        e2e_step()
    barrier_()
    e2e_ms = max_over_ranks_(event_time(e2e_step, e2e_steps, stream))
    launches += e2e_steps * w.B * -(-w.H // E2E_CHUNK_HEADS)  # one attn_fwd per chunk
    h2d = sum(t.numel() * t.element_size() for t in (q_p, k_p, v_p))
    d2h = o_p.numel() * o_p.element_size() + lse_p.numel() * lse_p.element_size()
    link = copy_only_step(stream, [(q, q_p), (k, k_p), (v, v_p)], [(o_p, o), (lse_p, lse)],
                          h2d, d2h)
    link["frac"] = link["both_ms"] / e2e_ms
    e2e = {"value": world * flops / (e2e_ms / 1e3) / 1e12, "unit": "TFLOPS",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
           "copy_only": link,
           "path": "attn_fwd_from_host (one C-ABI call per step, through binding.fwd_from_host): "
                   "pinned host -> device copies of Q, K, V, the forward, device -> pinned host "
                   "copies of O and LSE, pipelined in chunks of 8 heads over an upload stream, "
                   "the compute stream and a download stream; the host link (~210 GB/s each way "
                   "on this box) bounds it"}
    del q_p, k_p, v_p, o_p, lse_p

    others = []
    decode = None
    decode_gqa = None
    if not args.quick:
        # ---- the other prefill workloads
        for wo in (W.LONG_PREFILL_NONCAUSAL, W.PREFILL, W.LONG_PREFILL_D96,
                   W.LONG_PREFILL_D256):
            if wo.Nq == w.Nq and wo.d == w.d and wo.H == w.H:
                qq, kk, vv, oo, ll = q, k, v, o, lse
            else:
                qq, kk, vv = (t.to(dev) for t in W.make_qkv(wo))
                oo = torch.empty_like(qq)
                ll = torch.empty((wo.B, wo.H, wo.Nq), dtype=torch.float32, device=dev)

            def st(qq=qq, kk=kk, vv=vv, oo=oo, ll=ll, wo=wo):
                binding.attn_fwd(qq, kk, vv, wo.causal, wo.scale, o=oo, lse=ll, stream=stream)

            for _ in range(args.warmup):
                st()
            if wo.Nq >= 8192:
                n = args.steps
                m = max_over_ranks_(event_time(st, n, stream))
            else:
                # Short launches are timed one by one, L2 flushed before each;
                # the value is the per-call median, which one slow call (the
                # first after the flush buffer is allocated, ~4x the rest)
                # does not move.  The mean is reported beside it.
                n = args.steps
                scratch = torch.empty((256 << 20) // 4, dtype=torch.float32, device=dev)
                mean_ms, flushed_dist = event_time_flushed(st, n, stream, scratch)
                m = max_over_ranks_(flushed_dist["median"])
                del scratch
            launches += n
            tf = prefill_flops(wo) / (m / 1e3) / 1e12
            others.append({"workload": wo.name, "metric": "TFLOPS", "value": world * tf,
                           "ms_per_step": m,
                           "roofline": {"bound": "tensor", "achieved": tf,
                                        "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                                        "frac": tf / pk["bf16_tflops"],
                                        "peak_source": f"{pk_src} bf16 dense (burst)"},
                           "l2": "inputs > L2" if wo.Nq >= 8192 else
                                 "L2 flushed (256 MB rewrite) before each timed launch"})
            if wo.Nq < 8192:
                others[-1]["launch_ms"] = flushed_dist
                others[-1]["value_from"] = ("median of per-call times (mean "
                                            f"{mean_ms:.4f} ms over the same calls)")
                gms = graph_time(
                    lambda s, qq=qq, kk=kk, vv=vv, oo=oo, ll=ll, wo=wo: binding.attn_fwd(
                        qq, kk, vv, wo.causal, wo.scale, o=oo, lse=ll, stream=s), 100)
                if gms is not None:
                    launches += 601  # a warm-up call, one check replay, five timed replays of 100
                    others[-1]["graph_100_calls"] = {
                        "value": world * prefill_flops(wo) / (gms / 1e3) / 1e12,
                        "ms_per_call": gms,
                        "note": "100 calls captured in one CUDA graph, replayed back to back; "
                                "inputs stay L2-resident between calls (no flush), so this "
                                "is the launch-overhead-free rate, not the line's value"}
            if wo.d in (64, 96):  # the d = 64 and d = 96 backwards on the same inputs
                rb = run_backward(wo, qq, kk, vv, oo, ll, dev, stream, args, pk, pk_src, world,
                                  max_over_ranks_)
                if wo.d == 64:
                    rb["l2"] = "inputs (84 MB) fit in L2; not flushed"
                others.append(rb)
                launches += 3 * args.steps

        # ---- long prefill causal with FP8 (e4m3) Q K^T, P V in bf16
        wf = W.LONG_PREFILL_CAUSAL
        q8, k8, v8, qdesc, kdesc = W.make_qkv_fp8(wf)
        q8, k8, v8 = q8.to(dev), k8.to(dev), v8.to(dev)
        of = torch.empty((wf.B, wf.H, wf.Nq, wf.d), dtype=torch.bfloat16, device=dev)
        lf = torch.empty((wf.B, wf.H, wf.Nq), dtype=torch.float32, device=dev)

        def sf():
            binding.attn_fwd_fp8(q8, k8, v8, True, wf.scale, qdesc, kdesc, o=of, lse=lf,
                                 stream=stream)

        for _ in range(args.warmup):
            sf()
        mf = max_over_ranks_(event_time(sf, args.steps, stream))
        launches += args.steps
        tff = prefill_flops(wf) / (mf / 1e3) / 1e12
        # Half of the counted flops (Q K^T) run at the FP8 rate, half (P V)
        # at the bf16 rate.  FP8 peak = 2 x the measured bf16 peak (the
        # nominal dense ratio, 4.5 / 2.25 PFLOP/s); the mixed ceiling is the
        # rate at which both halves finish together: 1 / (0.5/(2P) + 0.5/P)
        # = 4P/3.
        mixed_peak = 4.0 * pk["bf16_tflops"] / 3.0
        others.append({"workload": wf.name + ", FP8 e4m3 Q K^T (P V bf16)", "metric": "TFLOPS",
                       "value": world * tff, "ms_per_step": mf,
                       "roofline": {"bound": "tensor", "achieved": tff, "peak": mixed_peak,
                                    "unit": "TFLOP/s", "frac": tff / mixed_peak,
                                    "peak_source": f"derived: half the flops at the FP8 rate "
                                                   f"(2 x {pk_src} bf16, the nominal ratio), "
                                                   f"half at the {pk_src} bf16 rate = 4/3 x "
                                                   f"{pk['bf16_tflops']:.1f}"},
                       "frac_of_bf16_peak": tff / pk["bf16_tflops"],
                       "l2": "inputs (269 MB) larger than L2"})
        del q8, k8, v8, of, lf

        # ---- backward of the long causal prefill (dQ, dK, dV from O, LSE, dO)
        others.append(run_backward(w, q, k, v, o, lse, dev, stream, args, pk, pk_src, world,
                                   max_over_ranks_))
        launches += 3 * args.steps

        # ---- decode (split-KV + combine), memory bound; MHA and grouped K/V heads
        def run_decode(wd):
            nonlocal launches
            qd, kd, vd = W.make_qkv(wd, device=dev)
            od = torch.empty_like(qd)
            ld = torch.empty((wd.B, wd.H, 1), dtype=torch.float32, device=dev)
            results = []
            calls = {}
            for S in wd.splits:
                need = binding.attn_splitkv_workspace_bytes(wd.B, wd.H, 1, wd.d, S)
                ws = torch.empty((need,), dtype=torch.uint8, device=dev)

                def sd(S=S, ws=ws):
                    binding.attn_fwd_splitkv(qd, kd, vd, False, wd.scale, S, workspace=ws, o=od,
                                             lse=ld, stream=stream)

                calls[S] = sd
                for _ in range(args.warmup):
                    sd()
                n = max(10, args.steps // 4)
                m = max_over_ranks_(event_time(sd, n, stream))
                launches += 2 * n
                gbs = decode_bytes(wd) / (m / 1e3) / 1e9
                results.append({"splits": S, "ms_per_step": m, "GB/s": gbs,
                                "workspace_bytes": need})
            best = max(results, key=lambda r: r["GB/s"])
            # Per-call distribution (partial + combine) at the best split count.
            best_dist = launch_stats(event_time_each(calls[best["splits"]], 30, stream))
            launches += 2 * 30
            del calls, qd, kd, vd
            return {"workload": wd.name, "metric": "HBM GB/s", "unit": "GB/s",
                    "value": world * best["GB/s"], "ms_per_step": best["ms_per_step"],
                    "splits": best["splits"], "per_split_count": results, "launch_ms": best_dist,
                    "algorithmic_bytes_per_step": decode_bytes(wd),
                    "roofline": {"bound": "hbm", "achieved": best["GB/s"],
                                 "peak": pk["hbm_gbs"], "unit": "GB/s",
                                 "frac": best["GB/s"] / pk["hbm_gbs"],
                                 "peak_source": f"{pk_src} copy bandwidth",
                                 "traffic": (recorded_traffic(
                                     DECODE_PROFILE_TXT, DECODE_SOURCES,
                                     "traffic_bytes_per_launch" if wd is W.DECODE
                                     else "gqa_traffic_bytes_per_launch")
                                     if wd in (W.DECODE, W.DECODE_GQA) else None)},
                    "l2": f"inputs {decode_bytes(wd) / 1e9:.1f} GB > L2"}

        decode = run_decode(W.DECODE)
        decode_gqa = run_decode(W.DECODE_GQA)
        others.append(run_decode(W.DECODE_GQA8))
        others.append(run_decode(W.DECODE_D256))

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_sample(w, q_h, k_h, v_h, target_s=10.0)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "launch_ms": main_dist,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
                   "causal": True, "flops_convention": "4*B*H*Nq*Nk*d, halved for causal",
                   "l2": "inputs (403 MB) larger than L2; no flush",
                   "parallelism": f"replicas x{world}"},
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
        "clocks": clocks, "decode_gqa": decode_gqa, "other_workloads": others,
        "kernel_source_sha256_16": kernel_source_hash(),
        "decode": decode,
    }
    # Last key: one short entry per measured line (value, unit, roofline
    # fraction, ms), so that the end of the line -- all a log tail keeps of
    # it -- still shows every workload.
    line["summary"] = summary_of(line)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
