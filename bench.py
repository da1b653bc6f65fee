#!/usr/bin/env python3
"""Throughput of the fused linear cross-entropy path (loss + dX + dW) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...     # the CPU oracle on a bounded sample

One step = one full call of the path (both logit passes, the row combine, the
dX and dW GEMMs over every vocabulary chunk) on one batch of synthetic input
already resident in HBM.  Steps run back to back on one stream; the timed
region is bracketed by a barrier and a device synchronise on both sides and
timed with CUDA events on that stream.  W (1.05 GB at the default workload)
is larger than L2, so consecutive steps cannot be served from L2.  A second
timed region of the same steps records the library's per-launch events
(per-kernel times, shares and the roofline); its total is reported as
ms_per_step_traced, the headline comes from the untraced region.

Prints one JSON line (rank 0).  With --gpus N > 1 each rank runs its own
replica on its own GPU (data-parallel shards, no collective on the data
path): value = all ranks' tokens / the slowest rank's time.  Started without
a launcher, --gpus N > 1 starts its N ranks itself through
torch.distributed.run (one process per GPU, rendezvous on 127.0.0.1).

The roofline's fraction is taken against the measured burst bf16 peak (the
timed region is well under a second of back-to-back steps); the fraction of
the sustained (seconds-long, power-capped) peak is given beside it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("tokens/s and % of bf16 dense peak (6·N·H·V FLOPs), "
          "fused linear CE fwd+bwd, 1 GB300")
DEFAULT_WORKLOAD = "llama3_8b_head_8192x4096x128256"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
GEMM_KINDS = ("logits_lse", "logits_grad", "dw", "dx")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _free_port() -> int:
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def launch_ranks(n: int, argv) -> int:
    """Run this script as n ranks on one node (one process per GPU) and
    return the launcher's exit code; rank 0 prints the JSON line."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr", "127.0.0.1",
           "--master-port", str(_free_port()), os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


class ClockSampler:
    """nvidia-smi samples of one GPU during the timed region."""
    Q = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, mx, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            if self.uuid and parts[0] != self.uuid:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "power_w_max": max(power), "samples": len(sm), "reasons": sorted(reasons)}


# The source files that make each kind of launch (its kernel code and the host
# code that picks its tile order and launch shape).
_GEMM_SOURCES = ["gemm.cuh", "epilogues.cuh", "sm103.cuh", "flce_internal.h",
                 "gemm_instances.cuh", "gemm_bf16.cu", "launch.h", "flce_api.cu"]
_SMALL_SOURCES = ["small_kernels.cu", "sm103.cuh", "flce_internal.h", "launch.h",
                  "flce_api.cu"]
KERNEL_SOURCES = {"logits_lse": _GEMM_SOURCES, "logits_grad": _GEMM_SOURCES,
                  "dw": _GEMM_SOURCES, "dx": _GEMM_SOURCES, "combine": _SMALL_SOURCES,
                  "convert": _SMALL_SOURCES, "ce_rows_bf16": _SMALL_SOURCES,
                  "ce_rows_fp32": _SMALL_SOURCES}


def code_only(src: str) -> str:
    """A C/C++/CUDA source without its comments and with its blank space
    collapsed: the part that decides what the compiler builds.  (The sources
    hashed here hold no comment markers inside string literals.)"""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def kernel_source_hash(kind: str, read=None) -> str:
    """Hash of the code (comments aside) of the sources a kind of launch is
    built from.  `read(name)` returns a source's text (default: the file in
    the package's csrc)."""
    d = os.path.join(ROOT, "linear_cross_entropy_fwd_gb300", "csrc")
    if read is None:
        def read(name):
            with open(os.path.join(d, name)) as fh:
                return fh.read()
    h = hashlib.sha256()
    for f in sorted(KERNEL_SOURCES[kind]):
        h.update(f.encode() + code_only(read(f)).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kind: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current sources of that kind of launch (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p) or kind not in KERNEL_SOURCES:
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kind, {})
    if e.get("source_hash") != kernel_source_hash(kind) or e.get("workload") != workload:
        return None
    return e.get("dram_bytes_per_launch")


def cpu_baseline(workload, X, W, t, budget_s: float = 15.0):
    """The oracle on the first few tokens of the workload (a prefix problem
    with the same H and V: loss, dX and dW in full), on this host's cores."""
    import oracle
    n0 = 2
    oracle.build()

    def run(n):
        t0 = time.perf_counter()
        oracle.flce(X[:n].contiguous(), W, t[:n].contiguous(), workload.ignore_index)
        return time.perf_counter() - t0

    dt0 = run(n0)
    n = int(max(n0, min(64, n0 * budget_s / max(dt0, 1e-3))))
    dt = run(n)
    return {"value": n / dt, "unit": "tokens/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": (f"first {n} tokens of {workload.name} as a problem of their own "
                       f"(loss, dX and dW in full, H={workload.H}, V={workload.V}), "
                       f"{dt:.1f} s of fp64 CPU work")}


def run_reference(args, workload):
    """--impl reference: the oracle, as it stands, on host cores; each step a
    bounded sample (the first --ref-tokens tokens of the workload)."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from flce_synth import make_inputs
    n = args.ref_tokens
    X, W, t = make_inputs(workload, rows=n)
    oracle.build()
    for _ in range(args.warmup):
        oracle.flce(X, W, t, workload.ignore_index)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.flce(X, W, t, workload.ignore_index)
        times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = n * args.steps / tot
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(workload, args.gpus),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"first {n} tokens of {workload.name} per step "
                                   f"(loss, dX and dW in full, fp64)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ce_logits(args, w):
    """Cross-entropy on materialised logits [N, V], bf16 or fp32 (loss + gradient into
    a separate buffer).  HBM-bound: the roofline is bytes moved per launch of
    the row kernel (one read and one write of the logits) over its time."""
    import torch

    import linear_cross_entropy_fwd_gb300 as flce
    from flce_synth import make_inputs
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    flce.load_library()
    peaks, peak_src = load_peaks()
    X, W, t = make_inputs(w)
    S = (X.to(dev) @ W.to(dev).t()).contiguous()  # input staging (cuBLAS), not timed
    if args.ce_dtype == "fp32":
        S = S.float()
    td = t.to(dev)
    dS = torch.empty_like(S)
    del X, W
    for _ in range(max(args.warmup, 1)):
        flce.flce_ce_fwd_bwd(S, td, w.ignore_index, dlogits=dS)
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(None)
    sampler.start()
    time.sleep(0.3)
    e0.record(stream)
    for _ in range(args.steps):
        flce.flce_ce_fwd_bwd(S, td, w.ignore_index, dlogits=dS)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1) / args.steps
    traces = [flce.Trace(capacity=8) for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    for k in range(args.steps):
        flce.flce_ce_fwd_bwd(S, td, w.ignore_index, dlogits=dS, trace=traces[k])
    torch.cuda.synchronize(dev)
    rows_ms = [t_ms for tr in traces for kind, t_ms in tr.launches() if kind == "ce_rows"]
    rows_avg = sum(rows_ms) / len(rows_ms)
    elt = S.element_size()
    algo_bytes = 2.0 * w.N * w.V * elt + w.N * (8 + 8)  # logits in, gradient out, target, stats
    achieved = algo_bytes / (rows_avg * 1e-3) / 1e9
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    line = {
        "metric": "tokens/s, cross-entropy on materialised logits (loss + gradient), 1 GB300",
        "value": w.N / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": args.ce_dtype,
        "data": "synthetic (logits = X W^T of the workload)",
        "config": workload_config(w, 1),
        "roofline": {"bound": "hbm", "kernel": "ce_rows", "achieved": achieved, "peak": hbm,
                     "unit": "GB/s", "frac": achieved / hbm,
                     "peak_kind": f"HBM copy ({peak_src})", "bytes_per_launch": algo_bytes,
                     "traffic": recorded_traffic(f"ce_rows_{args.ce_dtype}", w.name)},
        "gpu_launches": 4 * args.steps, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_fwd(args, w):
    """The loss-only evaluation path (flce_fwd): pass 1 and the combine, on
    inputs resident in HBM.  Useful work 2*N*H*V FLOP per call; the roofline
    is pass 1's executed FLOPs per launch over its mean event time."""
    import torch

    import linear_cross_entropy_fwd_gb300 as flce
    from flce_synth import make_inputs
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    flce.load_library()
    peaks, peak_src = load_peaks()
    X, W, t = make_inputs(w)
    Xd, Wd, td = X.to(dev), W.to(dev), t.to(dev)
    N, H, V = w.N, w.H, w.V
    for _ in range(max(args.warmup, 1)):
        flce.flce_fwd(Xd, Wd, td, w.ignore_index)
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(None)
    sampler.start()
    time.sleep(0.3)
    e0.record(stream)
    for _ in range(args.steps):
        flce.flce_fwd(Xd, Wd, td, w.ignore_index)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1) / args.steps
    traces = [flce.Trace(capacity=8) for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    for k in range(args.steps):
        flce.flce_fwd(Xd, Wd, td, w.ignore_index, trace=traces[k])
    torch.cuda.synchronize(dev)
    lse_ms = [t_ms for tr in traces for kind, t_ms in tr.launches() if kind == "logits_lse"]
    lse_avg = sum(lse_ms) / len(lse_ms)
    flops = 2.0 * N * H * V
    peak_sust = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    peak_burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    achieved = flops / (lse_avg * 1e-3) / 1e12
    useful = flops / (ms * 1e-3) / 1e12
    line = {
        "metric": "tokens/s, fused linear CE loss only (flce_fwd), 1 GB300",
        "value": N / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded SplitMix64 + Box-Muller inputs, random-init LM head)",
        "config": workload_config(w, 1),
        "useful_tflops": useful, "frac_of_bf16_peak": useful / peak_burst,
        "roofline": {"bound": "tensor", "kernel": "logits_lse", "achieved": achieved,
                     "peak": peak_burst, "unit": "TFLOP/s", "frac": achieved / peak_burst,
                     "peak_kind": f"bf16 dense, burst ({peak_src})",
                     "frac_of_sustained": achieved / peak_sust, "flops_per_launch": flops,
                     "traffic": recorded_traffic("logits_lse", w.name)},
        "gpu_launches": 3 * args.steps, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def pinned_copy_rate(src, dst, reps: int = 3) -> float:
    """Best-of-reps GB/s of one copy between pinned host and device memory."""
    import torch
    best = float("inf")
    for _ in range(reps):
        torch.cuda.synchronize()
        a = time.perf_counter()
        dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize()
        best = min(best, time.perf_counter() - a)
    return src.numel() * src.element_size() / best / 1e9


def workload_config(w, n_gpus):
    return {"workload": w.name, "N": w.N, "H": w.H, "V": w.V, "input_dtype": w.dtype,
            "ignored_rows": w.n_ignored, "targets": w.t_dist,
            "parallelism": f"replicas x{n_gpus} (data-parallel shards, no collective)",
            "l2": "inputs larger than L2 (W alone exceeds the 129 MB L2); no flush"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="flce", choices=["flce", "reference"])
    ap.add_argument("--ce-dtype", default="bf16", choices=["bf16", "fp32"],
                    help="element type of the logits for --op ce_logits")
    ap.add_argument("--op", default="flce", choices=["flce", "fwd", "ce_logits"],
                    help="flce: the fused path (default); fwd: the loss-only path "
                         "(flce_fwd); ce_logits: cross-entropy on logits already in HBM "
                         "(logits = X W^T of the workload)")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--shape", default=None,
                    help="N,H,V: a synthetic case of that size with the workload's recipe "
                         "(profiling runs; not a bench line)")
    ap.add_argument("--e2e-steps", type=int, default=16)
    ap.add_argument("--vocab-chunk", type=int, default=0,
                    help="chunk width override (0 = the library's planner)")
    ap.add_argument("--ref-tokens", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args()
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        return launch_ranks(args.gpus, sys.argv[1:])
    ws_env = int(os.environ.get("WORLD_SIZE", "1"))
    if ws_env != args.gpus:
        ap.error(f"--gpus {args.gpus} does not match the launcher's WORLD_SIZE={ws_env}")

    from dataclasses import replace

    from flce_synth import WORKLOADS
    workload = WORKLOADS[args.workload]
    if args.shape:
        n_, h_, v_ = (int(x) for x in args.shape.split(","))
        workload = replace(workload, name=f"custom_{n_}x{h_}x{v_}", N=n_, H=h_, V=v_)
    if args.impl == "reference":
        return run_reference(args, workload)
    if args.op == "ce_logits":
        return run_ce_logits(args, workload)
    if args.op == "fwd":
        return run_fwd(args, workload)

    import torch
    import torch.distributed as dist

    import linear_cross_entropy_fwd_gb300 as flce
    from flce_synth import make_inputs

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    flce.load_library()
    peaks, peak_src = load_peaks()
    w = workload
    N, H, V = w.N, w.H, w.V

    X, W, t = make_inputs(w)
    Xd, Wd, td = X.to(dev), W.to(dev), t.to(dev)
    dX = torch.empty_like(Xd)
    dW = torch.empty((V, H), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(trace=None, info=None):
        return flce.flce_fwd_bwd_ex(Xd, Wd, td, w.ignore_index, dX=dX, dW=dW, trace=trace,
                                    info=info, vocab_chunk=args.vocab_chunk)

    info = {}
    step(info=info)  # plans the call (chunk width) before the warm-up proper
    for _ in range(args.warmup):
        step(info=info)
    torch.cuda.synchronize(dev)
    st = int(info["status"].item())
    if st != 0:
        raise RuntimeError(f"warm-up call reported status {st}")

    n_chunks = -(-V // info["vocab_chunk"])
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    uuid = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    uuid = None if uuid is None else str(uuid)
    if uuid and not uuid.startswith("GPU-"):
        uuid = "GPU-" + uuid
    sampler = ClockSampler(uuid)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)  # let the sampler take its first reading
    ev0.record(stream)
    for k in range(args.steps):
        step(info=info)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    if ws > 1:
        dist.barrier()
    ms = ev0.elapsed_time(ev1) / args.steps
    if int(info["status"].item()) != 0:
        raise RuntimeError("a timed call reported a kernel-side error")

    # Second timed region, same steps, with the library's per-launch events:
    # the events between launches stop each kernel's prologue from
    # overlapping its predecessor's tail, so this pass gives the per-kernel
    # breakdown and the roofline but not the headline time.
    traces = [flce.Trace(capacity=8 + 3 * n_chunks) for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    ev2 = torch.cuda.Event(enable_timing=True)
    ev3 = torch.cuda.Event(enable_timing=True)
    ev2.record(stream)
    for k in range(args.steps):
        step(trace=traces[k], info=info)
    ev3.record(stream)
    torch.cuda.synchronize(dev)
    ms_traced = ev2.elapsed_time(ev3) / args.steps
    if int(info["status"].item()) != 0:
        raise RuntimeError("a traced call reported a kernel-side error")
    ms_t = torch.tensor([ms], dtype=torch.float64, device=dev)
    if ws > 1:
        dist.all_reduce(ms_t, op=dist.ReduceOp.MAX)
    ms_max = float(ms_t.item())

    # per-kernel times from the library's per-launch events
    per_kind, launches = {}, 0
    for tr in traces:
        for kind, t_ms in tr.launches():
            d = per_kind.setdefault(kind, {"launches": 0, "ms": 0.0})
            d["launches"] += 1
            d["ms"] += t_ms
            launches += 1
    launches += args.steps  # the status-word kernel of each call
    useful = 6.0 * N * H * V
    flops_per_step = {"logits_lse": 2.0 * N * H * V, "logits_grad": 2.0 * N * H * V,
                      "dw": 2.0 * N * H * V, "dx": 2.0 * N * H * V}
    kernels = {}
    for kind, d in per_kind.items():
        ms_step = d["ms"] / args.steps
        e = {"launches_per_step": d["launches"] / args.steps, "ms_per_step": ms_step,
             "share": d["ms"] / (ms_traced * args.steps)}
        if kind in flops_per_step:
            e["tflops"] = flops_per_step[kind] / (ms_step * 1e-3) / 1e12
        kernels[kind] = e
    dom = max((k for k in kernels if k in GEMM_KINDS), key=lambda k: kernels[k]["ms_per_step"])
    dom_launches = per_kind[dom]["launches"]
    dom_avg_ms = per_kind[dom]["ms"] / dom_launches
    flops_per_launch = flops_per_step[dom] * args.steps / dom_launches
    peak_sust = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    peak_burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    achieved = flops_per_launch / (dom_avg_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak_burst,
                "unit": "TFLOP/s", "frac": achieved / peak_burst,
                "peak_kind": f"bf16 dense, burst ({peak_src})",
                "frac_of_sustained": achieved / peak_sust,
                "flops_per_launch": flops_per_launch,
                "traffic": recorded_traffic(dom, w.name)}

    value = ws * N / (ms_max * 1e-3)
    useful_tflops = useful / (ms_max * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded SplitMix64 + Box-Muller inputs, random-init LM head)",
        "config": workload_config(w, ws),
        "useful_tflops": useful_tflops,
        "frac_of_bf16_peak": useful_tflops / peak_burst,
        "frac_of_bf16_peak_sustained": useful_tflops / peak_sust,
        "peaks": {"bf16_tflops": peak_burst, "bf16_tflops_sustained": peak_sust,
                  "source": peak_src},
        "workspace_bytes": info.get("workspace_bytes"),
        "vocab_chunk": info.get("vocab_chunk"),
        "logits_bytes_avoided": N * V * 4,
        "roofline": roofline, "kernels": kernels, "ms_per_step_traced": ms_traced,
        "gpu_launches": launches,
        "clocks": clocks,
    }

    # end to end through the host-buffer entry point (pinned memory)
    if not args.no_e2e:
        Xh, Wh, th = X.pin_memory(), W.pin_memory(), t.pin_memory()
        dXh = torch.empty_like(Xh).pin_memory()
        dWh = torch.empty((V, H), dtype=torch.float32).pin_memory()
        flce.flce_fwd_bwd_host(Xh, Wh, th, w.ignore_index, dX=dXh, dW=dWh)
        # the host link's rates just before the timed calls (context for e2e)
        link = {"h2d_gbs": pinned_copy_rate(Wh, Wd), "d2h_gbs": pinned_copy_rate(dW, dWh)}
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        per_call = []
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            a = time.perf_counter()
            flce.flce_fwd_bwd_host(Xh, Wh, th, w.ignore_index, dX=dXh, dW=dWh)
            per_call.append(time.perf_counter() - a)  # the call is synchronous
        torch.cuda.synchronize(dev)
        e2e_s = (time.perf_counter() - t0) / args.e2e_steps
        e_t = torch.tensor([e2e_s], dtype=torch.float64, device=dev)
        if ws > 1:
            dist.all_reduce(e_t, op=dist.ReduceOp.MAX)
        line["e2e"] = {"value": ws * N / float(e_t.item()), "unit": "tokens/s",
                       "h2d_bytes_per_step": Xh.numel() * Xh.element_size() +
                       Wh.numel() * Wh.element_size() + th.numel() * 8,
                       "d2h_bytes_per_step": dXh.numel() * dXh.element_size() +
                       dWh.numel() * 4 + 4,
                       "steps": args.e2e_steps,
                       "ms_per_call": [round(1e3 * x, 3) for x in per_call],
                       "host_link": link,
                       "timer": "host wall clock around synchronous calls"}
    if ws > 1:
        dist.barrier()
    if rank == 0:
        if ws == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w, X, W, t)
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
