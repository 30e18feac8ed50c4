"""Benchmark of the Laya BF16 encoder forward pass (embedding + 28 encoder +
2 decision layers) on GB300, one JSON line on stdout.

A step is one full forward pass over one batch of the workload (default: the
full-size stack at 1 x 48 tokens).  `value` is valid tokens per second with
ids and lengths already resident in device memory (graph replay through
laya_enc_run_device); `e2e` is the same metric through laya_enc_run with HOST
ids/lengths (H2D upload inside) plus a device-to-host read of the hidden
states every step.  Weights (735 MB of projections + 103 MB of embedding) are
larger than the 126 MB L2, so every step streams them from HBM; no flush.

Multi-GPU: the forward pass has no exchange step, so N GPUs run N independent
replicas (one process per GPU under torchrun), `value` counts every rank's
tokens over the slowest rank's time.

--impl reference times the CPU oracle (the only other implementation there
is) on the host cores, on the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from transformer_encoder_bf16_gb300 import synth  # noqa: E402

METRIC = "encoder fwd p50 ms & tokens/s (28+2 layers, BF16, 1 GB300); % of roofline"
UNIT = "tokens/s"
# H800 CUDA-event p50 of the Rust encoder at 1 x 48 (PR #49, run 1), other hardware
PUBLISHED_MS = {"full_1x48": 2.771, "full_4x64": 3.195, "full_1x464": 3.742,
                "full_4x464": 7.545, "full_16x512": 25.785}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# The roofline kernel is a projection: the sources its GEMM kernels are built from.
GEMM_SOURCES = ("gemm.cu", "internal.h", "packing.cuh", "ptx.cuh", "rowstats.cuh")


def csrc_sha16():
    """Hash of the GEMM kernel sources, to tell whether recorded ncu counters
    still apply: the code only (line comments and blank lines dropped, so that
    a comment edit does not void a capture)."""
    import hashlib
    import re
    d = os.path.join(ROOT, "transformer_encoder_bf16_gb300", "csrc")
    h = hashlib.sha256()
    for name in GEMM_SOURCES:
        with open(os.path.join(d, name), encoding="utf-8") as fh:
            for line in fh:
                code = re.sub(r"//.*$", "", line).strip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def recorded_traffic(workload, kernel_class):
    """DRAM bytes per launch from the committed ncu capture, or None when the
    kernels changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        if d.get("csrc_sha16") != csrc_sha16():
            return None
        v = d.get(workload, {}).get(kernel_class)
        return float(v) if v is not None else None
    except Exception:
        return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
            return d, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def peak_value(peaks, key):
    for k, v in peaks.items():
        if k == key and isinstance(v, (int, float)):
            return float(v)
    # tolerate nested layouts, e.g. {"hbm_gbs": {"value": ...}}
    v = peaks.get(key)
    if isinstance(v, dict):
        for kk in ("value", "median", "max"):
            if isinstance(v.get(kk), (int, float)):
                return float(v[kk])
    return FALLBACK_PEAKS[key]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=2)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(mx)) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def gemm_shapes(model):
    H, I = model["hidden"], model["intermediate"]
    # class -> (N_w, K, N_out, residual?)
    return {"qkv": (3 * H, H, 3 * H, False), "out_proj": (H, H, H, True),
            "up_geglu": (2 * I, H, I, False), "down": (H, I, H, True)}


def algorithmic(model, cls, M):
    """(bytes, flops) one launch of a kernel class must move / compute."""
    H = model["hidden"]
    g = gemm_shapes(model)
    if cls in g:
        Nw, K, N, res = g[cls]
        b = 2 * (Nw * K + M * K + M * N + (M * N if res else 0))
        return b, 2.0 * M * Nw * K
    if cls == "norm":
        return 2 * (2 * M * H + H), 0.0
    if cls == "embed_norm":
        return 2 * (2 * M * H + H) + 4 * M, 0.0
    if cls == "rope":
        return 2 * (2 * 2 * M * H), 0.0
    if cls == "attention":
        return 2 * (3 * M * H + M * H), 0.0
    if cls == "fused":
        # the whole forward: every layer's four projections (weights once)
        L = model["n_encoder_layers"] + model["n_decision_layers"]
        b = f = 0.0
        for k in g:
            kb, kf = algorithmic(model, k, M)
            b, f = b + kb, f + kf
        return L * b, L * f
    return 0, 0.0


def cpu_baseline(model, weights, ids, lengths, budget_s=12.0):
    """The oracle as it stands, on the host cores, for about budget_s seconds."""
    import oracle
    oracle.build()
    cores = oracle.set_threads(0)
    valid = int(np.sum(lengths))
    runs, t0 = 0, time.perf_counter()
    while True:
        oracle.forward(model, weights, ids, lengths)
        runs += 1
        el = time.perf_counter() - t0
        if el >= budget_s or runs >= 50:
            break
    return {"value": valid * runs / el, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{runs} full forward pass(es) of the workload ({valid} valid tokens each), "
                      f"{el:.1f} s, OpenMP over {cores} threads"}


def run_reference(args, model, weights, ids, lengths, world, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    cores = oracle.set_threads(0)
    valid = int(np.sum(lengths))
    for _ in range(args.warmup):
        oracle.forward(model, weights, ids, lengths)
    times = []
    t_all = time.perf_counter()
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.forward(model, weights, ids, lengths)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_all > args.reference_budget:
            break
    total = sum(times)
    value = valid * len(times) / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": len(times), "warmup": args.warmup,
            "ms_per_step": 1000 * total / len(times), "p50_ms": 1000 * float(np.median(times)),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": {"workload": args.workload, "batch": int(ids.shape[0]),
                                            "seq": int(ids.shape[1]), "valid_tokens": valid},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{len(times)} full forward passes of the workload on the "
                                       f"host cores (steps capped at {args.reference_budget:.0f} s)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="full_1x48", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--reference-budget", type=float, default=150.0)
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    rank, local_rank, world = dist_env()
    model, B, S, seed, lr = synth.WORKLOADS[args.workload]
    weights = synth.make_weights(model, seed)
    ids, lengths = synth.make_inputs(model, B, S, seed, lr)
    valid = int(np.sum(lengths))

    if args.impl == "reference":
        run_reference(args, model, weights, ids, lengths, world, rank)
        return

    import torch
    import transformer_encoder_bf16_gb300 as te
    from transformer_encoder_bf16_gb300 import build as tebuild

    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    else:
        torch.cuda.set_device(0)
    tebuild.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    enc = te.Encoder(model, te.upload_weights(weights, dev))
    stream = torch.cuda.Stream(device=dev)
    H = model["hidden"]
    out = torch.empty((B, S, H), dtype=torch.bfloat16, device=dev)
    ids_dev = torch.from_numpy(ids).to(dev)
    len_dev = torch.from_numpy(lengths).to(dev)

    # ---- device-resident timing (graph replay) -----------------------------
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            enc.run_device(ids_dev, len_dev, out, stream)
    enc.check(stream)
    # first run of the shape: workspace allocation, two eager warm-ups, graph
    # capture and instantiation (host wall time, reported apart from the replays)
    first_shape = enc.cache_stats()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(torch.cuda.current_device() if world == 1 else local_rank)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    first = torch.cuda.Event(enable_timing=True)
    last = torch.cuda.Event(enable_timing=True)
    first.record(stream)
    for i in range(args.steps):
        starts[i].record(stream)
        enc.run_device(ids_dev, len_dev, out, stream)
        ends[i].record(stream)
    last.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    enc.check(stream)
    total_ms = first.elapsed_time(last)
    step_ms = np.array([s.elapsed_time(e) for s, e in zip(starts, ends)])
    total_ms_max = max_over_ranks(total_ms, world)
    value = valid * args.steps * world / (total_ms_max / 1000.0)

    # ---- end-to-end through the public host API -----------------------------
    host_out = torch.empty((B, S, H), dtype=torch.bfloat16, pin_memory=True)
    for _ in range(3):
        enc.run(ids, lengths, out, stream)
        host_out.copy_(out, non_blocking=True)
        stream.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    e2e_times = []
    for _ in range(args.steps):
        ts = time.perf_counter()
        with torch.cuda.stream(stream):
            enc.run(ids, lengths, out, stream)
            host_out.copy_(out, non_blocking=True)
        stream.synchronize()
        e2e_times.append(time.perf_counter() - ts)
    e2e_total = max_over_ranks(time.perf_counter() - t0, world)
    enc.check(stream)

    # ---- per-kernel device time, eager launches bracketed by events ---------
    enc.set_profiling(True)
    enc.profile_read()
    for _ in range(args.steps):
        enc.run_device(ids_dev, len_dev, out, stream)
    prof = enc.profile_read()
    enc.set_profiling(False)
    peaks, peak_src = load_peaks()
    # tokens the kernels process: batches of several rows are packed (the
    # padding is skipped), a single row is processed whole
    M = valid if B > 1 else B * S
    best = None
    for cls, (ms, n) in prof.items():
        if n == 0:
            continue
        if best is None or ms > best[1]:
            best = (cls, ms, n)
    cls, ms, n = best
    avg_s = ms / n / 1000.0
    nbytes, flops = algorithmic(model, cls, M)
    hbm_peak = peak_value(peaks, "hbm_gbs")
    tc_peak = peak_value(peaks, "bf16_tflops")
    t_mem = nbytes / (hbm_peak * 1e9)
    t_tc = flops / (tc_peak * 1e12) if flops else 0.0
    if t_tc > t_mem:
        roof = {"bound": "tensor", "achieved": flops / avg_s / 1e12, "peak": tc_peak,
                "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": nbytes / avg_s / 1e9, "peak": hbm_peak, "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = recorded_traffic(args.workload, cls)
    roof["kernel"] = cls
    roof["avg_launch_us"] = avg_s * 1e6
    roof["launches"] = n
    roof["algorithmic_bytes_per_launch"] = nbytes
    roof["algorithmic_flops_per_launch"] = flops
    roof["peak_source"] = f"{peak_src} ({'MEASURED_PEAKS.json' if peak_src == 'measured' else 'fallback'})"
    kernel_ms_per_step = {k: (v[0] / args.steps) for k, v in prof.items()}

    # whole-forward roofline: weights + activations at HBM peak vs flops at tensor peak
    fwd_bytes = sum(algorithmic(model, k, M)[0] * (c / args.steps) for k, (_, c) in prof.items())
    fwd_flops = sum(algorithmic(model, k, M)[1] * (c / args.steps) for k, (_, c) in prof.items())
    t_roof = max(fwd_bytes / (hbm_peak * 1e9), fwd_flops / (tc_peak * 1e12))
    p50 = float(np.median(step_ms))

    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            try:
                cpu = cpu_baseline(model, weights, ids, lengths)
            except Exception as ex:  # the oracle is a baseline, not the product
                cpu = {"value": None, "unit": UNIT, "cores": 0, "kind": "oracle",
                       "sample": f"unavailable: {ex}"}
        pub = PUBLISHED_MS.get(args.workload)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_ms_max / args.steps,
            "padded_tokens_per_s": B * S * args.steps * world / (total_ms_max / 1000.0),
            "first_shape_ms": {"workspace_setup": first_shape["setup_ms"],
                               "warmup_capture_instantiate": first_shape["capture_ms"]},
            "p50_ms": p50, "p95_ms": float(np.percentile(step_ms, 95)),
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": (value / world) / (valid / (pub / 1000.0)) if pub else None,
            "vs_baseline_ref": (f"H800 CUDA-event p50 {pub} ms (PR #49, Rust, run 1); other hardware"
                                if pub else None),
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": args.workload, "batch": B, "seq": S, "valid_tokens": valid,
                       "l2": "weights 838 MB > L2 (129 MB): streamed from HBM every step, no flush",
                       "graphs": True, "pdl": os.environ.get("LAYA_NO_PDL", "0") in ("", "0"),
                       "parallelism": f"replicas x{world}"},
            "clocks": clk,
            "e2e": {"value": valid * args.steps * world / e2e_total, "unit": UNIT,
                    "p50_ms": 1000 * float(np.median(e2e_times)),
                    "h2d_bytes_per_step": 4 * (B * S + B), "d2h_bytes_per_step": 2 * B * S * H},
            "gpu_launches": enc.launch_count(B, S) * args.steps,
            "roofline": roof,
            "forward_roofline": {"bytes": fwd_bytes, "flops": fwd_flops,
                                 "t_roof_us": t_roof * 1e6, "frac_of_p50": t_roof / (p50 / 1000)},
            "kernel_ms_per_step": kernel_ms_per_step,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    enc.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
