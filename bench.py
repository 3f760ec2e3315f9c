#!/usr/bin/env python
"""Benchmark of the MoDA forward hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...        # the fp64 CPU oracle arm

One step = the whole hot path over one batch of synthetic input resident in
HBM: moda_fwd_layer_major(...) on the depth K/V as the layers wrote them
([L,T,Hk,d]); the depth relayout (the chunk-aware grouping) happens inside the
forward's copies. The packed path (moda_pack_depth(kd), moda_pack_depth(vd),
moda_fwd) is timed beside it. The headline workload is the long-context layer
(T=65536, Hq=16, Hk=4, d=128, L=48).
Throughput counts 4*d*Hq*(T(T+1)/2 + T*L) FLOPs per step (causal and valid
depth work only). Under torchrun each rank runs an independent replica on its
own GPU (weak scaling); value = all ranks' FLOPs / the slowest rank's time.

Also reported on the same JSON line:
  fwd             the step's forward (CUDA events on its stream), % of bf16 peak
  packed_path     pack kd + pack vd + moda_fwd on the packed streams
  overhead_vs_L0  t_fwd(L) / t_fwd(L=0) - 1 for the same T, Hq, Hk, d
  roofline        the dominant kernel (the forward) against the measured peak
  e2e             same metric through the host-buffer call
                  (moda_fwd_layer_major_host): inputs copied from pinned host
                  memory and o, lse copied back inside the timed region
  cpu_baseline    the fp64 oracle on the host cores, on a bounded row sample
  clocks          nvidia-smi samples taken during the timed region
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
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sequence_depth_attention_gb300 import inputs as wl  # noqa: E402

METRIC = "MoDA fwd TFLOP/s and % bf16 tensor peak at T=64K; overhead vs L=0"
FWD_SOURCES = ["sequence_depth_attention_gb300/csrc/fwd_tc.cu",
               "sequence_depth_attention_gb300/csrc/sm103.cuh",
               "sequence_depth_attention_gb300/csrc/softmax_block.cuh"]
PACK_SOURCES = ["sequence_depth_attention_gb300/csrc/pack_depth.cu"]
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# GB300 nominal dense bf16 tensor rate (no 2:4 sparsity), per GPU
NOMINAL_BF16_TFLOPS = 2250.0


def workload_by_name(name):
    for w in [*wl.ALL, wl.LONG_L0, wl.LONG_32K, *wl.TABLE2]:
        if w.name == name:
            return w
    raise SystemExit(f"unknown workload {name}; known: {[w.name for w in wl.ALL]}")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def sources_sha(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload, paths):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}_traffic.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha256") != sources_sha(paths):
            return None
        return float(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi -lms 200 while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device):
        self.proc = None
        self.lines = []
        ident = None
        try:
            u = str(torch.cuda.get_device_properties(device).uuid)
            ident = u if u.startswith("GPU-") else f"GPU-{u}"
        except Exception:
            ident = None
        self.ident = ident

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.ident:
            cmd += ["-i", self.ident]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- CPU arm
def oracle_sample(w, host, rows_budget_s, seed=0, nthreads=None):
    """Time the fp64 oracle on a seeded sample of rows for about rows_budget_s
    seconds. Returns (flops, seconds, rows, threads)."""
    import numpy as np

    import oracle
    from sequence_depth_attention_gb300.inputs import bf16_bits
    nthreads = nthreads or (os.cpu_count() or 1)
    b = {n: bf16_bits(t) for n, t in host.items()}
    kd = b["kd"] if w.L else None
    vd = b["vd"] if w.L else None
    rng = np.random.default_rng(seed)
    flops = 0.0
    rows = 0
    t0 = time.perf_counter()
    batch = nthreads
    while True:
        ts = rng.integers(0, w.T, size=batch)
        hs = rng.integers(0, w.Hq, size=batch)
        oracle.rows(b["q"], b["k"], b["v"], kd, vd, w.scale, ts, hs, nthreads=nthreads)
        flops += float(np.sum(4.0 * w.d * (ts + 1 + w.L)))
        rows += batch
        el = time.perf_counter() - t0
        if el >= rows_budget_s:
            return flops, el, rows, nthreads
        batch = min(batch * 2, max(nthreads, int(rows * (rows_budget_s - el) / max(el, 1e-3))))


def max_over_ranks(val, dist=None, device="cpu"):
    """Max of a per-rank float over all ranks (identity on one rank)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(val)
    t = torch.tensor([float(val)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank, ms_per_step, world):
    """Whole-job throughput: every rank's FLOPs over the slowest rank's time."""
    return world * flops_per_rank / (ms_per_step * 1e-3) / 1e12


def host_inputs(w):
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    x = wl.make_inputs(w, device=dev)
    return {n: t.cpu() for n, t in x.items()}


def run_reference(args, w, rank):
    if rank != 0:
        return
    host = host_inputs(w)
    per_step = args.cpu_seconds if args.cpu_seconds_set else \
        max(1.0, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    for i in range(args.warmup):
        oracle_sample(w, host, per_step, seed=1000 + i)
    flops = secs = 0.0
    rows = threads = 0
    for i in range(args.steps):
        f, s, r, threads = oracle_sample(w, host, per_step, seed=i)
        flops += f
        secs += s
        rows += r
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, args.gpus),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows} (t, h) rows drawn uniformly from the {w.name} workload "
                                   f"(seeded), ~{per_step:.0f} s of oracle work per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(w, n):
    kvd = 2 * w.L * w.T * w.Hk * w.d * 2
    return {"workload": w.name, "T": w.T, "Hq": w.Hq, "Hk": w.Hk, "G": w.G, "d": w.d, "L": w.L,
            "batch": 1, "causal": True, "scale": "1/sqrt(d)",
            "step": "moda_fwd_layer_major on kd, vd [L,T,Hk,d] (the depth relayout happens in the "
                    "forward's copies); the packed path is reported in packed_path",
            "l2": f"inputs larger than L2 (kd+vd {kvd / 1e9:.2f} GB, q {w.T * w.Hq * w.d * 2 / 1e6:.0f} MB)",
            "parallelism": f"replicas x{n}" if n > 1 else "single GPU"}


def time_calls(fn, stream, n, flush=None):
    """Median CUDA-event time (ms) of n calls of fn() on `stream`, each after
    an L2 flush (a write of `flush`, larger than L2) when one is given."""
    times = []
    for _ in range(n):
        if flush is not None:
            with torch.cuda.stream(stream):
                flush.fill_(1.0)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in times)


def config_sweep(moda, dev, stream, peaks, steps, warmup):
    """moda_fwd on every workload other than the headline one: time, TFLOP/s,
    fraction of peak, the L = 0 forward of the same shape and the overhead of
    the depth slots in both conventions, the CUDA-core depth variant beside
    the fused one, and the layer-major forward and the two depth packs (the
    two ways to the same result). L2 is flushed (512 MB written) before every
    timed call, so no workload runs out of a warm L2."""
    peak = float(peaks["bf16_tflops"])
    flush = torch.empty(128 << 20, dtype=torch.float32, device=dev)
    out = {}
    # the five workloads, then the pages' Table-2 kernel shape at T=16384 (d = 64) as context
    for w in [wl.TINY, wl.LAYER_700M, *wl.GQA_SWEEP, *wl.DEPTH_SWEEP, wl.TABLE2[2]]:
        x = wl.make_inputs(w, device=dev)
        q, k, v = x["q"], x["k"], x["v"]
        kd = moda.moda_pack_depth(x["kd"], stream=stream) if w.L else None
        vd = moda.moda_pack_depth(x["vd"], stream=stream) if w.L else None
        kd_lm, vd_lm = x["kd"], x["vd"]
        del x
        o = torch.empty_like(q)
        lse = torch.empty((w.T, w.Hq), dtype=torch.float32, device=dev)

        def fwd(cc=False, L=w.L):
            moda.moda_fwd(q, k, v, kd if L else None, vd if L else None, w.scale, o=o, lse=lse,
                          stream=stream, depth_on_cuda_cores=cc)

        for _ in range(warmup):
            fwd()
        ms = time_calls(fwd, stream, steps, flush)
        F = w.flops()
        tf = F / (ms * 1e-3) / 1e12
        rec = {"T": w.T, "Hq": w.Hq, "Hk": w.Hk, "G": w.G, "d": w.d, "L": w.L,
               "fwd_ms": ms, "tflops": tf, "pct_peak_burst": 100 * tf / peak,
               "pct_nominal_peak": 100 * tf / NOMINAL_BF16_TFLOPS}
        if w.L:
            for _ in range(warmup):
                fwd(L=0)
            ms0 = time_calls(lambda: fwd(L=0), stream, steps, flush)
            for _ in range(2):
                fwd(cc=True)
            ms_cc = time_calls(lambda: fwd(cc=True), stream, max(3, steps // 2), flush)
            def fwd_lm():
                moda.moda_fwd_layer_major(q, k, v, kd_lm, vd_lm, w.scale, o=o, lse=lse, stream=stream)

            def packs():
                moda.moda_pack_depth(kd_lm, kd, stream=stream)
                moda.moda_pack_depth(vd_lm, vd, stream=stream)

            for _ in range(warmup):
                fwd_lm()
            ms_lm = time_calls(fwd_lm, stream, steps, flush)
            ms_pack = time_calls(packs, stream, max(3, steps // 2), flush)
            rec.update({"L0_ms": ms0, "overhead_vs_L0": ms / ms0 - 1.0,
                        "extra_time_pages_convention": 1.0 - ms0 / ms,
                        "cuda_core_depth_ms": ms_cc,
                        "faster_depth": "tensor cores" if ms <= ms_cc else "cuda cores",
                        "layer_major_ms": ms_lm, "layer_major_tflops": F / (ms_lm * 1e-3) / 1e12,
                        "pack_kd_vd_ms": ms_pack})
        st = moda.moda_get_device_error(stream)
        if st != 0:
            raise SystemExit(f"device error in the sweep ({w.name}): {moda.moda_status_string(st)}")
        if w in wl.TABLE2:
            rec["note"] = "context: the pages' Table-2 kernel shape (B=1, d=64, G=8, L=64), not a workload"
        out[w.name] = rec
        del q, k, v, kd, vd, kd_lm, vd_lm, o, lse
    del flush
    torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------- GPU arm
def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="moda", choices=["moda", "reference"])
    ap.add_argument("--workload", default=wl.LONG.name)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--decode-steps", type=int, default=20,
                    help="timed moda_decode calls reported in the 'decode' object (0 = skip)")
    ap.add_argument("--bwd-steps", type=int, default=3,
                    help="timed moda_bwd calls reported in the 'bwd' object (0 = skip)")
    ap.add_argument("--proj-steps", type=int, default=5,
                    help="timed moda_kv_proj_write calls reported in the 'kv_proj' object (0 = skip)")
    ap.add_argument("--variant-steps", type=int, default=3,
                    help="timed moda_fwd_depth_cc calls for the 'depth_variant' object (0 = skip)")
    ap.add_argument("--config-steps", type=int, default=10,
                    help="timed moda_fwd calls per workload in the 'configs' object (0 = skip)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=None,
                    help="seconds of oracle work for cpu_baseline (default 10) or per "
                         "reference-arm step (default: sized to the run)")
    args = ap.parse_args(argv)
    args.cpu_seconds_set = args.cpu_seconds is not None
    if args.cpu_seconds is None:
        args.cpu_seconds = 10.0
    if args.warmup < 3 and args.impl == "moda":
        print("note: warm-up raised to the minimum of 3", file=sys.stderr)
        args.warmup = 3
    w = workload_by_name(args.workload)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, w, rank)

    import sequence_depth_attention_gb300 as moda
    from sequence_depth_attention_gb300 import build as mbuild
    mbuild.build()
    moda.load()

    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)

    x = wl.make_inputs(w, device=dev)
    q, k, v, kd_raw, vd_raw = (x[n] for n in ("q", "k", "v", "kd", "vd"))
    kd = torch.empty((w.Hk, w.T, w.L, w.d), dtype=torch.bfloat16, device=dev)
    vd = torch.empty_like(kd)
    o = torch.empty_like(q)
    lse = torch.empty((w.T, w.Hq), dtype=torch.float32, device=dev)
    K, W = args.steps, args.warmup
    fwd_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
    pack_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
    pfwd_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]

    # The step: the forward on the depth K/V as the layers wrote them
    # ([L,T,Hk,d]); its copies gather each tile's depth rows (the depth
    # relayout happens inside the forward, no separate pass).
    def step(i=None):
        if i is not None:
            fwd_ev[i][0].record(stream)
        moda.moda_fwd_layer_major(q, k, v, kd_raw if w.L else None, vd_raw if w.L else None,
                                  w.scale, o=o, lse=lse, stream=stream)
        if i is not None:
            fwd_ev[i][1].record(stream)

    # The packed path beside it: two moda_pack_depth passes, then moda_fwd on
    # the packed streams (timed after the headline, not part of its step).
    def packed_step(i):
        pack_ev[i][0].record(stream)
        if w.L:
            moda.moda_pack_depth(kd_raw, kd, stream=stream)
            moda.moda_pack_depth(vd_raw, vd, stream=stream)
        pack_ev[i][1].record(stream)
        pfwd_ev[i][0].record(stream)
        moda.moda_fwd(q, k, v, kd if w.L else None, vd if w.L else None, w.scale, o=o, lse=lse,
                      stream=stream)
        pfwd_ev[i][1].record(stream)

    launches_per_step = 1

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(W):
        step()
    st = moda.moda_get_device_error(stream)
    if st != 0:
        raise SystemExit(f"device error after warm-up: {moda.moda_status_string(st)}")

    clocks = ClockSampler(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    clocks.start()
    time.sleep(0.3)
    start.record(stream)
    for i in range(K):
        step(i)
    end.record(stream)
    barrier()
    clk = clocks.stop()
    ms_step = max_over_ranks(start.elapsed_time(end) / K, dist, dev)
    fwd_ms = statistics.mean(a.elapsed_time(b) for a, b in fwd_ev)
    st = moda.moda_get_device_error(stream)
    if st != 0:
        raise SystemExit(f"device error in timed region: {moda.moda_status_string(st)}")

    # the packed path: pack kd and vd, then moda_fwd on the packed streams
    for i in range(min(W, K)):
        packed_step(i)
    torch.cuda.synchronize(dev)
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    for i in range(K):
        packed_step(i)
    p1.record(stream)
    torch.cuda.synchronize(dev)
    packed_step_ms = p0.elapsed_time(p1) / K
    pack_ms = statistics.mean(a.elapsed_time(b) for a, b in pack_ev)
    pfwd_ms = statistics.mean(a.elapsed_time(b) for a, b in pfwd_ev)
    st = moda.moda_get_device_error(stream)
    if st != 0:
        raise SystemExit(f"device error in the packed path: {moda.moda_status_string(st)}")

    # plain causal GQA (L = 0) with the same kernel, same T/Hq/Hk/d
    w0 = w.with_L(0)
    for _ in range(W):
        moda.moda_fwd(q, k, v, None, None, w.scale, o=o, lse=lse, stream=stream)
    e0 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    torch.cuda.synchronize(dev)
    for a, b in e0:
        a.record(stream)
        moda.moda_fwd(q, k, v, None, None, w.scale, o=o, lse=lse, stream=stream)
        b.record(stream)
    torch.cuda.synchronize(dev)
    fwd0_ms = statistics.mean(a.elapsed_time(b) for a, b in e0)

    peaks, peaks_src = load_peaks()
    F = w.flops()
    value = job_tflops(F, ms_step, world)
    fwd_tflops = F / (fwd_ms * 1e-3) / 1e12
    fwd0_tflops = w0.flops() / (fwd0_ms * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    pack_bytes = 2 * 2 * (w.L * w.T * w.Hk * w.d * 2)  # read + write, kd and vd
    traffic = recorded_traffic("moda_fwd_layer_major", w.name, FWD_SOURCES)
    pfwd_tflops = F / (pfwd_ms * 1e-3) / 1e12

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_of(w, world),
        "fwd": {"ms": fwd_ms, "tflops": fwd_tflops,
                "pct_nominal_peak": 100 * fwd_tflops / NOMINAL_BF16_TFLOPS,
                "pct_peak_burst": 100 * fwd_tflops / peak,
                "flops_per_launch": F,
                "peaks": f"nominal {NOMINAL_BF16_TFLOPS:.0f} TFLOP/s dense bf16; measured burst "
                         f"{peak:.1f} (cuBLAS bf16 GEMM, {peaks_src})"},
        "fwd_L0": {"ms": fwd0_ms, "tflops": fwd0_tflops, "pct_peak_burst": 100 * fwd0_tflops / peak},
        "overhead_vs_L0": fwd_ms / fwd0_ms - 1.0,
        "extra_time_pages_convention": 1.0 - fwd0_ms / fwd_ms,
        "packed_path": {
            "step_ms": packed_step_ms, "tflops": F / (packed_step_ms * 1e-3) / 1e12,
            "fwd_ms": pfwd_ms, "fwd_tflops": pfwd_tflops,
            "fwd_pct_peak_burst": 100 * pfwd_tflops / peak,
            "pack": {"ms_for_kd_and_vd": pack_ms,
                     "gbs": (pack_bytes / (pack_ms * 1e-3) / 1e9) if w.L and pack_ms > 0 else None,
                     "pct_hbm": (100 * pack_bytes / (pack_ms * 1e-3) / 1e9 / peaks["hbm_gbs"])
                     if w.L and pack_ms > 0 else None},
            "note": "moda_pack_depth(kd) + moda_pack_depth(vd) + moda_fwd on the packed "
                    "[Hk,T,L,d] streams, the same result"},
        "roofline": {"bound": "tensor", "achieved": fwd_tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": fwd_tflops / peak, "traffic": traffic,
                     "peak_source": f"{peaks_src} bf16 dense burst (MEASURED_PEAKS.json)"
                     if peaks_src == "measured" else "fallback 1.9 PFLOP/s bf16",
                     "kernel": "moda_fwd_layer_major (moda_fwd_tc_kernel<128>)"},
        "gpu_launches": launches_per_step * K,
        "clocks": clk,
    }

    # ---- end to end: pinned host inputs in, o and lse out, every step ----
    # (measured right after the device-resident timing, before the other
    # phases' allocations can change the host link's behaviour)
    if not args.no_e2e:
        hq, hk_, hv = (t.cpu().pin_memory() for t in (q, k, v))
        hkd, hvd = (t.cpu().pin_memory() for t in (kd_raw, vd_raw))
        # The library's host-buffer forward: each call copies that step's
        # inputs (every byte of them, from pinned host memory) into a device
        # workspace, runs the forward and copies o and lse back. Calls
        # alternate between two streams, each with its own workspace and host
        # outputs, so one call's copies overlap the other's forward; the host
        # link is the bound.
        streams2 = [stream, torch.cuda.Stream(device=dev)]
        need = moda.moda_fwd_host_workspace_bytes(w.T, w.Hq, w.Hk, w.d, w.L)
        wss = [torch.empty((need,), dtype=torch.uint8, device=dev) for _ in range(2)]
        hos = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for _ in range(2)]
        hls = [torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True) for _ in range(2)]

        def e2e_step(i):
            j = i % 2
            moda.moda_fwd_layer_major_host(hq, hk_, hv, hkd if w.L else None,
                                           hvd if w.L else None, w.scale, o=hos[j], lse=hls[j],
                                           workspace=wss[j], stream=streams2[j])

        for i in range(W):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(streams2[0])
        streams2[1].wait_event(a)
        for i in range(K):
            e2e_step(i)
        joined = torch.cuda.Event()
        joined.record(streams2[1])
        streams2[0].wait_event(joined)
        b.record(streams2[0])
        barrier()
        e2e_ms = max_over_ranks(a.elapsed_time(b) / K, dist, dev)
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk_, hv)) + \
            (sum(t.numel() * t.element_size() for t in (hkd, hvd)) if w.L else 0)
        d2h = hos[0].numel() * hos[0].element_size() + hls[0].numel() * hls[0].element_size()
        line["e2e"] = {"value": job_tflops(F, e2e_ms, world), "unit": "TFLOP/s",
                       "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h,
                       "transfer": "moda_fwd_layer_major_host every step: q, k, v, kd, vd copied "
                                   "from pinned host memory into a device workspace, the forward, "
                                   "o and lse copied back; calls alternate between two streams "
                                   "and workspaces so one call's copies overlap the other's "
                                   "forward; the timed region runs from the first call's first "
                                   "copy to the last call's read-back"}
        host = {"q": hq, "k": hk_, "v": hv, "kd": hkd, "vd": hvd}
        del wss  # the two device workspaces
    else:
        host = None

    # ---- the depth variant choice: CUDA-core depth in a second pass ----
    if w.L and args.variant_steps > 0:
        moda.moda_fwd(q, k, v, kd, vd, w.scale, o=o, lse=lse, stream=stream,
                      depth_on_cuda_cores=True)
        ec = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.variant_steps)]
        torch.cuda.synchronize(dev)
        for a, b in ec:
            a.record(stream)
            moda.moda_fwd(q, k, v, kd, vd, w.scale, o=o, lse=lse, stream=stream,
                          depth_on_cuda_cores=True)
            b.record(stream)
        torch.cuda.synchronize(dev)
        cc_ms = statistics.median(a.elapsed_time(b) for a, b in ec)
        line["depth_variant"] = {
            "tensor_core_depth_ms": fwd_ms, "cuda_core_depth_ms": cc_ms,
            "L0_ms": fwd0_ms, "tensor_core_depth_cost_ms": fwd_ms - fwd0_ms,
            "cuda_core_depth_cost_ms": cc_ms - fwd0_ms,
            "chosen": "tensor cores (moda_fwd)" if fwd_ms <= cc_ms else "cuda cores",
            "note": "cuda-core variant = moda_fwd_depth_cc: the L=0 forward, then one warp per "
                    "(KV head, position) scoring its L slots and merging into o and lse"}

    # ---- layer-by-layer depth writes (the model path that replaces the pack) ----
    if w.L:
        layers_k = [kd_raw[l] for l in range(w.L)]
        layers_v = [vd_raw[l] for l in range(w.L)]
        for l in range(w.L):  # warm
            moda.moda_depth_write(layers_k[l], kd, l, stream=stream)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for l in range(w.L):
            moda.moda_depth_write(layers_k[l], kd, l, stream=stream)
            moda.moda_depth_write(layers_v[l], vd, l, stream=stream)
        b.record(stream)
        torch.cuda.synchronize(dev)
        wms = a.elapsed_time(b)
        line["depth_write"] = {"ms_all_layers_kd_and_vd": wms, "launches": 2 * w.L,
                               "gbs": pack_bytes / (wms * 1e-3) / 1e9,
                               "pct_hbm": 100 * pack_bytes / (wms * 1e-3) / 1e9 / peaks["hbm_gbs"]}

    # ---- bounded depth cache: slot utilities (depth mass) and the slot choice ----
    if w.L:
        mass = torch.empty((w.Hk, w.L), dtype=torch.float32, device=dev)
        mws = torch.empty(((moda.moda_depth_mass_workspace_bytes(w.T, w.Hk, w.L) + 3) // 4,),
                          dtype=torch.float32, device=dev)
        slot_age = torch.arange(w.L, dtype=torch.int32, device=dev)  # a full cache, oldest in slot 0
        slot = torch.empty((1,), dtype=torch.int32, device=dev)
        moda.moda_fwd(q, k, v, kd, vd, w.scale, o=o, lse=lse, stream=stream)
        for _ in range(2):
            moda.moda_depth_mass(q, kd, lse, w.scale, mass=mass, workspace=mws, stream=stream)
        em = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(5)]
        torch.cuda.synchronize(dev)
        for a, b in em:  # q and kd (3.5 GB at the long workload) are far larger than L2
            a.record(stream)
            moda.moda_depth_mass(q, kd, lse, w.scale, mass=mass, workspace=mws, stream=stream)
            b.record(stream)
        torch.cuda.synchronize(dev)
        mms = statistics.median(a.elapsed_time(b) for a, b in em)
        mbytes = q.numel() * 2 + kd.numel() * 2 + lse.numel() * 4 + mass.numel() * 4
        ea = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(5)]
        for i, (a, b) in enumerate(ea):
            a.record(stream)
            moda.moda_depth_cache_admit(slot_age, mass, w.L // 2, w.L + i, slot=slot, stream=stream)
            b.record(stream)
        torch.cuda.synchronize(dev)
        ams = statistics.median(a.elapsed_time(b) for a, b in ea)
        line["depth_cache"] = {
            "depth_mass_ms": mms, "depth_mass_bytes": mbytes,
            "gbs": mbytes / (mms * 1e-3) / 1e9,
            "pct_hbm": 100 * mbytes / (mms * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "admit_us": 1e3 * ams, "slots": w.L, "recent": w.L // 2,
            "note": "moda_depth_mass: each slot's probability mass in the joint softmax, summed "
                    "over rows and KV heads (reads q, the packed kd and lse once); "
                    "moda_depth_cache_admit: the hybrid slot choice on a full cache"}
        del mass, mws, slot_age, slot

    # ---- decode: the last position as a new token over the whole cache ----
    if args.decode_steps > 0:
        t = w.T - 1
        qt = q[t].contiguous()
        kt = kd[:, t] if w.L else None  # packed stream read in place
        vt = vd[:, t] if w.L else None
        ws = torch.empty((moda.moda_decode_workspace_bytes(w.T, w.Hq, w.d) + 3) // 4,
                         dtype=torch.float32, device=dev)
        od = torch.empty((w.Hq, w.d), dtype=torch.bfloat16, device=dev)
        ld = torch.empty((w.Hq,), dtype=torch.float32, device=dev)
        # > L2; read (not written) before each call so L2 holds clean lines
        flush = torch.ones(64 << 20, dtype=torch.float32, device=dev)
        for _ in range(3):
            moda.moda_decode(qt, k, v, kt, vt, w.scale, o=od, lse=ld, workspace=ws, stream=stream)
        times = []
        for _ in range(args.decode_steps):
            sink = flush.sum()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            moda.moda_decode(qt, k, v, kt, vt, w.scale, o=od, lse=ld, workspace=ws, stream=stream)
            b.record(stream)
            torch.cuda.synchronize(dev)
            times.append(a.elapsed_time(b))
        dms = statistics.median(times)
        dbytes = 2 * w.T * w.Hk * w.d * 2 + 2 * w.Hk * w.L * w.d * 2 + 2 * w.Hq * w.d * 2 + \
            2 * ws.numel() * 4
        line["decode"] = {"us_per_token": 1e3 * dms, "context": w.T, "bytes": dbytes,
                          "gbs": dbytes / (dms * 1e-3) / 1e9,
                          "pct_hbm": 100 * dbytes / (dms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                          "l2": "flushed (256 MB read) before every call",
                          "launches_per_token": 2}
        del flush, ws

    # ---- backward (a separate measurement; not part of the forward step) ----
    if args.bwd_steps > 0:
        g = torch.Generator(device=dev)
        g.manual_seed(1)
        dO = torch.randn((w.T, w.Hq, w.d), generator=g, device=dev).to(torch.bfloat16)
        f32 = dict(dtype=torch.float32, device=dev)
        grads = (torch.empty((w.T, w.Hq, w.d), **f32), torch.empty((w.T, w.Hk, w.d), **f32),
                 torch.empty((w.T, w.Hk, w.d), **f32),
                 torch.empty((w.Hk, w.T, w.L, w.d), **f32) if w.L else None,
                 torch.empty((w.Hk, w.T, w.L, w.d), **f32) if w.L else None)
        delta = torch.empty((w.T, w.Hq), **f32)
        moda.moda_fwd(q, k, v, kd if w.L else None, vd if w.L else None, w.scale, o=o, lse=lse,
                      stream=stream)
        bargs = (q, k, v, kd if w.L else None, vd if w.L else None, o, lse, dO, w.scale)
        moda.moda_bwd(*bargs, grads=grads, delta=delta, stream=stream)
        eb = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.bwd_steps)]
        torch.cuda.synchronize(dev)
        for a, b in eb:
            a.record(stream)
            moda.moda_bwd(*bargs, grads=grads, delta=delta, stream=stream)
            b.record(stream)
        torch.cuda.synchronize(dev)
        bwd_ms = statistics.median(a.elapsed_time(b) for a, b in eb)
        Fb = 2.5 * F  # five GEMM-shaped products (S, dP, dV, dK, dQ) vs the forward's two
        line["bwd"] = {"ms": bwd_ms, "tflops": Fb / (bwd_ms * 1e-3) / 1e12,
                       "pct_peak_burst": 100 * Fb / (bwd_ms * 1e-3) / 1e12 / peak,
                       "flops_counted": Fb, "fwd_plus_bwd_ms": fwd_ms + bwd_ms,
                       "kernels": "delta + depth (CUDA cores) + dq + dk/dv (tcgen05)"}
        del grads, delta, dO

    # ---- an FFN layer's depth K/V: projection GEMM writing its slot (separate) ----
    if args.proj_steps > 0 and w.L:
        pw = wl.ProjWorkload(f"kv-proj-{w.name}", T=w.T, Dm=w.Hq * w.d, Hk=w.Hk, d=w.d, L=w.L,
                             slot=w.L - 1)
        g = torch.Generator(device=dev)
        g.manual_seed(2)
        xp = torch.randn((pw.T, pw.Dm), generator=g, device=dev).to(torch.bfloat16)
        wk = (torch.randn((pw.Hk * pw.d, pw.Dm), generator=g, device=dev) / pw.Dm ** 0.5).to(torch.bfloat16)
        wv = (torch.randn((pw.Hk * pw.d, pw.Dm), generator=g, device=dev) / pw.Dm ** 0.5).to(torch.bfloat16)
        for _ in range(2):
            moda.moda_kv_proj_write(xp, wk, wv, kd, vd, pw.slot, stream=stream)
        ep = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.proj_steps)]
        torch.cuda.synchronize(dev)
        for a, b in ep:
            a.record(stream)
            moda.moda_kv_proj_write(xp, wk, wv, kd, vd, pw.slot, stream=stream)
            b.record(stream)
        torch.cuda.synchronize(dev)
        pms = statistics.median(a.elapsed_time(b) for a, b in ep)
        # context: the same projection as two cuBLAS GEMMs plus two slot writes
        with torch.cuda.stream(stream):
            for _ in range(2):
                moda.moda_depth_write((xp @ wk.t()).view(pw.T, pw.Hk, pw.d), kd, pw.slot, stream=stream)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(args.proj_steps):
                moda.moda_depth_write((xp @ wk.t()).view(pw.T, pw.Hk, pw.d), kd, pw.slot, stream=stream)
                moda.moda_depth_write((xp @ wv.t()).view(pw.T, pw.Hk, pw.d), vd, pw.slot, stream=stream)
            b.record(stream)
        torch.cuda.synchronize(dev)
        ums = a.elapsed_time(b) / args.proj_steps
        Fp = pw.flops()
        line["kv_proj"] = {"ms": pms, "tflops": Fp / (pms * 1e-3) / 1e12,
                           "pct_peak_burst": 100 * Fp / (pms * 1e-3) / 1e12 / peak,
                           "shape": {"T": pw.T, "Dm": pw.Dm, "Hk": pw.Hk, "d": pw.d, "L": pw.L,
                                     "slot": pw.slot},
                           "flops_counted": Fp,
                           "unfused_cublas_gemm_plus_slot_write_ms": ums}
        del xp, wk, wv

    # ---- every other workload: forward, L = 0 forward, depth variant ----
    if args.config_steps > 0:
        cfgs = config_sweep(moda, dev, stream, peaks, args.config_steps, W)
        cfgs[w.name] = {"T": w.T, "Hq": w.Hq, "Hk": w.Hk, "G": w.G, "d": w.d, "L": w.L,
                        "fwd_ms": fwd_ms, "tflops": fwd_tflops,
                        "pct_peak_burst": 100 * fwd_tflops / peak,
                        "pct_nominal_peak": 100 * fwd_tflops / NOMINAL_BF16_TFLOPS,
                        "L0_ms": fwd0_ms, "overhead_vs_L0": fwd_ms / fwd0_ms - 1.0,
                        "extra_time_pages_convention": 1.0 - fwd0_ms / fwd_ms,
                        "note": "the headline workload: the fwd and fwd_L0 objects above"}
        line["configs"] = cfgs

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        if host is None:
            host = {n: t.cpu() for n, t in (("q", q), ("k", k), ("v", v), ("kd", kd_raw),
                                              ("vd", vd_raw))}
        f, s, rows, threads = oracle_sample(w, host, args.cpu_seconds)
        line["cpu_baseline"] = {
            "value": f / s / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{rows} (t, h) rows drawn uniformly from the {w.name} workload (seeded), "
                      f"{s:.1f} s on {threads} host threads"}

    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
