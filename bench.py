"""Benchmark of batched quintic Newton–Schulz on one GB300.

    python bench.py [--steps K] [--warmup W] [--workload NAME] [--batch B]
                    [--impl ours|reference] [--no-per-shape] [--no-cpu-baseline]

A "step" is one whole NS call (norm, then 5 x Gram / polynomial / update)
over the workload's stack, inputs resident in HBM.  The default workload is
the 128-expert MoE stack 128 x 1536 x 2048 (bf16), one of the two shapes the
method is held to 60% of dense bf16 peak on; every other workload is timed
under "per_shape" (median, min and max of 20 calls each).  One JSON line.

This build is a single-GPU library: its short-contraction products load a
shared operand panel with TMA multicast inside a cluster of two CTAs, whose
tensor maps cover only the calling GPU's own buffers, and no data-path step
exchanges anything between GPUs.  `--impl ours` therefore refuses --gpus > 1
or WORLD_SIZE > 1 with a one-line error and exit status 2.

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (one matrix per step, scaled to a whole call).
"""
from __future__ import annotations

import argparse
import dataclasses
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import ns_inputs  # noqa: E402

METRIC = "ms per NS call and dense-equiv TFLOP/s (% of GB300 bf16 peak), per shape"
DEFAULT_WORKLOAD = "experts_128x1536x2048"
L2_BYTES = 129 * 1024 * 1024
PAGES_H200_QUACK_MS = {  # prime-rl PR #3873, Results, "NS microbenchmark on one H200" (context only)
    "square_4096": 2.71, "square_8192": 17.0, "wide_4096x14336": 7.07,
    "experts_128x1536x2048": 25.0, "stack_128x2048x768": 8.6, "stack_32x7168x2048": 33.0,
}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash():
    csrc = os.path.join(ROOT, "newton_schulz_07_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` on `workload` from a committed ncu
    summary, and a note saying where the figure comes from; (None, why) when it
    is absent or was taken on different kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None, "no committed ncu traffic summary"
    if rec.get("source_hash") != kernel_source_hash():
        return None, "kernel sources changed since the committed ncu traffic capture"
    ent = rec.get("kernels", {}).get(workload, {}).get(kernel)
    if ent is None:
        return None, f"no committed ncu traffic figure for {kernel} on {workload}"
    note = f"ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch on {ent['measured_on']}"
    if ent.get("scale", 1) != 1:
        note += f", scaled by {ent['scale']:g} (matrices are independent units of a launch)"
    if "algorithmic_bytes_per_launch" in ent:
        note += f"; algorithmic bytes per launch {ent['algorithmic_bytes_per_launch']:.4g}"
    return float(ent["dram_bytes_per_launch"]), note


def flop_counts(w, steps=5):
    """Per-launch useful FLOPs of each tensor-core kernel and the dense-
    equivalent total of one call."""
    m, n, b = float(w.m), float(w.n), float(w.batch)
    return {
        "gram": b * m * (m + 1) * n,
        "poly": b * m * m * (m + 1),
        "update": b * 2 * m * m * n,
        "norm_bytes": b * 2.0 * w.rows * w.cols,
        "dense_call": w.dense_flops(steps),
        "useful_call": w.useful_flops(steps),
    }


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    FIELDS = ["timestamp", "index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        """Stops sampling and keeps the samples as (time.time() seconds, fields)."""
        self.rows = []
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                ts = None
            self.rows.append((ts, parts))

    def summary(self, window):
        """Clock summary of the samples taken inside `window` = (t0, t1) in
        time.time() seconds (all samples if none falls inside)."""
        rows = getattr(self, "rows", [])
        inside = [r for r in rows if r[0] is not None and window[0] <= r[0] <= window[1]]
        used = inside if inside else rows
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, parts in used:
            try:
                sm.append(float(parts[2]))
                mx.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[6:]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(used), "window": "timed region" if inside else "whole sampling period"}


def gpu_id_for(torch, dev):
    try:
        p = torch.cuda.get_device_properties(dev)
        return f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
    except Exception:
        return str(dev)


# ------------------------------------------------------------- CPU oracle --

def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0]), "blas threadpool"
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var]), var
    return len(os.sched_getaffinity(0)), "affinity (BLAS default: all cores)"


def oracle_one(w, k):
    import oracle
    g = ns_inputs.bf16_bits_to_f64(ns_inputs.matrix_bits(w, k))
    t0 = time.perf_counter()
    oracle.newton_schulz(g)
    return time.perf_counter() - t0


def cpu_baseline(w, budget_s=12.0):
    """The oracle as it stands on a bounded sample of the workload: whole
    matrices, as many as fit in about `budget_s` seconds, scaled to a call."""
    times = [oracle_one(w, 0)]
    k = 1
    while sum(times) < budget_s and k < w.batch:
        times.append(oracle_one(w, k))
        k += 1
    per_matrix = sum(times) / len(times)
    cores, src = cpu_threads()
    return {"value": per_matrix * w.batch * 1e3, "unit": "ms", "cores": cores, "cores_source": src,
            "kind": "oracle",
            "sample": f"{len(times)} of {w.batch} matrices ({w.rows}x{w.cols}) of {w.name}, fp64 numpy oracle, "
                      f"{sum(times):.1f} s, scaled by {w.batch}/{len(times)}"}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    w = ns_inputs.WORKLOADS[args.workload]
    for i in range(args.warmup):
        oracle_one(w, i % w.batch)
    times = []
    t_all = time.perf_counter()
    for i in range(args.steps):
        times.append(oracle_one(w, (args.warmup + i) % w.batch) * w.batch)
    wall = time.perf_counter() - t_all
    ms = 1e3 * sum(times) / len(times)
    cores, src = cpu_threads()
    fl = flop_counts(w)
    line = {
        "impl": "reference", "metric": METRIC, "value": ms, "unit": "ms", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "rows": w.rows, "cols": w.cols, "ns_steps": 5,
                   "parallelism": "host cores"},
        "tflops_dense_equiv": fl["dense_call"] / (ms * 1e-3) / 1e12,
        "cpu_baseline": {"value": ms, "unit": "ms", "cores": cores, "cores_source": src, "kind": "oracle",
                         "sample": f"each step: 1 of {w.batch} matrices ({w.rows}x{w.cols}) through the fp64 "
                                   f"numpy oracle, scaled by {w.batch}; {args.steps} steps in {wall:.1f} s"},
        "e2e": {"value": ms, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------- GPU --

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(ns_inputs.WORKLOADS))
    ap.add_argument("--batch", type=int, default=0,
                    help="run the workload's shape with this many matrices (small profiling captures)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-per-shape", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if world > 1 or args.gpus > 1:
        print(f"bench.py: --impl ours runs on one GPU only (got --gpus {args.gpus}, WORLD_SIZE {world}): "
              "the library's multicast tensor maps cover the calling GPU's own buffers and the path has "
              "no multi-GPU step", file=sys.stderr, flush=True)
        return 2

    import torch

    import newton_schulz_07_gb300 as ns

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    peaks, peak_src = load_peaks()
    w = ns_inputs.WORKLOADS[args.workload]
    if args.batch > 0:
        w = dataclasses.replace(w, name=f"{w.name.split('_')[0]}_{args.batch}x{w.rows}x{w.cols}", batch=args.batch)
    fl = flop_counts(w)

    bits = ns_inputs.stack_bits(w)
    host_in = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    G = host_in.to(dev)
    out = torch.empty_like(G)
    ws = ns.alloc_workspace(w.batch, w.rows, w.cols, device=dev)
    working_set = 2 * G.numel() * 2 + ws.numel()
    flush = working_set < 4 * L2_BYTES
    scrub = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev) if flush else None
    stream = torch.cuda.current_stream(dev)

    def call():
        ns.muon_ns(G, out=out, workspace=ws)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()

    sampler = ClockSampler(gpu_id_for(torch, dev))
    sampler.start()
    time.sleep(0.3)
    # Per-kernel breakdown, before the long timed loop (so that it runs in the
    # clock state of a kernel timed alone, which the burst peak describes; the
    # clock record decides): the same kernels in the same launch configuration
    # and storage form (A and B half-stored, MUON_NS_HALF) as muon_ns_ws,
    # through the per-step entry points, with CUDA events on the launching
    # stream between launches.  Step 1 reads G and applies the per-matrix
    # scale in its epilogues, as the whole call does.
    nb = min(args.steps, 20)
    names = ["norm", "gram", "poly", "update"]
    acc = {k: 0.0 for k in names}
    a_buf = torch.empty((w.batch, w.m, w.m), dtype=torch.bfloat16, device=dev)
    b_buf = torch.empty_like(a_buf)
    x_bufs = [torch.empty_like(G), torch.empty_like(G)]
    err_word = torch.zeros(1, dtype=torch.int32, device=dev)
    d_buf = torch.empty((w.batch, w.m), dtype=torch.float32, device=dev)
    n_off, n_bytes = ns.workspace_region(w.batch, w.rows, w.cols, 2)
    norms_t = ws[n_off:n_off + n_bytes].view(torch.float32)
    a, b, c = ns.DEFAULT_COEFFS
    t_bd0 = time.time()
    bd_wall0 = time.perf_counter()
    for it in range(nb + 2):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(17)]
        ev[0].record(stream)
        ns.muon_ns_normalize(G, ws, norms_only=True)
        ev[1].record(stream)
        src, cur = G, 0
        for s in range(5):
            ns.muon_ns_gram(src, A=a_buf, device_error=err_word, norms=norms_t if s == 0 else None, half=True)
            ev[2 + 3 * s].record(stream)
            ns.muon_ns_poly(a_buf, b, c, B=b_buf, diag=d_buf, device_error=err_word, half=True)
            ev[3 + 3 * s].record(stream)
            ns.muon_ns_update(src, b_buf, a, Xn=x_bufs[cur], diag=d_buf, device_error=err_word,
                              norms=norms_t if s == 0 else None, half=True)
            ev[4 + 3 * s].record(stream)
            src, cur = x_bufs[cur], 1 - cur
        torch.cuda.synchronize()
        if it < 2:
            continue
        acc["norm"] += ev[0].elapsed_time(ev[1])
        for s in range(5):
            acc["gram"] += ev[1 + 3 * s].elapsed_time(ev[2 + 3 * s]) / 5
            acc["poly"] += ev[2 + 3 * s].elapsed_time(ev[3 + 3 * s]) / 5
            acc["update"] += ev[3 + 3 * s].elapsed_time(ev[4 + 3 * s]) / 5
    bd_wall = time.perf_counter() - bd_wall0
    t_bd1 = time.time()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    t_region0 = time.time()
    for i in range(args.steps):
        if scrub is not None:
            scrub.fill_(i & 0xFF)
        starts[i].record(stream)
        call()
        ends[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    t_region1 = time.time()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = sum(step_ms) / args.steps
    dev_err = ns.read_error(ws)

    sampler.stop()
    clocks = sampler.summary((t_region0, t_region1))
    bd_clocks = sampler.summary((t_bd0, t_bd1))
    per_launch_ms = {k: v / nb for k, v in acc.items()}
    share = {"norm": per_launch_ms["norm"]}
    for k in ("gram", "poly", "update"):
        share[k] = 5 * per_launch_ms[k]
    dominant = max(("gram", "poly", "update"), key=lambda k: share[k])
    achieved = fl[dominant] / (per_launch_ms[dominant] * 1e-3) / 1e12
    # Peak for the roofline: the burst figure when the breakdown loop is short
    # (under a second) or its sampled SM clock stays within 5 % of the maximum;
    # the sustained (power-capped) figure otherwise.
    near_max = bd_clocks is not None and bd_clocks["sm_mhz"] >= 0.95 * bd_clocks["sm_max_mhz"]
    use_burst = bd_wall < 1.0 or near_max
    peak = peaks["bf16_tflops"] if use_burst else peaks["bf16_tflops_sustained"]
    why = (f"breakdown loop {bd_wall:.2f} s" + (" (< 1 s)" if bd_wall < 1.0 else "") +
           (f", median SM clock {bd_clocks['sm_mhz']:.0f} of {bd_clocks['sm_max_mhz']:.0f} MHz"
            if bd_clocks else ", no clock samples"))
    traffic, traffic_note = recorded_traffic(dominant, w.name)
    roofline = {"bound": "tensor", "kernel": f"ns_tc_gemm ({dominant})", "achieved": achieved,
                "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "frac_of_burst_peak": achieved / peaks["bf16_tflops"],
                "frac_of_sustained_peak": achieved / peaks["bf16_tflops_sustained"],
                "peak_source": f"{peak_src} bf16 {'burst' if use_burst else 'sustained'} ({why})",
                "traffic": traffic, "traffic_note": traffic_note,
                "algorithmic_flops_per_launch": fl[dominant],
                "avg_launch_ms": per_launch_ms[dominant]}
    norm_gbs = fl["norm_bytes"] / (per_launch_ms["norm"] * 1e-3) / 1e9
    breakdown = {
        "storage": "A and B half-stored, as muon_ns_ws keeps them (per-step entry points with MUON_NS_HALF)",
        "per_launch_ms": per_launch_ms,
        "per_call_ms": share,
        "norm_hbm": {"achieved_gbs": norm_gbs, "peak_gbs": peaks["hbm_gbs"],
                     "frac": norm_gbs / peaks["hbm_gbs"], "bytes_per_call": fl["norm_bytes"]},
        "tensor_tflops_useful": {k: fl[k] / (per_launch_ms[k] * 1e-3) / 1e12 for k in ("gram", "poly", "update")},
        "frac_of_peak_useful": {k: fl[k] / (per_launch_ms[k] * 1e-3) / 1e12 / peak for k in ("gram", "poly", "update")},
        "clocks": bd_clocks,
        "wall_s": bd_wall,
    }
    del a_buf, b_buf, x_bufs, d_buf

    # End to end through the C ABI with host buffers (muon_ns_host): every step
    # uploads the pinned host stack, orthogonalises it and downloads the
    # result, chunk by chunk with the copies overlapping the compute.
    host_out = torch.empty_like(host_in).pin_memory()
    hws = torch.empty(ns.host_workspace_size(*host_in.shape), dtype=torch.uint8, device=dev)
    # Twenty calls back to back (each one's copies inside its own events), at
    # least as many as the timed steps: the value is the median call, so one
    # slow call on a shared host does not move it; the spread is recorded.
    ne = max(min(args.steps, 100), 20)
    ns.muon_ns_host(host_in, out=host_out, workspace=hws, device=dev)
    torch.cuda.synchronize()
    e2e_same = bool(torch.equal(host_out, out.cpu()))  # the device-resident call's result, bit for bit
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(ne + 1)]
    evs[0].record(stream)
    for i in range(ne):
        ns.muon_ns_host(host_in, out=host_out, workspace=hws, device=dev, sync=False)
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    e2e_calls = [evs[i].elapsed_time(evs[i + 1]) for i in range(ne)]
    e2e_ms = statistics.median(e2e_calls)
    io_bytes = host_in.numel() * 2
    del hws
    # The machine's host link, for reading e2e: one upload and one download of the
    # whole stack between the same pinned buffers and device tensors, each
    # alone, with CUDA events on the current stream.
    link = {}
    for name, dst, src in (("h2d", G, host_in), ("d2h", host_out, out)):
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        c0.record(stream)
        dst.copy_(src, non_blocking=True)
        c1.record(stream)
        torch.cuda.synchronize()
        link[name + "_gbs"] = io_bytes / (c0.elapsed_time(c1) * 1e-3) / 1e9
    link["copy_floor_ms"] = io_bytes / (min(link["h2d_gbs"], link["d2h_gbs"]) * 1e9) * 1e3

    # Spot parity of the timed call's output (untimed; matrix 0 vs the oracle).
    import oracle
    got = ns_inputs.bf16_bits_to_f64(host_out[0].view(torch.int16).numpy().view(np.uint16))
    ref = oracle.newton_schulz(ns_inputs.bf16_bits_to_f64(bits[0]))
    parity = {"matrix": 0, "rel_fro_err_vs_fp64_oracle": float(np.linalg.norm(got - ref) / np.linalg.norm(ref)),
              "tolerance": 1.5e-2}

    per_shape = None
    if not args.no_per_shape:
        per_shape = {}
        for name, ow in ns_inputs.WORKLOADS.items():
            if name == w.name:
                continue
            per_shape[name] = time_workload(torch, ns, ow, dev, peaks)
        per_shape[w.name + "_fp32_mode"] = time_f32(torch, ns, w, dev, peaks)
        per_shape["muon_step_" + w.name.split("_", 1)[1]] = time_muon_step(torch, ns, w, dev, peaks)
        step_mix = ["experts_16x1536x2048", "stack_128x2048x768", "tiny_4x256x512"]
        per_shape["muon_step_grouped_" + "+".join(n.split("_", 1)[1] for n in step_mix)] = time_muon_step_grouped(
            torch, ns, [ns_inputs.WORKLOADS[n] for n in step_mix], dev, peaks)
        for names in (["stack_32x7168x2048", "stack_128x2048x768"],
                      ["experts_16x1536x2048", "stack_128x2048x768", "tiny_4x256x512"]):
            per_shape["grouped_" + "+".join(n.split("_", 1)[1] for n in names)] = time_grouped(
                torch, ns, [ns_inputs.WORKLOADS[n] for n in names], dev, peaks)

    cpu = None if args.no_cpu_baseline else cpu_baseline(w)

    tf_dense = fl["dense_call"] / (ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": ms, "unit": "ms", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": ms / PAGES_H200_QUACK_MS[w.name] if w.name in PAGES_H200_QUACK_MS else None,
        "vs_baseline_note": "ms ratio to the pages' H200 QuACK figure for this shape (another GPU; context)",
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "rows": w.rows, "cols": w.cols, "ns_steps": 5,
                   "coeffs": list(ns.DEFAULT_COEFFS), "eps": ns.DEFAULT_EPS,
                   "distribution": w.dist, "parallelism": "single GPU",
                   "l2": ("flushed between timed steps (256 MiB write)" if flush else
                          f"working set {working_set / 2**30:.1f} GiB >> L2, no flush")},
        "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms), "max": max(step_ms)},
        "tflops_dense_equiv": tf_dense,
        "tflops_useful": fl["useful_call"] / (ms * 1e-3) / 1e12,
        "pct_dense_bf16_peak": 100.0 * tf_dense / peaks["bf16_tflops"],
        "pct_dense_bf16_peak_sustained": 100.0 * tf_dense / peaks["bf16_tflops_sustained"],
        "peak_source": peak_src,
        "gpu_launches": args.steps * ns.launches_per_call(5),
        "launches_per_step": ns.launches_per_call(5),
        "wall_s_timed": wall,
        "device_error_word": dev_err,
        "roofline": roofline,
        "breakdown": breakdown,
        "clocks": clocks,
        "e2e": {"value": e2e_ms, "unit": "ms", "h2d_bytes_per_step": io_bytes, "d2h_bytes_per_step": io_bytes,
                "steps": ne, "stat": "median of back-to-back calls",
                "ms_min": min(e2e_calls), "ms_max": max(e2e_calls), "ms_mean": statistics.fmean(e2e_calls),
                "api": "newton_schulz_07_gb300.muon_ns_host -> muon_ns_host (C ABI, pinned host buffers)",
                "largest_chunk_matrices": ns.host_chunk(*host_in.shape), "equals_device_result": e2e_same,
                "host_link": link},
        "parity": parity,
        "cpu_baseline": cpu,
        "per_shape": per_shape,
        "kernel_source_hash": kernel_source_hash(),
    }
    print(json.dumps(line), flush=True)
    return 0


def time_calls(torch, fns, stream, calls=20, warmup=3, scrub=None):
    """Times each function of `fns` (a dict name -> callable), one call of each
    per round, `calls` rounds, with CUDA events on `stream` around each call and
    L2 flushed before it.  Returns name -> {median, min, max, mean, calls} in ms."""
    for fn in fns.values():
        for _ in range(warmup):
            fn()
    torch.cuda.synchronize()
    ms = {k: [] for k in fns}
    for i in range(calls):
        for k, fn in fns.items():
            if scrub is not None:
                scrub.fill_(i & 0xFF)
            s = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            s.record(stream)
            fn()
            e.record(stream)
            torch.cuda.synchronize()
            ms[k].append(s.elapsed_time(e))
    return {k: {"median": statistics.median(v), "min": min(v), "max": max(v), "mean": sum(v) / len(v),
                "calls": len(v)} for k, v in ms.items()}


def rates(w_dense, w_useful, ms, peaks):
    tf = w_dense / (ms * 1e-3) / 1e12
    return {"tflops_dense_equiv": tf, "tflops_useful": w_useful / (ms * 1e-3) / 1e12,
            "pct_dense_bf16_peak": 100 * tf / peaks["bf16_tflops"]}


def time_workload(torch, ns, w, dev, peaks, calls=20, warmup=3):
    """Whole muon_ns_ws calls on workload w: median, min and max of `calls`."""
    bits = ns_inputs.stack_bits(w)
    G = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)
    out = torch.empty_like(G)
    ws = ns.alloc_workspace(w.batch, w.rows, w.cols, device=dev)
    scrub = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    t = time_calls(torch, {"call": lambda: ns.muon_ns(G, out=out, workspace=ws)},
                   torch.cuda.current_stream(dev), calls, warmup, scrub)["call"]
    res = {"ms": t["median"], "ms_min": t["min"], "ms_max": t["max"], "ms_mean": t["mean"], "calls": t["calls"],
           **rates(w.dense_flops(), w.useful_flops(), t["median"], peaks),
           "batch": w.batch, "rows": w.rows, "cols": w.cols, "l2": "flushed before each timed call",
           "device_error_word": ns.read_error(ws)}
    if w.name in PAGES_H200_QUACK_MS:
        res["pages_h200_quack_ms"] = PAGES_H200_QUACK_MS[w.name]
    del G, out, ws, scrub
    torch.cuda.empty_cache()
    return res


def time_f32(torch, ns, w, dev, peaks, calls=20, warmup=3):
    """The fp32 NS mode (tf32 tensor cores, fp32 storage) on workload w, with
    matrix 0's error against the fp64 oracle."""
    x = np.stack([ns_inputs.matrix_f32(w, k) for k in range(w.batch)])
    G = torch.from_numpy(x).to(dev)
    out = torch.empty_like(G)
    ws = torch.empty(ns.f32_workspace_size(w.batch, w.rows, w.cols), dtype=torch.uint8, device=dev)
    t = time_calls(torch, {"call": lambda: ns.muon_ns_f32(G, out=out, workspace=ws)},
                   torch.cuda.current_stream(dev), calls, warmup)["call"]
    import oracle
    ref = oracle.newton_schulz(x[0].astype(np.float64))
    err = float(np.linalg.norm(out[0].double().cpu().numpy() - ref) / np.linalg.norm(ref))
    tf = w.dense_flops() / (t["median"] * 1e-3) / 1e12
    res = {"ms": t["median"], "ms_min": t["min"], "ms_max": t["max"], "calls": t["calls"],
           "tflops_dense_equiv": tf, "pct_dense_bf16_peak": 100 * tf / peaks["bf16_tflops"],
           "mode": "fp32 in/out, tf32 tensor cores", "rel_fro_err_matrix0_vs_fp64_oracle": err,
           "l2": f"working set >> L2 ({w.name})", "device_error_word": ns.read_error(ws)}
    del G, out, ws
    torch.cuda.empty_cache()
    return res


def time_grouped(torch, ns, wls, dev, peaks, calls=20, warmup=3):
    """One muon_ns_grouped call over several stacks (one optimizer step's NS
    over parameter groups of different shapes) against the same stacks as
    back-to-back muon_ns_ws calls, interleaved call by call."""
    Gs = [torch.from_numpy(ns_inputs.stack_bits(w).view(np.int16)).view(torch.bfloat16).to(dev) for w in wls]
    outs = [torch.empty_like(G) for G in Gs]
    ws = torch.empty(ns.grouped_workspace_size(Gs), dtype=torch.uint8, device=dev)
    scrub = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    sws = [ns.alloc_workspace(*G.shape, device=dev) for G in Gs]

    def grouped():
        ns.muon_ns_grouped(Gs, outs=outs, workspace=ws)

    def separate():
        for G, o, wsi in zip(Gs, outs, sws):
            ns.muon_ns(G, out=o, workspace=wsi)

    t = time_calls(torch, {"separate": separate, "grouped": grouped}, torch.cuda.current_stream(dev),
                   calls, warmup, scrub)
    g, sp = t["grouped"], t["separate"]
    res = {"ms": g["median"], "ms_min": g["min"], "ms_max": g["max"], "calls": g["calls"],
           **rates(sum(w.dense_flops() for w in wls), sum(w.useful_flops() for w in wls), g["median"], peaks),
           "stacks": [w.name for w in wls], "api": "muon_ns_grouped (one call)",
           "separate_calls_ms": sp["median"], "separate_calls_ms_min": sp["min"], "separate_calls_ms_max": sp["max"],
           "grouped_over_separate": g["median"] / sp["median"],
           "l2": "flushed before each timed call", "device_error_word": ns.read_error(ws)}
    if all(w.name in PAGES_H200_QUACK_MS for w in wls):
        res["pages_h200_quack_ms_sum"] = sum(PAGES_H200_QUACK_MS[w.name] for w in wls)
    del Gs, outs, ws, sws, scrub
    torch.cuda.empty_cache()
    return res


def time_muon_step(torch, ns, w, dev, peaks, calls=20, warmup=3):
    """The Muon step around NS on workload w's shape: fp32 masters W, momentum
    M and gradient G (G from the workload's distribution), one fused
    muon_step_ws call against the chain muon_momentum -> muon_ns_ws ->
    muon_apply, interleaved call by call; plus the momentum kernel alone
    (HBM-bound) and matrix 0 against the fp64 oracle step."""
    lr, mu, wd = 0.02, 0.95, 0.01
    G = torch.from_numpy(np.stack([ns_inputs.matrix_f32(w, k) for k in range(w.batch)])).to(dev)
    gen = torch.Generator(device=dev).manual_seed(1234)
    W = torch.randn(G.shape, generator=gen, device=dev) * 0.02
    M = torch.randn(G.shape, generator=gen, device=dev) * 0.02
    W0, M0 = W[0].cpu().numpy(), M[0].cpu().numpy()
    sws = torch.empty(ns.step_workspace_size(w.batch, w.rows, w.cols), dtype=torch.uint8, device=dev)
    ws1, ws2 = ns.alloc_workspace(w.batch, w.rows, w.cols, device=dev), ns.alloc_workspace(w.batch, w.rows, w.cols, device=dev)
    U = torch.empty(G.shape, dtype=torch.bfloat16, device=dev)
    O = torch.empty_like(U)
    # Parity of one fused step on matrix 0 (untimed, before W and M move on).
    ns.muon_step(W, M, G, lr, momentum=mu, weight_decay=wd, workspace=sws)
    torch.cuda.synchronize()
    import oracle
    W_ref, M_ref, O_ref = oracle.muon_step(W0, M0, G[0].cpu().numpy(), lr, mu, weight_decay=wd)
    upd = lr * ns.default_scale(w.rows, w.cols) * np.linalg.norm(O_ref)
    parity = {"matrix": 0, "w_update_rel_err_vs_fp64_oracle": float(np.linalg.norm(W[0].cpu().numpy() - W_ref) / upd),
              "m_max_abs_err": float(np.max(np.abs(M[0].cpu().numpy() - M_ref))), "tolerance": 1.5e-2}

    def fused():
        ns.muon_step(W, M, G, lr, momentum=mu, weight_decay=wd, workspace=sws)

    def chain():
        ns.muon_momentum(M, G, ws1, momentum=mu, U=U)
        ns.muon_ns(U, out=O, workspace=ws2)
        ns.muon_apply(W, O, lr, weight_decay=wd)

    def momentum_only():
        ns.muon_momentum(M, G, ws1, momentum=mu, U=U)

    stream = torch.cuda.current_stream(dev)
    t = time_calls(torch, {"fused": fused, "chain": chain, "momentum": momentum_only}, stream, calls, warmup)
    f, c, mo = t["fused"], t["chain"], t["momentum"]
    mom_bytes = w.batch * w.rows * w.cols * (4 + 4 + 4 + 2)  # read G, M; write M, U
    res = {"ms": f["median"], "ms_min": f["min"], "ms_max": f["max"], "calls": f["calls"],
           **rates(w.dense_flops(), w.useful_flops(), f["median"], peaks),
           "api": "muon_step_ws (one call: momentum + norm, NS, update fused into the last product)",
           "launches": ns.step_launches(5),
           "chain_ms": c["median"], "chain_ms_min": c["min"],
           "chain_api": "muon_momentum -> muon_ns_ws -> muon_apply (separate passes)",
           "fused_over_chain": f["median"] / c["median"],
           "momentum_kernel": {"ms": mo["median"], "bytes": mom_bytes,
                               "gbs": mom_bytes / (mo["median"] * 1e-3) / 1e9,
                               "frac_of_hbm_peak": mom_bytes / (mo["median"] * 1e-3) / 1e9 / peaks["hbm_gbs"]},
           "hparams": {"lr": lr, "momentum": mu, "nesterov": True, "weight_decay": wd,
                       "scale": ns.default_scale(w.rows, w.cols)},
           "parity": parity, "device_error_word": ns.read_error(sws),
           "l2": "working set >> L2"}
    del G, W, M, sws, ws1, ws2, U, O
    torch.cuda.empty_cache()
    return res


def time_muon_step_grouped(torch, ns, wls, dev, peaks, calls=20, warmup=3):
    """One Muon step over several parameter groups (fp32 W, M, G per stack) as
    one muon_step_grouped call, against one muon_step_ws call per group,
    interleaved call by call."""
    gen = torch.Generator(device=dev).manual_seed(4321)
    groups = []
    for i, w in enumerate(wls):
        G = torch.from_numpy(np.stack([ns_inputs.matrix_f32(w, k) for k in range(w.batch)])).to(dev)
        groups.append(dict(W=torch.randn(G.shape, generator=gen, device=dev) * 0.02,
                           M=torch.randn(G.shape, generator=gen, device=dev) * 0.02, G=G,
                           lr=0.02 / (i + 1), momentum=0.95, weight_decay=0.01))
    gws = torch.empty(ns.step_grouped_workspace_size(groups), dtype=torch.uint8, device=dev)
    sws = [torch.empty(ns.step_workspace_size(*g["W"].shape), dtype=torch.uint8, device=dev) for g in groups]

    def grouped():
        ns.muon_step_grouped(groups, workspace=gws)

    def separate():
        for g, w in zip(groups, sws):
            ns.muon_step(g["W"], g["M"], g["G"], g["lr"], momentum=g["momentum"], weight_decay=g["weight_decay"],
                         workspace=w)

    t = time_calls(torch, {"separate": separate, "grouped": grouped}, torch.cuda.current_stream(dev), calls, warmup)
    g, sp = t["grouped"], t["separate"]
    res = {"ms": g["median"], "ms_min": g["min"], "ms_max": g["max"], "calls": g["calls"],
           "stacks": [w.name for w in wls], "api": "muon_step_grouped (one call)",
           "separate_calls_ms": sp["median"], "separate_calls_ms_min": sp["min"],
           "grouped_over_separate": g["median"] / sp["median"], "device_error_word": ns.read_error(gws)}
    del groups, gws, sws
    torch.cuda.empty_cache()
    return res


if __name__ == "__main__":
    sys.exit(main())
