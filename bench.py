#!/usr/bin/env python3
"""Benchmark of the per-output-channel scaled FP8 linear layer on GB300.

One step = one call of the layer (one kernel launch) over one batch of
synthetic input already resident in HBM.  The headline workload is the
square prefill GEMM M = N = K = 4096 (seed 1); its throughput in TFLOP/s is
`value`.  Successive steps rotate through enough copies of the operands that
the working set is more than twice the L2 cache, so no step reads another
step's operands from L2.

Prints ONE JSON line on rank 0.  `--impl reference` times the CPU oracle on
the host cores instead (a bounded sample of the same workload per step).

Multi-GPU (torchrun): every rank runs its own copy of the workload
(independent problems, weak scaling, no collective on the data path); the
time is the maximum over ranks.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "FP8 GEMM TFLOP/s (GB/s at M=32) per config; fraction of GB300 roofline"
HEADLINE = "square"
FP8_OVER_BF16 = 2.0          # nominal dense fp8 / bf16 tensor rate (4.5 / 2.25 PFLOP/s)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
_CSRC = "fp8_channel_scaled_gb300/csrc/"
# the files each kernel is compiled from (its recorded DRAM traffic holds while they are unchanged)
TC2_SOURCES = [_CSRC + f for f in ("gemm_tc2.cu", "kernels.h", "ptx.cuh", "sched.cuh")]
TC_SOURCES = [_CSRC + f for f in ("gemm_tc.cu", "kernels.h", "ptx.cuh", "realign.cuh", "sched.cuh")]
DEC_SOURCES = [_CSRC + f for f in ("gemm_decode.cu", "kernels.h", "ptx.cuh", "realign.cuh")]


# ---------------------------------------------------------------- distributed plumbing
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(value: float, device=None) -> float:
    """Largest `value` across ranks (a host scalar; not on the data path)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------- peaks, clocks, traffic
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def sources_sha(paths) -> str:
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, paths):
    """DRAM bytes (read + write) per launch of the workload's GEMM kernel from
    the committed ncu record, if it was taken on the current kernel source;
    else None."""
    fn = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(fn) as f:
            entries = json.load(f)["entries"]
    except (OSError, ValueError, KeyError):
        return None
    sha = sources_sha(paths)
    for e in entries:
        if e.get("workload") == workload and e.get("sources_sha") == sha:
            return int(e["dram_read_bytes"]) + int(e["dram_write_bytes"])
    return None


class ClockSampler:
    """nvidia-smi sampled every 50 ms while the timed region runs."""

    FIELDS = ("timestamp,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = (uuid or "").lower().replace("gpu-", "")
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

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
        rows = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            if self.uuid and self.uuid not in parts[1].lower():
                continue
            rows.append((t, parts))
        if not rows:
            return None
        inside = [r for r in rows if self.t0 is not None and self.t0 - 0.06 <= r[0] <= self.t1 + 0.06]
        used = inside or rows
        mhz = [float(r[1][2]) for r in used if r[1][2].replace(".", "").isdigit()]
        max_mhz = [float(r[1][3]) for r in used if r[1][3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in used for n, v in zip(names, r[1][6:10]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(mhz) if mhz else None,
                "sm_max_mhz": max(max_mhz) if max_mhz else None,
                "reasons": reasons, "samples": len(used), "in_timed_region": bool(inside)}


# ---------------------------------------------------------------- workload on the device
def rotation_count(bytes_per_set: int, l2_bytes: int, cap: int = 64) -> int:
    """Copies of the operands so that the rotation covers more than 2x L2."""
    return max(2, min(cap, math.ceil(2 * l2_bytes / max(bytes_per_set, 1)) + 1))


def prepare(key: str, device, l2_bytes: int, rotate: bool = True):
    import torch
    import synth
    wl = synth.WORKLOADS[key]
    x, w, s = synth.workload_inputs(key)
    xd = torch.from_numpy(x).to(device)
    wd = torch.from_numpy(w).to(device)
    sd = torch.from_numpy(s).to(device)
    per_set = x.nbytes + w.nbytes + s.nbytes + 2 * wl.M * wl.N
    n = rotation_count(per_set, l2_bytes) if rotate else 1
    sets = []
    for i in range(n):
        sets.append((xd if i == 0 else xd.clone(), wd if i == 0 else wd.clone(),
                     sd if i == 0 else sd.clone(),
                     torch.empty((wl.M, wl.N), dtype=torch.bfloat16, device=device)))
    return wl, (x, w, s), sets, per_set


def time_steps(sets, steps: int, warmup: int, stream, call):
    """Warm up, then time `steps` calls back to back between two CUDA events on
    `stream`; returns the region in seconds.  No event sits between calls: an
    event record between two launches would stop the next kernel from
    starting its set-up while the previous one drains (programmatic
    dependent launch), so per-call times are region / steps."""
    import torch
    for i in range(warmup):
        call(*sets[i % len(sets)])
    torch.cuda.synchronize()
    region0 = torch.cuda.Event(enable_timing=True)
    region1 = torch.cuda.Event(enable_timing=True)
    region0.record(stream)
    for i in range(steps):
        call(*sets[i % len(sets)])
    region1.record(stream)
    torch.cuda.synchronize()
    return region0.elapsed_time(region1) / 1e3


def cpu_baseline(x, w, s, wl, target_s: float = 12.0, rows=None):
    """Time the oracle on a bounded sample of the workload's rows."""
    import numpy as np
    import oracle
    cores = oracle.default_threads()
    probe_rows = np.arange(min(wl.M, max(1, cores // 2)), dtype=np.int64)
    t0 = time.perf_counter()
    oracle.linear_rows(x, w, s, probe_rows)
    t_probe = time.perf_counter() - t0
    per_row = t_probe / probe_rows.size
    if rows is None:
        n = int(max(1, min(wl.M, target_s / max(per_row, 1e-9))))
        n = max(cores, (n // cores) * cores) if n >= cores else n
        n = min(n, wl.M)
        rows = np.linspace(0, wl.M - 1, n).round().astype(np.int64)
    t0 = time.perf_counter()
    y = oracle.linear_rows(x, w, s, rows)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows.size * wl.N * wl.K
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{rows.size} of {wl.M} rows (full N={wl.N}, K={wl.K}), {dt:.1f} s",
            "seconds": dt}, rows, y


def bench_workload(key, steps, warmup, device, l2_bytes, stream, fg, prepared_weight=False):
    """Time `steps` back-to-back calls of a workload.  prepared_weight: each
    set's w is first copied once (outside the timed region) to a 64-byte row
    pitch with fp8_gemm_prepare_weight, as a deployment that keeps its
    weights in that layout would."""
    import torch
    wl, host, sets, per_set = prepare(key, device, l2_bytes, rotate=(key != "small"))
    if prepared_weight:
        kp = (wl.K + 63) // 64 * 64
        prepped = []
        for x, w, s, y in sets:
            buf = torch.empty((wl.N, kp), dtype=torch.uint8, device=device)
            prepped.append((x, fg.fp8_gemm_prepare_weight(w, buf, stream), s, y))
        sets = prepped
        torch.cuda.synchronize(device)
    if prepared_weight:  # strided w views go through the options entry point
        call = lambda x, w, s, y: fg.fp8_gemm_scaled_ex(x, w, s, y, None, stream)  # noqa: E731
    else:
        call = lambda x, w, s, y: fg.fp8_gemm_scaled(x, w, s, y, stream)  # noqa: E731
    region = time_steps(sets, steps, warmup, stream, call)
    fg.check_device_error(stream)
    return wl, host, sets, region, per_set


def bench_grouped(device, l2_bytes, stream, fg, peak_tf_burst, steps=200, warmup=10):
    """Context timing of the grouped layer: 8 groups (experts) sharing 8192
    rows with a seeded skewed split, N = 2048, K = 4096 (the same FLOPs as the
    square workload); operand sets rotated past 2x L2."""
    import numpy as np
    import torch
    import synth
    G, M, N, K, seed = 8, 8192, 2048, 4096, 5
    rng = np.random.default_rng(seed)
    share = rng.dirichlet(np.full(G, 2.0))
    counts = np.floor(share * M).astype(np.int64)
    counts[-1] += M - counts.sum()
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x, _, _ = synth.make_inputs(M, 8, K, seed=seed)
    w = np.stack([synth.make_inputs(8, N, K, seed=seed + 1 + g)[1] for g in range(G)])
    s = (rng.uniform(0.5, 1.5, (G, N)) / np.sqrt(K)).astype(np.float32)
    per_set = x.nbytes + w.nbytes + 2 * M * N
    n = max(2, math.ceil(2 * l2_bytes / per_set) + 1)
    xd, wd, sd = (torch.from_numpy(a).to(device) for a in (x, w, s))
    od = torch.from_numpy(offs).to(device)
    sets = [(xd.clone(), wd.clone(), sd, torch.empty((M, N), dtype=torch.bfloat16, device=device))
            for _ in range(n)]
    call = lambda x_, w_, s_, y_: fg.fp8_gemm_grouped(x_, w_, s_, y_, od, None, stream)  # noqa: E731
    region = time_steps(sets, steps, warmup, stream, call)
    fg.check_device_error(stream)
    t = region / steps
    tf = 2.0 * M * N * K / t / 1e12
    return {"workload": f"grouped {G} groups, rows {counts.tolist()}, N={N}, K={K}",
            "us_per_call": round(t * 1e6, 2), "TFLOP/s": round(tf, 1),
            "frac_fp8_measured_burst": round(tf / peak_tf_burst, 4), "launches": 1,
            "l2": f"rotating {n} sets"}


# ---------------------------------------------------------------- arms
def run_ours(args):
    import torch
    world, rank, local = dist_env()
    device = torch.device("cuda", local if torch.cuda.device_count() > local else 0)
    torch.cuda.set_device(device)
    init_dist(world, "nccl")
    from fp8_channel_scaled_gb300 import build
    build.build()
    import fp8_channel_scaled_gb300 as fg

    props = torch.cuda.get_device_properties(device)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    stream = torch.cuda.current_stream(device)
    peaks, peak_src = load_peaks()

    # ---- headline workload, timed region with clock sampling
    sampler = ClockSampler(str(getattr(props, "uuid", "")) if rank == 0 else None)
    if rank == 0:
        sampler.start()
    key = args.workload
    wl, host, sets, per_set = prepare(key, device, l2, rotate=(key != "small"))
    call = lambda x, w, s, y: fg.fp8_gemm_scaled(x, w, s, y, stream)  # noqa: E731
    for i in range(args.warmup):
        call(*sets[i % len(sets)])
    torch.cuda.synchronize(device)
    barrier(device)
    torch.cuda.synchronize(device)
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.mark("t0")
    r0.record(stream)
    for i in range(args.steps):
        call(*sets[i % len(sets)])
    r1.record(stream)
    torch.cuda.synchronize(device)
    sampler.mark("t1")
    barrier(device)
    torch.cuda.synchronize(device)
    clocks = sampler.stop() if rank == 0 else None
    fg.check_device_error(stream)
    region = r0.elapsed_time(r1) / 1e3
    region_max = max_over_ranks(region, device)
    flops = float(wl.flops)
    # TFLOP/s, or GB/s of algorithmic bytes for the skinny (M <= 64) workloads
    hbm_metric = wl.M <= 64
    unit = "GB/s" if hbm_metric else "TFLOP/s"
    work = float(wl.algorithmic_bytes) / 1e9 if hbm_metric else flops / 1e12
    value = world * args.steps * work / region_max
    plan = fg.plan(wl.M, wl.N, wl.K, x=sets[0][0], w=sets[0][1])
    # average launch duration of the dominant kernel over the timed region
    # (the headline workload runs one kernel per call)
    kern = region / (args.steps * plan.launches)

    # ---- end to end through the public API from pinned host buffers.  Every
    # step copies its inputs (x, w, scale) host -> device and reads its result
    # y back device -> host; steps are pipelined over three streams (copy in,
    # compute, copy out) and two device buffer sets, so step i's copy-out,
    # step i+1's kernel and step i+2's copy-in can overlap on the full-duplex
    # host link.  Buffer reuse is ordered by events.
    x_h, w_h, s_h = host
    xp = torch.from_numpy(x_h).pin_memory()
    wp = torch.from_numpy(w_h).pin_memory()
    sp = torch.from_numpy(s_h).pin_memory()
    yps = [torch.empty((wl.M, wl.N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    bufs = [sets[0], sets[1] if len(sets) > 1 else tuple(t.clone() for t in sets[0])]
    s_in = torch.cuda.Stream(device)
    s_out = torch.cuda.Stream(device)
    e2e_steps = max(3, min(args.steps, 30))

    def e2e_run(n):
        in_done = [torch.cuda.Event() for _ in range(n)]
        comp_done = [torch.cuda.Event() for _ in range(n)]
        out_done = [torch.cuda.Event() for _ in range(n)]
        for i in range(n):
            xd, wd, sd, yd = bufs[i % 2]
            if i >= 2:
                s_in.wait_event(comp_done[i - 2])   # kernel i-2 has read this buffer set
            with torch.cuda.stream(s_in):
                xd.copy_(xp, non_blocking=True)
                wd.copy_(wp, non_blocking=True)
                sd.copy_(sp, non_blocking=True)
            in_done[i].record(s_in)
            stream.wait_event(in_done[i])
            if i >= 2:
                stream.wait_event(out_done[i - 2])  # y of step i-2 has been read back
            fg.fp8_gemm_scaled(xd, wd, sd, yd, stream)
            comp_done[i].record(stream)
            s_out.wait_event(comp_done[i])
            with torch.cuda.stream(s_out):
                yps[i % 2].copy_(yd, non_blocking=True)
            out_done[i].record(s_out)
        return out_done[-1]

    e2e_run(2)
    torch.cuda.synchronize(device)
    barrier(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    last = e2e_run(e2e_steps)
    s_out.wait_event(last)
    e1.record(s_out)
    torch.cuda.synchronize(device)
    fg.check_device_error(stream)
    e2e_t = max_over_ranks(e0.elapsed_time(e1) / 1e3, device)
    e2e = {"value": world * e2e_steps * work / e2e_t, "unit": unit,
           "h2d_bytes_per_step": int(x_h.nbytes + w_h.nbytes + s_h.nbytes),
           "d2h_bytes_per_step": int(2 * wl.M * wl.N), "steps": e2e_steps,
           "pipeline": "copy-in / compute / copy-out streams, two buffer sets"}

    # ---- roofline of the dominant (only) kernel.  The denominator is the
    # sustained bf16 figure (x2 for fp8) when the timed region is a long run
    # of back-to-back launches (power capping then sets the clock, as in the
    # sustained measurement), the burst figure for a short region.
    long_region = region_max >= 0.5
    peak_key = "bf16_tflops_sustained" if long_region else "bf16_tflops"
    peak_tf = peaks[peak_key] * FP8_OVER_BF16
    peak_tf_burst = peaks["bf16_tflops"] * FP8_OVER_BF16
    srcs = (DEC_SOURCES if plan.path == fg.PATH_DECODE
            else TC2_SOURCES if plan.cluster == 2 else TC_SOURCES)
    if hbm_metric:
        achieved = wl.algorithmic_bytes / kern / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                    "peak_source": f"{peak_src} copy bandwidth",
                    "frac_nominal_8000": round(achieved / 8000.0, 4)}
    else:
        achieved = flops / kern / 1e12
        kind = "sustained" if long_region else "burst"
        roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak_tf, 1),
                    "unit": "TFLOP/s", "frac": round(achieved / peak_tf, 4),
                    "peak_source": f"{peak_src} bf16 {kind} {peaks[peak_key]} x {FP8_OVER_BF16} "
                                   f"(fp8/bf16 nominal); timed region {region_max:.2f} s",
                    "frac_of_burst": round(achieved / peak_tf_burst, 4),
                    "frac_nominal_4500": round(achieved / 4500.0, 4)}
    roofline.update({"traffic": recorded_traffic(key, srcs),
                     "algorithmic_bytes": int(wl.algorithmic_bytes),
                     "kernel_us": round(kern * 1e6, 3)})

    line = {"metric": METRIC, "value": round(value, 2), "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(region_max / args.steps * 1e3, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate, bf16 out)",
            "data": "synthetic (seeded numpy PCG64 draws quantised to E4M3)",
            "config": {"workload": wl.name, "M": wl.M, "N": wl.N, "K": wl.K, "seed": wl.seed,
                       "path": "main" if plan.path == fg.PATH_MAIN else "decode",
                       "tile": f"{plan.tile_m}x{plan.tile_n}x128", "stages": plan.stages,
                       "grid": plan.grid, "parallelism": f"replicas x{world}",
                       "l2": f"rotating {len(sets)} operand sets ({len(sets) * per_set / 2**20:.0f} MiB > 2x L2 {l2 / 2**20:.0f} MiB), no flush kernel"},
            "roofline": roofline, "gpu_launches": args.steps * plan.launches, "e2e": e2e,
            "clocks": clocks}

    # ---- the other workloads (parity cases; reported for context)
    if rank == 0 and not args.headline_only:
        others = {}
        for key2 in [k for k in ("small", "square", "decode", "oddk", "oddk_prepared_w", "mlp")
                     if k != key]:
            base = key2.replace("_prepared_w", "")
            st = {"small": 2000, "square": 400, "decode": 400, "oddk": 400, "mlp": 60}[base]
            wl2, _, sets2, region2, per_set2 = bench_workload(
                base, st, 10, device, l2, stream, fg, prepared_weight=key2 != base)
            k2 = region2 / st
            tf = wl2.flops / k2 / 1e12
            gbs = wl2.algorithmic_bytes / k2 / 1e9
            roof_t = max(wl2.flops / 4.5e15, wl2.algorithmic_bytes / 8e12)
            p2 = fg.plan(wl2.M, wl2.N, wl2.K, x=sets2[0][0], w=sets2[0][1])
            srcs2 = (DEC_SOURCES if p2.path == fg.PATH_DECODE
                     else TC2_SOURCES if p2.cluster == 2 else TC_SOURCES)
            others[key2] = {"workload": wl2.name + (" (w prepared once to a 64-byte pitch; x repitched per call)" if key2 != base else ""),
                            "us_per_call": round(k2 * 1e6, 2),
                           "TFLOP/s": round(tf, 1), "GB/s": round(gbs, 1),
                           "frac_roofline_nominal": round(roof_t / k2, 4),
                           "frac_hbm_measured": round(gbs / peaks["hbm_gbs"], 4),
                           "frac_fp8_measured_burst": round(tf / peak_tf_burst, 4),
                           "path": "main" if p2.path == fg.PATH_MAIN else "decode",
                           "splits": p2.splits, "realign": p2.realign,
                           "launches": p2.launches,
                           "traffic": recorded_traffic(key2, srcs2) if key2 == base else None,
                           "l2": "no rotation (launch-bound)" if key2 == "small" else f"rotating {len(sets2)} sets"}
            del sets2
            torch.cuda.empty_cache()
        others["grouped_moe"] = bench_grouped(device, l2, stream, fg, peak_tf_burst)
        line["workloads"] = others

    # ---- CPU baseline (oracle on host cores, bounded sample) and a parity check of that sample
    if rank == 0 and not args.no_cpu_baseline:
        x_h, w_h, s_h = host
        cb, rows, yref = cpu_baseline(x_h, w_h, s_h, wl, target_s=args.cpu_seconds)
        if hbm_metric:
            cb["value"] = cb["value"] * 1e12 / wl.flops * wl.algorithmic_bytes / 1e9
            cb["unit"] = "GB/s"
        cb.pop("seconds")
        line["cpu_baseline"] = cb
        import numpy as np
        got = sets[0][3][torch.from_numpy(rows).to(device)].view(torch.int16).cpu().numpy().view(np.uint16)
        g = (got.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        r = (yref.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        bad = int(np.sum(np.abs(g - r) > 2.0 ** -7 * np.abs(r) + 1e-3))
        line["parity_sample"] = {"rows": int(rows.size), "elements": int(r.size), "outside_tolerance": bad}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args):
    """The oracle, as it stands, timed on the host cores; one bounded sample
    of the headline workload per step."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    import oracle
    import synth
    oracle.build()
    wl = synth.WORKLOADS[HEADLINE]
    x, w, s = synth.workload_inputs(HEADLINE)
    cores = oracle.default_threads()
    rng = np.random.default_rng(0)
    # time per output element, measured on a probe spread over all cores
    probe = 64 * cores
    t0 = time.perf_counter()
    oracle.linear_elems(x, w, s, rng.integers(0, wl.M, probe), rng.integers(0, wl.N, probe))
    per_elem = (time.perf_counter() - t0) / probe
    # each step is a bounded sample of output elements, sized so that the
    # whole --steps/--warmup run takes about 4x --cpu-seconds
    total = args.steps + args.warmup
    n = int(max(cores, min(wl.M * wl.N, args.cpu_seconds * 4 / max(total, 1) / max(per_elem, 1e-12))))
    samples = [(rng.integers(0, wl.M, n), rng.integers(0, wl.N, n)) for _ in range(min(total, 8))]
    for i in range(args.warmup):
        oracle.linear_elems(x, w, s, *samples[i % len(samples)])
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.linear_elems(x, w, s, *samples[i % len(samples)])
    dt = time.perf_counter() - t0
    flops = 2.0 * n * wl.K * args.steps
    value = flops / dt / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 (exact dot, one bf16 rounding)",
            "data": "synthetic (seeded numpy PCG64 draws quantised to E4M3)",
            "config": {"workload": wl.name, "M": wl.M, "N": wl.N, "K": wl.K, "seed": wl.seed,
                       "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": f"{n} random output elements of {wl.M}x{wl.N} per step (full K={wl.K})"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE,
                    choices=["small", "square", "decode", "oddk", "mlp"],
                    help="workload of the timed region (default: the square prefill GEMM)")
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the context timings of the other four workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="approximate CPU seconds spent in the oracle sample")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
