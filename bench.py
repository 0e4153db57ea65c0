#!/usr/bin/env python3
"""Benchmark of the out-of-place transpose on one GB300 (or N replicas).

Default workload: fp32 8192 x 8192 (256 MiB in, 256 MiB out), uniform[-1,1)
from seed 1, dense pitches.  A step is one whole transpose of that matrix
through the C ABI (``tr_transpose_ex`` with the AUTO variant).  Inputs and
outputs are larger than the 129 MB L2, so no flush is needed between steps.
A workload whose input or output fits in L2 (the 1024 x 1024 cases) is timed
with a 2x-L2 buffer written before every step and events around each transpose
alone; its hot-cache figure is reported beside it.

Prints ONE JSON line on rank 0:
  value     effective GB/s = (bytes read + bytes written) / device time, from
            CUDA events around exactly K back-to-back steps (max over ranks);
  roofline  the transpose kernel against the measured HBM copy peak;
  copy      tr_copy on the same byte count, timed the same way (the ceiling);
  e2e       the same metric with the host->device copy of the input (pinned)
            and the device->host copy of the output inside every step;
  cpu_baseline  the CPU oracle timed on a bounded sample of the workload.

``--impl reference`` times the CPU oracle instead (the only other place this
script runs it) and prints the same line with ``"impl": "reference"``.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from shared_memory_tiled_gb300 import workloads as W  # noqa: E402

METRIC = "transpose effective GB/s (read+write bytes/time) and % of GB300 HBM peak and of copy"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129e6


# --------------------------------------------------------------------------- utils

def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# Source files each kernel is built from (the hash of these decides whether a
# recorded ncu traffic figure still describes the kernel that runs).
KERNEL_SOURCES = {
    "k_tile_vec": ["tile_vec_kernel.cuh", "vec_common.cuh", "tile_geom.cuh", "tr_internal.h"],
    "k_tma": ["tile_tma.cu", "ptx.cuh", "tr_internal.h"],
    "k_tma_warp": ["tile_tma.cu", "ptx.cuh", "tr_internal.h"],
    "k_tma_ldst": ["tile_tma.cu", "ptx.cuh", "tr_internal.h"],
    "k_tma_ws": ["tile_tma.cu", "ptx.cuh", "tr_internal.h"],
    "k_tile_pad": ["tile_lsu.cu", "tile_geom.cuh", "tr_internal.h"],
    "k_naive": ["tile_lsu.cu", "tile_geom.cuh", "tr_internal.h"],
    "k_copy_aligned": ["copy.cu", "tr_internal.h"],
    "k_inplace": ["inplace.cu", "vec_common.cuh", "tile_geom.cuh", "tr_internal.h"],
}


def kernel_source_hash(kernel):
    """Hash of the sources a kernel is built from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "shared_memory_tiled_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, or None when there
    is none or the kernel's sources changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        rec = d.get(f"{kernel}:{workload}")
        if rec and kernel in KERNEL_SOURCES and rec.get("source_hash") == kernel_source_hash(kernel):
            return rec.get("dram_bytes_per_launch"), rec.get("note")
    except Exception:
        pass
    return None, None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            if not (t0 <= ts <= t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[4:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for _, _, flags in rows:
            for n, v in zip(names, flags[1:]):
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows)}


def nvsmi_id(local_rank):
    """The id nvidia-smi knows CUDA device ``local_rank`` by: its UUID when
    torch reports one and nvidia-smi accepts it, else the entry of
    CUDA_VISIBLE_DEVICES, else the ordinal (CUDA ordinals and nvidia-smi
    indices differ once CUDA_VISIBLE_DEVICES remaps the devices)."""
    candidates = []
    try:
        import torch
        u = str(torch.cuda.get_device_properties(local_rank).uuid)
        if u:
            candidates.append(u if u.startswith("GPU-") else "GPU-" + u)
    except Exception:
        pass
    vis = [v.strip() for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    if local_rank < len(vis):
        candidates.append(vis[local_rank])
    for c in candidates:
        try:
            r = subprocess.run(["nvidia-smi", f"--id={c}", "--query-gpu=index",
                                "--format=csv,noheader"], capture_output=True, text=True,
                               timeout=10)
            if r.returncode == 0 and r.stdout.strip():
                return c
        except Exception:
            break
    return str(local_rank)


def host_cpu_model():
    """The host CPU's model name, as lscpu or /proc/cpuinfo report it."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine() or "unknown"


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value, world):
    """Max of a float over all ranks (identity on one rank)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------- CPU oracle timing

def time_oracle(w, budget_s, max_reps=None, x=None):
    """Time the oracle on bands of rows of the workload until ``budget_s`` has
    passed.  Returns (GB/s, seconds, description, reps)."""
    import numpy as np
    import oracle
    if x is None:
        x = W.make_input(w)
    out = W.make_output(w)
    band = min(w.rows, 1024)
    band_bytes = 2 * w.esize * band * w.cols
    reps, t_total, r0 = 0, 0.0, 0
    while True:
        t = time.perf_counter()
        oracle.transpose(x[r0 * w.ld_in:], out[r0:], rows=min(band, w.rows - r0), cols=w.cols,
                         ld_in=w.ld_in, ld_out=w.ld_out)
        t_total += time.perf_counter() - t
        reps += 1
        r0 = (r0 + band) % w.rows
        done = reps >= max_reps if max_reps else t_total >= budget_s
        if done:
            break
    desc = (f"{reps} oracle transposes of {band}-row bands ({band}x{w.cols}, "
            f"{band_bytes / 1e6:.1f} MB read+written each) of the {w.name} matrix")
    return band_bytes * reps / t_total / 1e9, t_total, desc, reps


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    w = W.WORKLOADS[args.workload]
    x = W.make_input(w)
    for _ in range(args.warmup):
        time_oracle(w, 0.0, max_reps=1, x=x)
    gbs, secs, desc, reps = time_oracle(w, 0.0, max_reps=args.steps, x=x)
    line = {
        "metric": METRIC, "value": round(gbs, 3), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs * 1e3 / reps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u32" if w.esize == 4 else "u16", "data": "synthetic",
        "config": {"workload": w.name, "description": W.DESCRIPTION[w.name],
                   "step": "one 1024-row band of the matrix through the CPU oracle"},
        "impl": "reference",
        "cpu_baseline": {"value": round(gbs, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": desc, "host_cpus": os.cpu_count(),
                         "host_cpu_model": host_cpu_model()},
        "e2e": {"value": round(gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------ GPU arm

def run_ours(args):
    import numpy as np
    import torch

    from shared_memory_tiled_gb300 import binding as B

    rank, world, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    B.load()
    w = W.WORKLOADS[args.workload]
    dt = B.DType.F32 if w.esize == 4 else B.DType.BF16
    tdt = torch.int32 if w.esize == 4 else torch.int16
    ndt = np.int32 if w.esize == 4 else np.int16

    x_host = W.make_input(w)
    pin_in = torch.from_numpy(x_host.view(ndt)).pin_memory()
    pin_out = torch.empty(w.out_elems, dtype=tdt).pin_memory()
    d_in = torch.empty(w.in_elems, dtype=tdt, device=dev)
    d_out = torch.empty(w.out_elems, dtype=tdt, device=dev)
    d_in.copy_(pin_in)
    # Rewrite the uploaded input in place with an elementwise kernel (values
    # unchanged), so its pages were last written by SM stores, as data made by
    # an earlier kernel on the device would be.  Pages last written by the copy
    # engine were measured to read up to 4% slower under the transposed
    # access, by an amount that depended on what the GPU had run before.
    d_in.add_(0)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    variant = B.Variant[args.variant.upper()]
    targs = B.make_args(d_in.data_ptr(), d_out.data_ptr(), dt, w.batch, w.rows, w.cols, w.ld_in,
                        w.ld_out, w.sin, w.sout, sptr)
    topts = B.make_options(variant, pad=args.pad, stages=args.stages,
                           ctas_per_sm=args.ctas_per_sm, tile_order=args.tile_order,
                           out_stages=args.out_stages, tile_rows=args.tile_rows,
                           tile_cols=args.tile_cols, schedule=args.schedule,
                           threads=args.threads)
    planned = B.Variant(B.tr_plan_variant(targs, topts))
    lib = B.load()
    ex = lib.tr_transpose_ex
    import ctypes
    pa, po = ctypes.byref(targs), ctypes.byref(topts)
    inplace = args.op == "inplace"
    if inplace and (w.rows != w.cols or w.batch != 1):
        raise SystemExit("bench: the in-place transpose needs a square single-plane workload")
    ipf = lib.tr_transpose_inplace_f32 if w.esize == 4 else lib.tr_transpose_inplace_bf16

    runs = [0]  # transposes launched on d_in/d_out (the in-place parity check needs the count)

    def step():
        st = ipf(d_in.data_ptr(), 1, w.rows, w.ld_in, w.sin, sptr) if inplace else ex(pa, po)
        if st:
            B.check(st)
        runs[0] += 1

    copy_bytes = w.logical_elems * w.esize
    c_in = torch.empty(copy_bytes, dtype=torch.uint8, device=dev)
    c_out = torch.empty(copy_bytes, dtype=torch.uint8, device=dev)
    cfn = lib.tr_copy

    def copy_step():
        st = cfn(c_in.data_ptr(), c_out.data_ptr(), copy_bytes, sptr)
        if st:
            B.check(st)

    def timed(fn, k, warm):
        # One event before and one after the K back-to-back steps: an event
        # recorded between two launches holds the second one back until the
        # first has drained (about 3% of an 86 us step), so per-step times are
        # taken in a separate pass (step_times) and never enter the total.
        for _ in range(warm):
            fn()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(k):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        return e0.elapsed_time(e1)

    # A workload that fits in L2 would be timed hot by back-to-back steps: for
    # those, a buffer twice the L2 size is written before every step and the
    # events bracket the transpose alone.
    flush_l2 = min(w.in_elems, w.out_elems) * w.esize < L2_BYTES
    scratch = torch.empty(int(2 * L2_BYTES) // 4 + 1024, dtype=torch.int32, device=dev) if flush_l2 else None

    def timed_flushed(fn, k, warm):
        for _ in range(warm):
            scratch.zero_()
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(k)]
        barrier(world)
        torch.cuda.synchronize(dev)
        for a, b in evs:
            scratch.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        return sum(a.elapsed_time(b) for a, b in evs)

    def step_times(fn, k):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(k + 1)]
        torch.cuda.synchronize(dev)
        evs[0].record(stream)
        for i in range(k):
            fn()
            evs[i + 1].record(stream)
        torch.cuda.synchronize(dev)
        return [evs[i].elapsed_time(evs[i + 1]) for i in range(k)]

    sampler = ClockSampler(nvsmi_id(local_rank))
    sampler.start()
    # ---- the timed region: exactly K transposes
    t_wall0 = time.time()
    total_ms = (timed_flushed if flush_l2 else timed)(step, args.steps, args.warmup)
    t_wall1 = time.time()
    # keep the same kernel running for ~1 s more if the timed region was too
    # short for the 100 ms clock samples (the samples then cover this window)
    extra_window = None
    if t_wall1 - t_wall0 < args.clock_window:
        reps = max(1, int(args.clock_window / max(total_ms / args.steps / 1e3, 1e-6)))
        tw0 = time.time()
        timed(step, reps, 0)
        extra_window = (tw0, time.time())
    sampler.stop()
    clocks = sampler.summary(*(extra_window or (t_wall0, t_wall1)))
    if extra_window:
        clocks["window"] = (f"timed region shorter than the 100 ms sampling: same kernel "
                            f"re-run untimed for {args.clock_window:g} s right after it")

    # per-launch statistics from a separate pass with an event after every step
    per_ms = step_times(step, args.steps)
    # the median of repeated runs: more passes of K back-to-back steps, each
    # between two events like the timed region (not part of `value`)
    rep_ms = [max_over_ranks((timed_flushed if flush_l2 else timed)(step, args.steps, 0), world)
              for _ in range(args.repeats)]
    hot_ms = max_over_ranks(timed(step, args.steps, args.warmup), world) if flush_l2 else None
    total_ms = max_over_ranks(total_ms, world)
    ms_step = total_ms / args.steps
    gbs = w.algorithmic_bytes * args.steps * world / (total_ms / 1e3) / 1e9
    med_ms = statistics.median(per_ms)
    # the timed region launches nothing but this kernel, K times
    kernel_gbs = w.algorithmic_bytes / (ms_step / 1e3) / 1e9

    # ---- parity guard on the timed output: sampled positions vs the definition
    rng = np.random.default_rng(123)
    n = 4096
    bb = rng.integers(0, w.batch, n)
    ii = rng.integers(0, w.rows, n)
    jj = rng.integers(0, w.cols, n)
    src = x_host[bb * w.sin + ii * w.ld_in + jj]
    if inplace:
        # every step transposes the buffer in place: an even number of steps
        # (warm-up, timed and clock-window runs together) restores the input
        got = d_in.cpu().numpy().view(x_host.dtype)
        dst = got[ii * w.ld_in + jj] if runs[0] % 2 == 0 else got[jj * w.ld_in + ii]
    else:
        got = d_out.cpu().numpy().view(x_host.dtype)
        dst = got[bb * w.sout + jj * w.ld_out + ii]
    if not np.array_equal(src, dst):
        raise SystemExit("bench: the timed output differs from the input at sampled positions")

    # ---- copy ceiling on the same bytes
    c_in.random_(0, 255)
    c_total = (timed_flushed if flush_l2 else timed)(copy_step, args.steps, args.warmup)
    c_total = max_over_ranks(c_total, world)
    copy_gbs = 2 * copy_bytes * args.steps / (c_total / 1e3) / 1e9
    # context: torch's own device copy of the same bytes, timed the same way
    tc_total = (timed_flushed if flush_l2 else timed)(lambda: c_out.copy_(c_in), args.steps,
                                                      args.warmup)
    tc_total = max_over_ranks(tc_total, world)
    torch_copy_gbs = 2 * copy_bytes * args.steps / (tc_total / 1e3) / 1e9

    # ---- end to end: pinned host input -> device -> transpose -> pinned host output.
    # Steps rotate over `e2e_streams` streams, each with its own device and
    # pinned output buffers, so the device->host copy of one step overlaps the
    # host->device copy of the next (the link carries both directions at once);
    # within a step the three operations stay ordered on its stream.
    k_e2e = max(3, min(args.steps, 20))
    ns = max(2, args.e2e_streams)
    streams = [torch.cuda.Stream(dev) for _ in range(ns)]
    pins_out = [pin_out] + [torch.empty_like(pin_out).pin_memory() for _ in range(ns - 1)]
    bufs = [(d_in, d_in if inplace else d_out)]
    for _ in range(ns - 1):
        di = torch.empty_like(d_in)
        bufs.append((di, di if inplace else torch.empty_like(d_out)))
    e_args = []
    for i, st in enumerate(streams):
        di, do = bufs[i]
        a = B.make_args(di.data_ptr(), do.data_ptr(), dt, w.batch, w.rows, w.cols, w.ld_in,
                        w.ld_out, w.sin, w.sout, st.cuda_stream)
        e_args.append((a, ctypes.byref(a)))

    def e2e_step_on(i):
        st = streams[i]
        di, do = bufs[i]
        with torch.cuda.stream(st):
            di.copy_(pin_in, non_blocking=True)
            if inplace:
                rc = ipf(di.data_ptr(), 1, w.rows, w.ld_in, w.sin, st.cuda_stream)
            else:
                rc = ex(e_args[i][1], po)
            if rc:
                B.check(rc)
            pins_out[i].copy_(do, non_blocking=True)

    def e2e_run(k):
        for j in range(k):
            e2e_step_on(j % ns)

    e2e_run(ns)  # warm-up
    torch.cuda.synchronize(dev)
    barrier(world)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(streams[0])
    for st in streams[1:]:
        st.wait_event(t0)
    e2e_run(k_e2e)
    for st in streams[1:]:
        done = torch.cuda.Event()
        done.record(st)
        streams[0].wait_event(done)
    t1.record(streams[0])
    torch.cuda.synchronize(dev)
    barrier(world)
    e_total = max_over_ranks(t0.elapsed_time(t1), world)
    e2e_gbs = w.algorithmic_bytes * k_e2e * world / (e_total / 1e3) / 1e9
    # every end-to-end step uploads the input and transposes it once
    e2e_got = pins_out[(k_e2e - 1) % ns].numpy().view(x_host.dtype)
    e2e_dst = (e2e_got[jj * w.ld_in + ii] if inplace
               else e2e_got[bb * w.sout + jj * w.ld_out + ii])
    if not np.array_equal(e2e_dst, src):
        raise SystemExit("bench: end-to-end output differs from the transposed input")

    peak, peak_kind = read_peaks()
    kname = {B.Variant.TMA: {1: "k_tma", 3: "k_tma_ldst", 4: "k_tma_ws"}.get(args.schedule, "k_tma_warp"),
             B.Variant.TILE_VEC: "k_tile_vec", B.Variant.TILE_PAD: "k_tile_pad",
             B.Variant.NAIVE_ROW: "k_naive", B.Variant.NAIVE_COL: "k_naive"}.get(planned, "?")
    if inplace:
        kname = "k_inplace"
    traffic, traffic_note = recorded_traffic(kname, w.name)

    line = {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u32" if w.esize == 4 else "u16", "data": "synthetic",
        "config": {"workload": w.name + ("_inplace" if inplace else ""),
                   "description": W.DESCRIPTION[w.name] + (", transposed in place" if inplace else ""),
                   "bytes_per_step": w.algorithmic_bytes,
                   "input_placement": ("uploaded from pinned host memory, then rewritten in "
                                       "place by an elementwise device kernel (values unchanged)"),
                   "variant": "INPLACE" if inplace else planned.name,
                   "l2": ("flushed: a 2x-L2 buffer is written before every step; events around "
                          "each transpose (and each copy) alone" if flush_l2 else
                          "no flush: input and output each larger than the 129 MB L2"),
                   "parallelism": f"replicas x{world}"},
        "pct_of_hbm_measured": round(100 * gbs / world / peak, 2),
        "pct_of_hbm_nominal": round(100 * gbs / world / NOMINAL_HBM_GBS, 2),
        "pct_of_copy": round(100 * gbs / (copy_gbs * world), 2),
        "repeats": {"n": len(rep_ms), "unit": "GB/s",
                    "median": round(w.algorithmic_bytes * args.steps / (statistics.median(rep_ms) / 1e3) / 1e9, 2) if rep_ms else None,
                    "min": round(w.algorithmic_bytes * args.steps / (max(rep_ms) / 1e3) / 1e9, 2) if rep_ms else None,
                    "max": round(w.algorithmic_bytes * args.steps / (min(rep_ms) / 1e3) / 1e9, 2) if rep_ms else None,
                    "pass": "further passes of K back-to-back steps between two events (not in value)"},
        "step_ms": {"median": round(med_ms, 5), "min": round(min(per_ms), 5),
                    "p90": round(sorted(per_ms)[int(0.9 * (len(per_ms) - 1))], 5),
                    "pass": "separate pass of K steps with an event after each (not in value)"},
        "copy": {"value": round(copy_gbs, 2), "unit": "GB/s", "bytes_per_step": 2 * copy_bytes,
                 "kernel": "tr_copy", "torch_copy_GBps": round(torch_copy_gbs, 2)},
        "roofline": {"bound": "hbm", "achieved": round(kernel_gbs, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(kernel_gbs / peak, 4),
                     "traffic": traffic, "peak_source": peak_kind, "kernel": kname,
                     "bytes_per_launch": w.algorithmic_bytes},
        "e2e": {"value": round(e2e_gbs, 2), "unit": "GB/s", "steps": k_e2e,
                "overlap": (f"{ns} streams: one step's device->host copy runs with the next one's "
                            "host->device copy"),
                "h2d_bytes_per_step": w.in_elems * w.esize,
                "d2h_bytes_per_step": w.out_elems * w.esize},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if traffic_note:
        line["roofline"]["traffic_note"] = traffic_note
    if flush_l2:
        line["hot"] = {"value": round(w.algorithmic_bytes * args.steps * world / (hot_ms / 1e3) / 1e9, 2),
                       "unit": "GB/s", "ms_per_step": round(hot_ms / args.steps, 5),
                       "note": "K back-to-back steps between two events, data resident in L2"}
        line["roofline"]["note"] = "input and output fit in L2: not an HBM roofline figure"
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cgbs, csecs, desc, _ = time_oracle(w, args.cpu_seconds, x=x_host)
        line["cpu_baseline"] = {"value": round(cgbs, 3), "unit": "GB/s", "cores": 1,
                                "kind": "oracle", "sample": desc,
                                "seconds": round(csecs, 2), "host_cpus": os.cpu_count(),
                                "host_cpu_model": host_cpu_model()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(W.WORKLOADS), default="c2")
    ap.add_argument("--op", choices=["transpose", "inplace"], default="transpose",
                    help="out-of-place transpose (default) or in-place square transpose")
    ap.add_argument("--variant", default="auto",
                    choices=["auto", "naive_row", "naive_col", "tile_pad", "tile_vec", "tma"])
    ap.add_argument("--pad", type=int, default=1)
    ap.add_argument("--stages", type=int, default=0)
    ap.add_argument("--ctas-per-sm", dest="ctas_per_sm", type=int, default=0)
    ap.add_argument("--tile-order", dest="tile_order", type=int, default=0)
    ap.add_argument("--out-stages", dest="out_stages", type=int, default=0)
    ap.add_argument("--tile-rows", dest="tile_rows", type=int, default=0)
    ap.add_argument("--tile-cols", dest="tile_cols", type=int, default=0)
    ap.add_argument("--threads", type=int, default=0, help="vector tile threads per block")
    ap.add_argument("--schedule", type=int, default=0,
                    help="vector tile: 1 = one tile per block, 2 = persistent with prefetch")
    ap.add_argument("--cpu-seconds", dest="cpu_seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", dest="no_cpu_baseline", action="store_true")
    ap.add_argument("--repeats", type=int, default=5,
                    help="extra passes of K steps whose median is reported beside the value")
    ap.add_argument("--e2e-streams", dest="e2e_streams", type=int, default=3,
                    help="streams (and buffer sets) the end-to-end steps rotate over")
    ap.add_argument("--clock-window", dest="clock_window", type=float, default=1.0,
                    help="seconds of untimed re-runs for clock sampling when the timed "
                         "region is shorter than this (0 = none)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # never fewer than 3 untimed warm-up steps
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
