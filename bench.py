#!/usr/bin/env python3
"""Benchmark of the out-of-place transpose on one GB300 (or N replicas).

Default workload: fp32 8192 x 8192 (256 MiB in, 256 MiB out), uniform[-1,1)
from seed 1, dense pitches.  A step is one whole transpose of that matrix
through the C ABI (``tr_transpose_ex`` with the AUTO variant).  Inputs and
outputs are larger than the 129 MB L2, so no flush is needed between steps.
A workload whose input or output fits in L2 (the 1024 x 1024 cases) is timed
with a 2x-L2 buffer written before every step and events around each transpose
alone; its hot-cache figure is reported beside it.

Timing: after W untimed warm-up steps, R >= 5 passes of exactly K steps, each
pass between a barrier and a device synchronize, timed by two CUDA events on
the launching stream around its K back-to-back steps; the reported figure is
the median pass ("Shared memory and the bank conflict", "What to record": the
median of repeated runs after a warm-up, every variant next to the copy).

Prints ONE JSON line on rank 0:
  value       effective GB/s = (bytes read + bytes written) / device time of
              the median pass (max over ranks per pass);
  roofline    the transpose kernel against the measured HBM copy peak;
  copy        tr_copy on the same byte count, timed the same way (the ceiling);
  per_config  (default run) every configuration -- c1 index-valued and
              uniform, c2, c3, c4, c5 -- then the misaligned-pitch cases
              and c2 / c5 transposed in place, measured the same way, each
              with its own copy ceiling, roofline fraction and clock record;
  e2e         the same metric with the host->device copy of the input (pinned)
              and the device->host copy of the output inside every step, next
              to what the host link moves on its own;
  cpu_baseline / cpu_baseline_all_cores
              the CPU oracle on one core and on every host core, timed on a
              bounded sample of the workload.

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
    "k_tile_vec": ["tile_vec_kernel.cuh", "vec_common.cuh", "tile_geom.cuh", "tr_internal.h",
                   "bounds.cuh"],
    "k_tma": ["tile_tma.cu", "ptx.cuh", "tr_internal.h", "bounds.cuh"],
    "k_tma_warp": ["tile_tma.cu", "ptx.cuh", "tr_internal.h", "bounds.cuh"],
    "k_tma_ldst": ["tile_tma.cu", "ptx.cuh", "tr_internal.h", "bounds.cuh"],
    "k_tma_ws": ["tile_tma.cu", "ptx.cuh", "tr_internal.h", "bounds.cuh"],
    "k_tile_pad": ["tile_lsu.cu", "tile_geom.cuh", "tr_internal.h", "bounds.cuh"],
    "k_naive": ["tile_lsu.cu", "tile_geom.cuh", "tr_internal.h", "bounds.cuh"],
    "k_copy_aligned": ["copy.cu", "tr_internal.h", "bounds.cuh"],
    "k_inplace": ["inplace.cu", "vec_common.cuh", "tile_geom.cuh", "tr_internal.h",
                  "bounds.cuh", "ptx.cuh"],
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

def host_cores():
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def time_oracle(w, budget_s, max_reps=None, x=None):
    """Time the oracle on bands of rows of the workload until ``budget_s`` has
    passed.  Returns (GB/s, seconds, description, reps)."""
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


def time_oracle_all_cores(w, budget_s, x=None, threads=None):
    """The same oracle, unchanged, on every host core at once: the first plane's
    rows are split into one band per thread and each thread transposes its band
    (the oracle's C loop runs without the interpreter lock), whole plane after
    whole plane, until ``budget_s`` has passed.  Returns (GB/s, seconds,
    description, threads)."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    if x is None:
        x = W.make_input(w)
    out = W.make_output(w)
    n = threads or host_cores()
    step = -(-w.rows // n)
    bands = [(r0, min(step, w.rows - r0)) for r0 in range(0, w.rows, step)]

    def one(band):
        r0, nr = band
        oracle.transpose(x[r0 * w.ld_in:], out[r0:], rows=nr, cols=w.cols, ld_in=w.ld_in,
                         ld_out=w.ld_out)

    plane_bytes = 2 * w.esize * w.rows * w.cols
    planes = 0
    with ThreadPoolExecutor(max_workers=len(bands)) as pool:
        t0 = time.perf_counter()
        while True:
            list(pool.map(one, bands))
            planes += 1
            secs = time.perf_counter() - t0
            if secs >= budget_s:
                break
    desc = (f"{planes} oracle transposes of the whole {w.rows}x{w.cols} plane of the {w.name} "
            f"workload, its rows split into {len(bands)} bands of up to {step} rows, one per "
            f"thread ({plane_bytes / 1e6:.1f} MB read+written per plane)")
    return plane_bytes * planes / secs / 1e9, secs, desc, len(bands)


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

# The configurations measured side by side in the default run (``per_config``),
# then the misaligned-pitch cases and the in-place transpose of the square ones.
PER_CONFIG = ("c1_index", "c1_uniform", "c2", "c3", "c4", "c5")
PER_CONFIG_EXTRA = ("c3_back", "c5_oddin", "c5_oddout", "c5_oddboth", "c2_oddout")
PER_CONFIG_INPLACE = ("c2", "c5")


def gbps(nbytes, ms):
    return nbytes / (ms / 1e3) / 1e9


# Device cycles of sleep queued before a timed pass, per step: about 25 us of
# host time to issue one launch through the binding, at the 2 GHz SM clock.
LAUNCH_QUEUE_CYCLES = 50_000


class Gpu:
    """Device, stream, library handle and timing helpers of one rank."""

    def __init__(self, args):
        import torch

        from shared_memory_tiled_gb300 import binding as B
        self.args = args
        self.rank, self.world, self.local_rank = dist_env()
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group("nccl")
        torch.cuda.set_device(self.local_rank)
        self.dev = torch.device("cuda", self.local_rank)
        self.B = B
        self.lib = B.load()
        self.stream = torch.cuda.current_stream(self.dev)
        self.sptr = self.stream.cuda_stream
        self.sampler = ClockSampler(nvsmi_id(self.local_rank))
        self._scratch = None

    def scratch(self):
        """A buffer twice the L2 size, written before each step of an L2-resident workload."""
        import torch
        if self._scratch is None:
            self._scratch = torch.empty(int(2 * L2_BYTES) // 4 + 1024, dtype=torch.int32,
                                        device=self.dev)
        return self._scratch

    def passes(self, fn, k, warm, n, flush):
        """``n`` passes of exactly ``k`` steps after ``warm`` untimed ones; each
        pass is bracketed by a barrier and a device synchronize on both sides.
        Without ``flush``: one CUDA event before and one after the k
        back-to-back steps (an event between two launches would hold the
        second back until the first has drained); a bounded device-side
        sleep queued before the first event keeps the GPU busy while the
        host queues the k launches, so the pass times the device running
        them back to back rather than the host issuing the first one.  With ``flush``: the 2x-L2
        buffer is written before every step and events bracket each step
        alone.  Returns the milliseconds of each pass, max over ranks."""
        import torch
        for _ in range(warm):
            if flush:
                self.scratch().zero_()
            fn()
        out = []
        for _ in range(n):
            barrier(self.world)
            torch.cuda.synchronize(self.dev)
            if flush:
                evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(k)]
                for a, b in evs:
                    self.scratch().zero_()
                    a.record(self.stream)
                    fn()
                    b.record(self.stream)
                torch.cuda.synchronize(self.dev)
                ms = sum(a.elapsed_time(b) for a, b in evs)
            else:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                torch.cuda._sleep(LAUNCH_QUEUE_CYCLES * k)  # not timed: precedes e0
                e0.record(self.stream)
                for _ in range(k):
                    fn()
                e1.record(self.stream)
                torch.cuda.synchronize(self.dev)
                ms = e0.elapsed_time(e1)
            barrier(self.world)
            out.append(max_over_ranks(ms, self.world))
        return out

    def step_times(self, fn, k):
        import torch
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(k + 1)]
        torch.cuda.synchronize(self.dev)
        evs[0].record(self.stream)
        for i in range(k):
            fn()
            evs[i + 1].record(self.stream)
        torch.cuda.synchronize(self.dev)
        return [evs[i].elapsed_time(evs[i + 1]) for i in range(k)]

    def clock_window(self, fn, ms_per_step, t0, t1):
        """The wall-clock window whose nvidia-smi samples describe ``fn``: the
        timed passes themselves when they lasted at least ``--clock-window``
        seconds, else an untimed re-run of the same steps for that long right
        after them.  Returns (clocks summary, re-run note or None)."""
        import torch
        if t1 - t0 >= self.args.clock_window or self.args.clock_window <= 0:
            return self.sampler.summary(t0, t1), None
        reps = max(1, int(self.args.clock_window / max(ms_per_step / 1e3, 1e-6)))
        torch.cuda.synchronize(self.dev)
        w0 = time.time()
        for _ in range(reps):
            fn()
        torch.cuda.synchronize(self.dev)
        clocks = self.sampler.summary(w0, time.time())
        return clocks, (f"timed passes shorter than the 100 ms sampling: same kernel re-run "
                        f"untimed for {self.args.clock_window:g} s right after them")


class Measured:
    """One workload's buffers and its measured figures."""


def measure(gpu, w, opts, inplace=False):
    """Time one workload: the transpose (median of passes), its parity at
    sampled positions, and ``tr_copy`` on the same byte count timed the same
    way.  Returns a ``Measured`` holding the buffers and the figures."""
    import ctypes

    import numpy as np
    import torch
    B, args = gpu.B, gpu.args
    m = Measured()
    m.w, m.k, m.world = w, args.steps, gpu.world
    dt = B.DType.F32 if w.esize == 4 else B.DType.BF16
    m.tdt = torch.int32 if w.esize == 4 else torch.int16
    ndt = np.int32 if w.esize == 4 else np.int16
    m.dt = dt
    m.x_host = W.make_input(w)
    m.pin_in = torch.from_numpy(m.x_host.view(ndt)).pin_memory()
    m.d_in = torch.empty(w.in_elems, dtype=m.tdt, device=gpu.dev)
    # in place there is no output buffer (and no out-of-place plan)
    m.d_out = None if inplace else torch.empty(w.out_elems, dtype=m.tdt, device=gpu.dev)
    m.d_in.copy_(m.pin_in)
    # Rewrite the uploaded input in place with an elementwise kernel (values
    # unchanged), so its pages were last written by SM stores, as data made by
    # an earlier kernel on the device would be.  Pages last written by the copy
    # engine were measured to read up to 4% slower under the transposed
    # access, by an amount that depended on what the GPU had run before.
    m.d_in.add_(0)
    m.topts = opts
    m.plan = m.planned = m.targs = None
    if not inplace:
        m.targs = B.make_args(m.d_in.data_ptr(), m.d_out.data_ptr(), dt, w.batch, w.rows, w.cols,
                              w.ld_in, w.ld_out, w.sin, w.sout, gpu.sptr)
        plan = B.Plan()
        B.check(B.tr_plan_ex(m.targs, opts, plan))
        m.plan = plan
        m.planned = B.Variant(plan.variant)
    ex = gpu.lib.tr_transpose_ex
    pa = ctypes.byref(m.targs) if m.targs is not None else None
    po = ctypes.byref(opts)
    m.po = po
    ipf = gpu.lib.tr_transpose_inplace_f32 if w.esize == 4 else gpu.lib.tr_transpose_inplace_bf16
    m.ipf = ipf
    m.inplace = inplace
    m.runs = 0

    def step():
        st = ipf(m.d_in.data_ptr(), 1, w.rows, w.ld_in, w.sin, gpu.sptr) if inplace else ex(pa, po)
        if st:
            B.check(st)
        m.runs += 1

    m.step = step
    k, warm, npass = args.steps, args.warmup, args.passes
    m.flush = min(w.in_elems, w.out_elems) * w.esize < L2_BYTES
    t0 = time.time()
    m.pass_ms = gpu.passes(step, k, warm, npass, m.flush)
    t1 = time.time()
    m.med_ms = statistics.median(m.pass_ms)
    m.ms_step = m.med_ms / k
    m.value = gbps(w.algorithmic_bytes * k * gpu.world, m.med_ms)
    m.clocks, m.clock_note = gpu.clock_window(step, m.ms_step, t0, t1)
    m.hot_ms = (statistics.median(gpu.passes(step, k, warm, npass, False)) if m.flush else None)

    # parity guard on the timed output: sampled positions against the definition
    rng = np.random.default_rng(123)
    n = 4096
    m.bb = rng.integers(0, w.batch, n)
    m.ii = rng.integers(0, w.rows, n)
    m.jj = rng.integers(0, w.cols, n)
    m.src = m.x_host[m.bb * w.sin + m.ii * w.ld_in + m.jj]
    if inplace:
        # every step transposes the buffer in place: an even number of steps
        # (warm-up, timed and clock-window runs together) restores the input
        got = m.d_in.cpu().numpy().view(m.x_host.dtype)
        dst = got[m.ii * w.ld_in + m.jj] if m.runs % 2 == 0 else got[m.jj * w.ld_in + m.ii]
    else:
        got = m.d_out.cpu().numpy().view(m.x_host.dtype)
        dst = got[m.bb * w.sout + m.jj * w.ld_out + m.ii]
    if not np.array_equal(m.src, dst):
        raise SystemExit(f"bench: the timed output of {w.name} differs from the input at "
                         "sampled positions")

    # copy ceiling on the same bytes, timed the same way
    m.copy_bytes = w.logical_elems * w.esize
    m.c_in = torch.empty(m.copy_bytes, dtype=torch.uint8, device=gpu.dev)
    m.c_out = torch.empty(m.copy_bytes, dtype=torch.uint8, device=gpu.dev)
    m.c_in.random_(0, 255)
    cfn = gpu.lib.tr_copy

    def copy_step():
        st = cfn(m.c_in.data_ptr(), m.c_out.data_ptr(), m.copy_bytes, gpu.sptr)
        if st:
            B.check(st)

    m.copy_step = copy_step
    m.copy_pass_ms = gpu.passes(copy_step, k, warm, npass, m.flush)
    m.copy_value = gbps(2 * m.copy_bytes * k * gpu.world, statistics.median(m.copy_pass_ms))
    return m


def config_entry(m, peak, inplace=False):
    """The per-configuration summary of one measured workload."""
    w = m.w
    e = {
        "workload": w.name + ("_inplace" if inplace else ""),
        "description": W.DESCRIPTION[w.name] + (", transposed in place" if inplace else ""),
        "bytes_per_step": w.algorithmic_bytes,
        "variant": "INPLACE" if inplace else m.planned.name,
        "value": round(m.value, 2), "unit": "GB/s", "statistic": "median of passes",
        "ms_per_step": round(m.ms_step, 5),
        "passes_GBps": [round(m.value * m.med_ms / p, 2) for p in m.pass_ms],
        "pct_of_hbm_measured": round(100 * m.value / m.world / peak, 2),
        "pct_of_hbm_nominal": round(100 * m.value / m.world / NOMINAL_HBM_GBS, 2),
        "copy_GBps": round(m.copy_value, 2),
        "pct_of_copy": round(100 * m.value / m.copy_value, 2),
        "roofline_frac": None if m.flush else round(m.value / m.world / peak, 4),
        "l2": "flushed before every step" if m.flush else "no flush (input and output > L2)",
        "clocks": m.clocks,
    }
    if not inplace and m.planned.name == "TILE_VEC":
        e["tile"] = f"{m.plan.tile_rows}x{m.plan.tile_cols}, {m.plan.threads} threads"
        e["aligned_sides"] = {"input": bool(m.plan.vec_in), "output": bool(m.plan.vec_out)}
    if m.flush:
        e["hot_GBps"] = round(gbps(w.algorithmic_bytes * m.k * m.world, m.hot_ms), 2)
        e["roofline_note"] = "input and output fit in L2: not an HBM roofline figure"
    if m.clock_note:
        e["clocks"] = dict(m.clocks, window=m.clock_note)
    return e


def e2e_measure(gpu, m, passes):
    """End to end through the C ABI: pinned host input -> device -> transpose
    -> pinned host output in every step.  Steps rotate over ``--e2e-streams``
    streams, each with its own device and pinned output buffers, so the
    device->host copy of one step overlaps the host->device copy of the next
    (the link carries both directions at once); within a step the three
    operations stay ordered on its stream.  Also times the link alone, one
    direction and both at once, on the same byte counts.  Returns the line's
    ``e2e`` object."""
    import ctypes

    import numpy as np
    import torch
    B, w, args = gpu.B, m.w, gpu.args
    dev = gpu.dev
    k_e2e = max(3, min(args.steps, 20))
    ns = max(2, args.e2e_streams)
    streams = [torch.cuda.Stream(dev) for _ in range(ns)]
    pin_out = torch.empty(w.out_elems, dtype=m.tdt).pin_memory()
    pins_out = [pin_out] + [torch.empty_like(pin_out).pin_memory() for _ in range(ns - 1)]
    bufs = [(m.d_in, m.d_in if m.inplace else m.d_out)]
    for _ in range(ns - 1):
        di = torch.empty_like(m.d_in)
        bufs.append((di, di if m.inplace else torch.empty_like(m.d_out)))
    e_args = []
    for i, st in enumerate(streams):
        di, do = bufs[i]
        a = B.make_args(di.data_ptr(), do.data_ptr(), m.dt, w.batch, w.rows, w.cols, w.ld_in,
                        w.ld_out, w.sin, w.sout, st.cuda_stream)
        e_args.append((a, ctypes.byref(a)))
    ex = gpu.lib.tr_transpose_ex

    def e2e_step_on(i):
        st = streams[i]
        di, do = bufs[i]
        with torch.cuda.stream(st):
            di.copy_(m.pin_in, non_blocking=True)
            if m.inplace:
                rc = m.ipf(di.data_ptr(), 1, w.rows, w.ld_in, w.sin, st.cuda_stream)
            else:
                rc = ex(e_args[i][1], m.po)
            if rc:
                B.check(rc)
            pins_out[i].copy_(do, non_blocking=True)

    def timed_rotation(body, k):
        torch.cuda.synchronize(dev)
        barrier(gpu.world)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(streams[0])
        for st in streams[1:]:
            st.wait_event(t0)
        for j in range(k):
            body(j % ns)
        for st in streams[1:]:
            done = torch.cuda.Event()
            done.record(st)
            streams[0].wait_event(done)
        t1.record(streams[0])
        torch.cuda.synchronize(dev)
        barrier(gpu.world)
        return max_over_ranks(t0.elapsed_time(t1), gpu.world)

    for j in range(ns):  # warm-up
        e2e_step_on(j)
    e_ms = [timed_rotation(e2e_step_on, k_e2e) for _ in range(passes)]
    e_med = statistics.median(e_ms)
    value = gbps(w.algorithmic_bytes * k_e2e * gpu.world, e_med)
    # every end-to-end step uploads the input and transposes it once
    got = pins_out[(k_e2e - 1) % ns].numpy().view(m.x_host.dtype)
    dst = (got[m.jj * w.ld_in + m.ii] if m.inplace
           else got[m.bb * w.sout + m.jj * w.ld_out + m.ii])
    if not np.array_equal(dst, m.src):
        raise SystemExit("bench: end-to-end output differs from the transposed input")

    # the link alone on the same byte counts: uploads, downloads, and both at once
    def up(i):
        with torch.cuda.stream(streams[i]):
            bufs[i][0].copy_(m.pin_in, non_blocking=True)

    def down(i):
        with torch.cuda.stream(streams[i]):
            pins_out[i].copy_(bufs[i][1], non_blocking=True)

    def both(i):
        up(i)
        down((i + 1) % ns)

    h2d_b, d2h_b = w.in_elems * w.esize, w.out_elems * w.esize
    up_ms = statistics.median(timed_rotation(up, k_e2e) for _ in range(passes))
    down_ms = statistics.median(timed_rotation(down, k_e2e) for _ in range(passes))
    both_ms = statistics.median(timed_rotation(both, k_e2e) for _ in range(passes))
    link_both = gbps((h2d_b + d2h_b) * k_e2e * gpu.world, both_ms)
    del bufs, pins_out
    return {"value": round(value, 2), "unit": "GB/s", "statistic": "median of passes",
            "steps": k_e2e, "passes_GBps": [round(gbps(w.algorithmic_bytes * k_e2e * gpu.world, t), 2)
                                            for t in e_ms],
            "overlap": (f"{ns} streams: one step's device->host copy runs with the next one's "
                        "host->device copy"),
            "h2d_bytes_per_step": h2d_b, "d2h_bytes_per_step": d2h_b,
            "link": {"h2d_GBps": round(gbps(h2d_b * k_e2e * gpu.world, up_ms), 2),
                     "d2h_GBps": round(gbps(d2h_b * k_e2e * gpu.world, down_ms), 2),
                     "both_directions_GBps": round(link_both, 2),
                     "note": ("pinned host <-> device copies alone, same bytes and stream "
                              "rotation, no transpose")},
            "pct_of_link": round(100 * value / link_both, 2)}


def run_ours(args):
    import torch

    gpu = Gpu(args)
    B = gpu.B
    w = W.WORKLOADS[args.workload]
    inplace = args.op == "inplace"
    if inplace and (w.rows != w.cols or w.batch != 1):
        raise SystemExit("bench: the in-place transpose needs a square single-plane workload")
    opts = B.make_options(B.Variant[args.variant.upper()], pad=args.pad, stages=args.stages,
                          ctas_per_sm=args.ctas_per_sm, tile_order=args.tile_order,
                          out_stages=args.out_stages, tile_rows=args.tile_rows,
                          tile_cols=args.tile_cols, schedule=args.schedule,
                          threads=args.threads)
    peak, peak_kind = read_peaks()
    per_config = args.per_config == "on" or (
        args.per_config == "auto" and args.workload == DEFAULT_WORKLOAD and not inplace
        and args.variant == "auto" and not any((args.tile_rows, args.tile_cols, args.threads,
                                                args.schedule, args.stages, args.ctas_per_sm,
                                                args.tile_order, args.out_stages)))
    gpu.sampler.start()

    # ---- the headline workload: R passes of exactly K steps each; value = median pass
    m = measure(gpu, w, opts, inplace=inplace)
    per_ms = gpu.step_times(m.step, args.steps)
    tc_ms = statistics.median(gpu.passes(lambda: m.c_out.copy_(m.c_in), args.steps, args.warmup,
                                         args.passes, m.flush))
    torch_copy_gbs = gbps(2 * m.copy_bytes * args.steps * gpu.world, tc_ms)
    e2e = e2e_measure(gpu, m, args.passes)
    head = config_entry(m, peak, inplace)
    kname = {B.Variant.TMA: {1: "k_tma", 3: "k_tma_ldst", 4: "k_tma_ws"}.get(args.schedule, "k_tma_warp"),
             B.Variant.TILE_VEC: "k_tile_vec", B.Variant.TILE_PAD: "k_tile_pad",
             B.Variant.NAIVE_ROW: "k_naive", B.Variant.NAIVE_COL: "k_naive"}.get(m.planned, "?")
    if inplace:
        kname = "k_inplace"
    traffic, traffic_note = recorded_traffic(kname, w.name)
    # the timed passes launch nothing but this kernel, K times each
    kernel_gbs = w.algorithmic_bytes / (m.ms_step / 1e3) / 1e9
    headline = m
    del m

    # ---- every configuration of the workload set, measured the same way
    entries = []
    if per_config:
        for name in PER_CONFIG + PER_CONFIG_EXTRA:
            if name == w.name:
                entries.append(head)
                continue
            mc = measure(gpu, W.WORKLOADS[name], B.make_options(B.Variant.AUTO))
            entries.append(config_entry(mc, peak))
            del mc
            torch.cuda.empty_cache()
        for name in PER_CONFIG_INPLACE:
            mc = measure(gpu, W.WORKLOADS[name], B.make_options(B.Variant.AUTO), inplace=True)
            entries.append(config_entry(mc, peak, inplace=True))
            del mc
            torch.cuda.empty_cache()
    gpu.sampler.stop()

    m = headline
    line = {
        "metric": METRIC, "value": round(m.value, 2), "unit": "GB/s", "n_gpus": gpu.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(m.ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u32" if w.esize == 4 else "u16", "data": "synthetic",
        "config": {"workload": head["workload"],
                   "description": W.DESCRIPTION[w.name] + (", transposed in place" if inplace else ""),
                   "bytes_per_step": w.algorithmic_bytes,
                   "timing": (f"{args.passes} passes of exactly {args.steps} steps after "
                              f"{args.warmup} warm-up steps, each pass between a barrier and a "
                              "device synchronize and timed by CUDA events on the launching "
                              "stream, a bounded device sleep queued before the start event so "
                              "that the host has queued the steps when timing starts; value and "
                              "ms_per_step are the median pass"),
                   "input_placement": ("uploaded from pinned host memory, then rewritten in "
                                       "place by an elementwise device kernel (values unchanged)"),
                   "variant": head["variant"],
                   "l2": ("flushed: a 2x-L2 buffer is written before every step; events around "
                          "each transpose (and each copy) alone" if m.flush else
                          "no flush: input and output each larger than the 129 MB L2"),
                   "parallelism": f"replicas x{gpu.world}"},
        "passes": {"n": len(m.pass_ms), "statistic": "median", "GBps": head["passes_GBps"]},
        "pct_of_hbm_measured": head["pct_of_hbm_measured"],
        "pct_of_hbm_nominal": head["pct_of_hbm_nominal"],
        "pct_of_copy": head["pct_of_copy"],
        "step_ms": {"median": round(statistics.median(per_ms), 5), "min": round(min(per_ms), 5),
                    "p90": round(sorted(per_ms)[int(0.9 * (len(per_ms) - 1))], 5),
                    "pass": "separate pass of K steps with an event after each (not in value)"},
        "copy": {"value": round(m.copy_value, 2), "unit": "GB/s",
                 "bytes_per_step": 2 * m.copy_bytes, "kernel": "tr_copy",
                 "statistic": "median of passes", "torch_copy_GBps": round(torch_copy_gbs, 2)},
        "roofline": {"bound": "hbm", "achieved": round(kernel_gbs, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(kernel_gbs / peak, 4),
                     "traffic": traffic, "peak_source": peak_kind, "kernel": kname,
                     "bytes_per_launch": w.algorithmic_bytes},
        "e2e": e2e,
        "gpu_launches": args.steps * args.passes,
        "clocks": head["clocks"],
    }
    if head.get("tile"):
        line["config"]["tile"] = head["tile"]
    if traffic_note:
        line["roofline"]["traffic_note"] = traffic_note
    if m.flush:
        line["hot"] = {"value": head["hot_GBps"], "unit": "GB/s",
                       "ms_per_step": round(m.hot_ms / args.steps, 5),
                       "note": "median pass of K back-to-back steps, data resident in L2"}
        line["roofline"]["note"] = "input and output fit in L2: not an HBM roofline figure"
    if entries:
        line["per_config"] = entries
    if gpu.rank == 0 and gpu.world == 1 and not args.no_cpu_baseline:
        cgbs, csecs, desc, _ = time_oracle(w, args.cpu_seconds, x=m.x_host)
        line["cpu_baseline"] = {"value": round(cgbs, 3), "unit": "GB/s", "cores": 1,
                                "kind": "oracle", "sample": desc,
                                "seconds": round(csecs, 2), "host_cpus": os.cpu_count(),
                                "host_cpu_model": host_cpu_model()}
        agbs, asecs, adesc, threads = time_oracle_all_cores(w, args.cpu_seconds, x=m.x_host)
        line["cpu_baseline_all_cores"] = {"value": round(agbs, 3), "unit": "GB/s",
                                          "cores": threads, "kind": "oracle", "sample": adesc,
                                          "seconds": round(asecs, 2),
                                          "host_cpus": os.cpu_count(),
                                          "host_cpu_model": host_cpu_model()}
    if gpu.rank == 0:
        print(json.dumps(line), flush=True)
    if gpu.world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


DEFAULT_WORKLOAD = "c2"


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(W.WORKLOADS), default=DEFAULT_WORKLOAD)
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
    ap.add_argument("--passes", type=int, default=5,
                    help="timed passes of K steps; value is the median pass (at least 5)")
    ap.add_argument("--per-config", dest="per_config", choices=["auto", "on", "off"],
                    default="auto",
                    help="also measure every configuration (c1_index, c1_uniform, c2, c3, c4, "
                         "c5), the misaligned-pitch cases and c2 / c5 in place with AUTO; "
                         "auto = only for the default workload and options")
    ap.add_argument("--e2e-streams", dest="e2e_streams", type=int, default=3,
                    help="streams (and buffer sets) the end-to-end steps rotate over")
    ap.add_argument("--clock-window", dest="clock_window", type=float, default=0.5,
                    help="seconds of untimed re-runs for clock sampling when the timed "
                         "passes are shorter than this (0 = none)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # never fewer than 3 untimed warm-up steps
    args.passes = max(5, args.passes)  # the median of at least five passes
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
