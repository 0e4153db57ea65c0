"""Host-side pieces of the benchmark: max-over-ranks timing with two gloo
ranks on the CPU, the reference arm's JSON line, and the recorded-traffic
bookkeeping (no GPU)."""
import json
import os
import socket
import subprocess
import sys


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    got = bench.max_over_ranks(10.0 + rank, world)
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 11.0, 1: 11.0}


def test_reference_arm_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "c1_uniform", "--steps", "3", "--warmup", "3"],
                         capture_output=True, text=True, timeout=300, check=True)
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["steps"] == 3


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "c1_uniform", "--steps", "3"], capture_output=True,
                         text=True, timeout=120, env=env)
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_recorded_traffic_tracks_kernel_sources(tmp_path, monkeypatch):
    import bench
    rec = bench.recorded_traffic("k_tile_vec", "c2")
    path = os.path.join(ROOT, "profiles", "traffic.json")
    data = json.load(open(path))
    entry = data.get("k_tile_vec:c2")
    if entry and entry["source_hash"] == bench.kernel_source_hash("k_tile_vec"):
        assert rec[0] == entry["dram_bytes_per_launch"]
    else:
        assert rec == (None, None)
    assert bench.recorded_traffic("k_tile_vec", "no_such_workload") == (None, None)


def test_clock_samples_follow_the_visible_device(monkeypatch):
    """With CUDA_VISIBLE_DEVICES remapping devices, the clock sampler asks
    nvidia-smi for the GPU the process runs on, not the one with its ordinal."""
    import bench

    def fake_run(cmd, **kw):
        ok = cmd[:2] == ["nvidia-smi", "--id=5"]
        return subprocess.CompletedProcess(cmd, 0 if ok else 6, stdout="5\n" if ok else "",
                                           stderr="")

    monkeypatch.setattr(bench.subprocess, "run", fake_run)
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "3,5")
    assert bench.nvsmi_id(1) == "5"
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "")
    assert bench.nvsmi_id(1) == "1"


def test_all_core_oracle_baseline_covers_the_plane():
    """The all-core CPU baseline runs the oracle band by band on several
    threads; one pass of the bands is the whole transpose."""
    import numpy as np

    import bench
    import oracle
    from shared_memory_tiled_gb300 import workloads as W
    w = W.WORKLOADS["c1_uniform"]
    x = W.make_input(w)
    gbs, secs, desc, threads = bench.time_oracle_all_cores(w, 0.05, x=x, threads=3)
    assert gbs > 0 and secs >= 0.05 and threads == 3 and "3 bands" in desc


def test_config_entry_fields():
    """A per-configuration entry carries the value, its copy ratio and roofline
    fraction from the median pass."""
    import bench
    from shared_memory_tiled_gb300 import workloads as W

    class Plan:
        tile_rows, tile_cols, threads, vec_in, vec_out = 64, 64, 256, 1, 1

    class V:
        name = "TILE_VEC"

    m = bench.Measured()
    m.w, m.k, m.world = W.WORKLOADS["c2"], 20, 1
    m.pass_ms = [1.7, 1.6, 1.65, 1.8, 1.62]
    m.med_ms = 1.65
    m.ms_step = m.med_ms / m.k
    m.value = bench.gbps(m.w.algorithmic_bytes * m.k, m.med_ms)
    m.copy_value = 7000.0
    m.flush, m.hot_ms = False, None
    m.planned, m.plan = V(), Plan()
    m.clocks, m.clock_note = {"sm_mhz": 2070.0}, None
    e = bench.config_entry(m, 6769.8)
    assert e["workload"] == "c2" and e["variant"] == "TILE_VEC"
    assert abs(e["value"] - m.w.algorithmic_bytes * 20 / 1.65e-3 / 1e9) < 0.01
    assert e["passes_GBps"][0] < e["value"] < e["passes_GBps"][1]
    assert e["pct_of_copy"] == round(100 * m.value / 7000.0, 2)
    assert e["roofline_frac"] == round(m.value / 6769.8, 4)
    assert e["tile"] == "64x64, 256 threads"
