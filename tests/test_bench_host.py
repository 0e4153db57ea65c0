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
