"""Register and spill budget of the kernels, read from ptxas's resource report
(no GPU).  The default vector tile reaches six resident 256-thread blocks per
SM only at 40 registers or fewer; one more live value in its index path cost
7% on the 8192 x 8192 fp32 workload, so the budget is pinned here."""
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "shared_memory_tiled_gb300", "csrc")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None, reason="nvcc not available")


def ptxas_report(src):
    cmd = ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
           "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"),
           "-I", CSRC, "-Xptxas", "-v", "-c", os.path.join(CSRC, src), "-o", os.devnull]
    out = subprocess.run(cmd, capture_output=True, text=True, check=True).stderr
    kernels, cur = {}, None
    for line in out.splitlines():
        m = re.search(r"Compiling entry function '(\S+)'", line)
        if m:
            cur = m.group(1)
            kernels[cur] = {}
            continue
        if cur is None:
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m:
            kernels[cur]["spill"] = int(m.group(1)) + int(m.group(2))
        m = re.search(r"Used (\d+) registers", line)
        if m:
            kernels[cur]["regs"] = int(m.group(1))
    return kernels


@pytest.fixture(scope="module")
def vec_report():
    import concurrent.futures as cf
    with cf.ThreadPoolExecutor(2) as ex:
        parts = list(ex.map(ptxas_report, ["tile_vec_u32.cu", "tile_vec_u16.cu"]))
    return {**parts[0], **parts[1]}


def _find(report, mangled_part):
    hits = [v for k, v in report.items() if mangled_part in k]
    assert hits, mangled_part
    return hits[0]


def test_default_fp32_vector_tile_fits_six_blocks(vec_report):
    # k_tile_vec<uint32_t, 16, 16, 256, VEC_IN, aligned out, no prefetch>
    k = _find(vec_report, "k_tile_vecIjLi16ELi16ELi256ELb1ELb0ELb0E")
    assert k["regs"] <= 40 and k["spill"] == 0


def test_default_bf16_vector_tile_budget(vec_report):
    k = _find(vec_report, "k_tile_vecItLi16ELi16ELi256ELb1ELb0ELb0E")
    assert k["regs"] <= 80 and k["spill"] == 0


def test_shifted_store_tile_budget(vec_report):
    # 64 registers keep 4 blocks of 256 threads per SM
    k = _find(vec_report, "k_tile_vecIjLi32ELi16ELi256ELb1ELb1ELb0E")  # C3's 128x64 tile
    assert k["regs"] <= 64 and k["spill"] == 0
    # bf16 shifted stores are compiled for 64 registers (4 blocks of 256 / 8 of 128
    # threads per SM) at the price of a few spilled words
    k = _find(vec_report, "k_tile_vecItLi16ELi16ELi256ELb1ELb1ELb0E")  # bf16 128x128, shifted
    assert k["regs"] <= 64 and k["spill"] <= 160
    k = _find(vec_report, "k_tile_vecItLi8ELi16ELi128ELb0ELb1ELb0E")  # both pitches odd
    assert k["regs"] <= 64 and k["spill"] <= 64


def test_realigned_input_tile_budget(vec_report):
    # bf16 128x128 with misaligned input rows (aligned chunks realigned on
    # chip): 80 registers keep 3 blocks of 256 threads per SM
    k = _find(vec_report, "k_tile_vecItLi16ELi16ELi256ELb0ELb0ELb0E")
    assert k["regs"] <= 80 and k["spill"] == 0


def test_inplace_budgets():
    # whole tiles are copied into shared memory asynchronously, so no register
    # holds loaded data: fp32 fits 40 registers (6 blocks/SM, 32 KiB of shared
    # memory each) with at most a few words of the pair walk spilled; bf16 80
    # (3 blocks/SM, 64 KiB of shared memory each), nothing spilled
    rep = ptxas_report("inplace.cu")
    for big in "01":
        k = _find(rep, f"k_inplaceIjLb1ELb{big}E")
        assert k["regs"] <= 40 and k.get("spill", 0) <= 32  # spill stores + loads, bytes
        k = _find(rep, f"k_inplaceItLb1ELb{big}E")
        assert k["regs"] <= 80 and k.get("spill", 0) == 0


@pytest.mark.parametrize("src", ["tile_tma.cu", "inplace.cu", "copy.cu", "tile_lsu.cu"])
def test_no_spills(src):
    for name, k in ptxas_report(src).items():
        if src == "inplace.cu" and "k_inplaceIjLb1E" in name:
            continue  # capped at 40 registers; its allowance is pinned above
        assert k.get("spill", 0) == 0, name
