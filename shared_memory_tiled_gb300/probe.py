"""Shared-memory layout microbenchmarks of libtranspose, one JSON line per run.

    python -m shared_memory_tiled_gb300.probe banks [--reps N] [--blocks-per-sm K]
    python -m shared_memory_tiled_gb300.probe operand [--m M] [--k K] [--bm BM] [--bk BK] [--pad P]

``banks`` times ``tr_bank_probe`` for each tile layout: 0 the unpadded 32 x 32
tile read by columns, 1 the padded 32 x 33 tile, 2 the XOR-swizzled tile, 3
the unpadded tile read by rows.  ``operand`` times ``tr_operand_tiles_f32``
(the padded-SGEMM transposed operand store) with the given As padding
(negative = the rule (32 / BK) % 8).  Every result is checked against its
closed form before its time is reported.
"""
from __future__ import annotations

import argparse
import json
import statistics

import numpy as np

from . import binding as B

LAYOUTS = {0: "pitch 32, column read", 1: "pitch 33, column read",
           2: "xor swizzle, column read", 3: "pitch 32, row read"}


def expected(layout: int, reps: int, threads: int = 256) -> np.ndarray:
    """Each thread's fold: acc = rotl(acc, 1) ^ value, value = row*32 + col."""
    t = np.arange(threads, dtype=np.uint64)
    lane, warp = t & 31, t >> 5
    acc = np.zeros(threads, dtype=np.uint64)
    for r in range(reps):
        c = (r + warp) & 31
        v = c * 32 + lane if layout == 3 else lane * 32 + c
        acc = (((acc << np.uint64(1)) | (acc >> np.uint64(31))) & np.uint64(0xFFFFFFFF)) ^ v
    return acc.astype(np.uint32)


def run(layout: int, reps: int, blocks: int, trials: int = 9):
    import torch
    out = torch.empty(blocks * 256, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    B.check(B.tr_bank_probe(layout, reps, blocks, out.data_ptr(), stream))  # warm-up
    times = []
    for _ in range(trials):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        B.check(B.tr_bank_probe(layout, reps, blocks, out.data_ptr(), stream))
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    got = out.cpu().numpy().view(np.uint32).reshape(blocks, 256)
    ok = bool(np.all(got == expected(layout, reps)[None, :]))
    return statistics.median(times), ok


def run_operand(m, k, bm, bk, pad, trials=9):
    """Time the operand-tile stage on an index-valued M x K matrix; check the
    blocked transposed result against its closed form."""
    import torch
    a = torch.arange(m * k, dtype=torch.int32, device="cuda")
    out = torch.empty(m * k, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    args = (a.data_ptr(), out.data_ptr(), m, k, k, bm, bk, pad, stream)
    B.check(B.tr_operand_tiles_f32(*args))
    times = []
    for _ in range(trials):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        B.check(B.tr_operand_tiles_f32(*args))
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    mt, kt, kk, mm = torch.meshgrid(*(torch.arange(n, device="cuda") for n in
                                      (m // bm, k // bk, bk, bm)), indexing="ij")
    want = ((mt * bm + mm) * k + kt * bk + kk).to(torch.int32).reshape(-1)
    return statistics.median(times), bool(torch.equal(out, want))


def main(argv=None):
    import torch
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    sub = ap.add_subparsers(dest="cmd")
    pb = sub.add_parser("banks")
    pb.add_argument("--reps", type=int, default=4096)
    pb.add_argument("--blocks-per-sm", dest="bps", type=int, default=8)
    po = sub.add_parser("operand")
    po.add_argument("--m", type=int, default=8192)
    po.add_argument("--k", type=int, default=8192)
    po.add_argument("--bm", type=int, default=128)
    po.add_argument("--bk", type=int, default=16)
    po.add_argument("--pad", type=int, default=-1)
    args = ap.parse_args(argv)
    if args.cmd == "operand":
        ms, ok = run_operand(args.m, args.k, args.bm, args.bk, args.pad)
        pad = args.pad if args.pad >= 0 else (32 // args.bk) % 8
        print(json.dumps({"stage": "operand_tiles", "m": args.m, "k": args.k, "bm": args.bm,
                          "bk": args.bk, "pad": pad, "a_stride": args.bm + pad,
                          "median_ms": round(ms, 4),
                          "GBps": round(2 * 4 * args.m * args.k / (ms / 1e3) / 1e9, 1),
                          "result_ok": ok}), flush=True)
        return 0 if ok else 1
    reps = getattr(args, "reps", 4096)
    bps = getattr(args, "bps", 8)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    blocks = sms * bps
    all_ok = True
    for layout, name in LAYOUTS.items():
        ms, ok = run(layout, reps, blocks)
        all_ok &= ok
        reads = blocks * 8 * reps  # warp-level shared loads
        print(json.dumps({"layout": layout, "name": name, "median_ms": round(ms, 4),
                          "warp_reads": reads, "ns_per_warp_read_per_sm":
                          round(ms * 1e6 / (reads / sms), 4), "result_ok": ok}), flush=True)
    return 0 if all_ok else 1


if __name__ == "__main__":
    raise SystemExit(main())
