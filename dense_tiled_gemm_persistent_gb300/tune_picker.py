"""Measure every kernel configuration over a grid of shapes and write the
picker table the library compiles in.

For each grid point (M, N, K, B layout, operand class) the script times each
candidate configuration through tgemm_run_config on the current GPU
(back-to-back launches over enough rotating operand copies to exceed L2),
twice (forward and reverse candidate order, best of the two), keeps the
fastest, and writes

  * picker_table.csv              every measurement (committed, for review);
  * csrc/tgemm_picker_table.inc   the winner per grid point, as a C array.

Operand classes: 0 = FP16/BF16 (measured FP16 in, FP16 out, both B
layouts, the skinny band included), 1 = FP8 (E4M3 in, BF16 out; the skinny
band on the in-cluster kernel) and 2 = FP32 read as TF32 (FP32 in and out,
more than 64 rows of A); the last two only with B stored N x K, which is all
their kernels take.

Launches are timed from a replayed CUDA graph.  tgemm_run rounds log2 of
each of M, N and K to the nearest grid exponent and uses the winner of its
operand class there; off the grid it falls back to its wave cost model.

Usage (on the GPU machine):
  python -m dense_tiled_gemm_persistent_gb300.tune_picker [--classes 0,1,2] [--skinny-only]
"""
from __future__ import annotations

import argparse
import csv
import ctypes
import math
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

CSV_PATH = os.path.join(HERE, "picker_table.csv")
INC_PATH = os.path.join(HERE, "csrc", "tgemm_picker_table.inc")

# grid exponents: large shapes and the skinny (M <= 64) band
BIG_M = [8, 9, 10, 11, 12, 13, 14]          # 256 .. 16384
BIG_N = [8, 9, 10, 11, 12, 13, 14]
BIG_K = [7, 8, 9, 10, 11, 12, 13]           # 128 .. 8192
SKINNY_M = [0, 3, 4, 5, 6, 7]               # 1, 8, 16, 32, 64, 128
SKINNY_N = [10, 12, 14]                     # 1024, 4096, 16384
SKINNY_K = [10, 12, 13]

L2 = 129 * 1000 * 1000


# operand class -> (input type, output type) the class is measured with
CLASS_TYPES = {0: (0, 0), 1: (3, 1), 2: (2, 2)}


def candidates(tg, M, N=0, dclass=0):
    """(kind, Config) pairs valid for M rows of A (and N columns of B)."""
    C = tg.Config
    out = []
    if M <= 64 and dclass == 0:
        npad = 16 if M <= 16 else (32 if M <= 32 else 64)
        st = {16: 12, 32: 10, 64: 9}[npad]
        mx = {16: 8, 32: 8, 64: 7}[npad]
        for s in (1, 2, 3, 4, 6, 8):
            if s <= mx:
                out.append(("cluster%d" % s, C(bm=128, bn=npad, bk=64, stages=st, cluster_m=s, group_m=1,
                                             split_k=s, swap_ab=2, grid=0)))
        # the half-size ring (two CTAs per SM): twice the resident clusters
        st_h = {16: 6, 32: 5, 64: 4}[npad]
        mx_h = {16: 8, 32: 7, 64: 4}[npad]
        for s in (1, 2, 3, 4, 6, 8):
            if s <= mx_h:
                out.append(("cluster%dh" % s, C(bm=128, bn=npad, bk=64, stages=st_h, cluster_m=s, group_m=1,
                                              split_k=s, swap_ab=2, grid=0)))
        for s in (4, 8, 16):
            out.append(("workspace%d" % s, C(bm=128, bn=npad, bk=64, stages=4, cluster_m=1, group_m=1,
                                             split_k=s, swap_ab=1, grid=0)))
    elif M <= 64 and dclass == 1:
        # FP8: the in-cluster kernel only (no FP8 workspace reduction)
        npad = 16 if M <= 16 else (32 if M <= 32 else 64)
        st = {16: 12, 32: 10, 64: 9}[npad]
        mx = {16: 8, 32: 8, 64: 7}[npad]
        st_h = {16: 6, 32: 5, 64: 4}[npad]
        mx_h = {16: 8, 32: 7, 64: 4}[npad]
        for s in (1, 2, 3, 4, 6, 8):
            if s <= mx:
                out.append(("cluster%d" % s, C(bm=128, bn=npad, bk=64, stages=st, cluster_m=s, group_m=1,
                                             split_k=s, swap_ab=2, grid=0)))
            if s <= mx_h:
                out.append(("cluster%dh" % s, C(bm=128, bn=npad, bk=64, stages=st_h, cluster_m=s, group_m=1,
                                              split_k=s, swap_ab=2, grid=0)))
    elif M <= 128 and dclass in (0, 1):
        # 65-128 rows: the in-cluster kernel padded to 128 (full ring only, up to 4 splits)
        for s in (1, 2, 3, 4):
            out.append(("cluster%d" % s, C(bm=128, bn=128, bk=64, stages=6, cluster_m=s, group_m=1, split_k=s,
                                           swap_ab=2, grid=0)))
    out.append(("pair256", C(bm=256, bn=256, bk=64, stages=6, cluster_m=2, group_m=8, split_k=1, swap_ab=0, grid=0)))
    out.append(("pair256sk", C(bm=256, bn=256, bk=64, stages=6, cluster_m=2, group_m=8, split_k=0, swap_ab=0,
                               grid=0)))
    if M >= 256 and N >= 512:
        # two pairs sharing A (cluster of four): a quarter fewer operand loads per CTA;
        # with a stream-K tail when the leftover wave of blocks is at most half full
        out.append(("quad256", C(bm=256, bn=256, bk=64, stages=6, cluster_m=4, group_m=8, split_k=1, swap_ab=0,
                                 grid=0)))
        out.append(("quad256sk", C(bm=256, bn=256, bk=64, stages=6, cluster_m=4, group_m=8, split_k=0, swap_ab=0,
                                   grid=0)))
    if M >= 4096 and N >= 4096:
        # wider raster bands: more A reuse in L2 per wave on the largest shapes
        out.append(("pair256g16", C(bm=256, bn=256, bk=64, stages=6, cluster_m=2, group_m=16, split_k=1, swap_ab=0,
                                    grid=0)))
    out.append(("cta256", C(bm=128, bn=256, bk=64, stages=4, cluster_m=1, group_m=8, split_k=1, swap_ab=0, grid=0)))
    out.append(("cta128", C(bm=128, bn=128, bk=64, stages=6, cluster_m=1, group_m=8, split_k=1, swap_ab=0, grid=0)))
    if dclass == 0:
        # two-stage ring, two CTAs per SM (16-bit operands only)
        out.append(("cta128s2", C(bm=128, bn=128, bk=64, stages=2, cluster_m=1, group_m=8, split_k=1, swap_ab=0,
                                  grid=0)))
    return out


def time_config(torch, tg, M, N, K, layout, cfg, copies, stream, iters, sustained=False, types=(0, 0)):
    """Microseconds per launch, replaying `iters` launches from a CUDA graph
    (so the host's per-call cost does not hide the kernel's own time)."""
    n = len(copies)
    cap = torch.cuda.Stream()
    sh = ctypes.c_void_p(cap.cuda_stream)

    def run(i):
        A, B, C = copies[i % n]
        return tg.tgemm_run_config(M, N, K, A.data_ptr(), A.shape[1], B.data_ptr(), B.shape[1], layout,
                                   C.data_ptr(), C.shape[1], types[0], types[1], sh, cfg)

    with torch.cuda.stream(cap):
        for i in range(3):
            if run(i) != 0:
                return None
    torch.cuda.synchronize()
    if tg.tgemm_check(sh) != 0:
        return None
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        for i in range(iters):
            if run(i) != 0:
                return None
    graph.replay()
    torch.cuda.synchronize()
    # Long launches are timed in the GPU's steady, power-capped state (a
    # quarter second of warm-up replays, then a quarter second timed): a
    # burst from a cool GPU runs at higher clocks and favours configurations
    # that move more data.
    replays = 1
    if sustained:
        t0 = time.time()
        n = 0
        while time.time() - t0 < 0.25:
            graph.replay()
            torch.cuda.synchronize()
            n += 1
        replays = n                          # as many again, timed: about a quarter second
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(replays):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    if tg.tgemm_check(ctypes.c_void_p(stream.cuda_stream)) != 0:
        return None
    return e0.elapsed_time(e1) / (iters * replays) * 1000.0   # microseconds


def read_rows(path):
    """CSV rows with integer keys; rows written before the operand class
    existed are class 0."""
    with open(path, newline="") as f:
        out = []
        for r in csv.DictReader(f):
            r = dict(r)
            r["dclass"] = int(r.get("dclass") or 0)
            for k in ("em", "en", "ek", "layout"):
                r[k] = int(r[k])
            out.append(r)
        return out


def point_key(r):
    return (r["em"], r["en"], r["ek"], r["layout"], r["dclass"])


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--quick", action="store_true", help="a few grid points only (smoke)")
    ap.add_argument("--skinny-only", action="store_true",
                    help="re-measure the M <= 128 band only and merge it into the existing table and CSV")
    ap.add_argument("--k-exps", default="",
                    help="measure only these log2 K grid exponents (comma-separated); the others are kept")
    ap.add_argument("--classes", default="0,1,2",
                    help="operand classes to measure (0 FP16/BF16, 1 FP8, 2 TF32); the others are kept")
    ap.add_argument("--csv", default=CSV_PATH)
    ap.add_argument("--inc", default=INC_PATH)
    args = ap.parse_args()
    classes = [int(x) for x in args.classes.split(",") if x]

    import torch
    from dense_tiled_gemm_persistent_gb300 import build as lb
    from dense_tiled_gemm_persistent_gb300 import tgemm as tg
    lb.build()
    tg.load()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)

    all_points = []
    for dclass in (0, 1, 2):
        for layout in ((tg.B_NK, tg.B_KN) if dclass == 0 else (tg.B_NK,)):
            for em in BIG_M:
                for en in BIG_N:
                    for ek in BIG_K:
                        all_points.append((em, en, ek, layout, dclass))
            if dclass in (0, 1):
                for em in SKINNY_M:
                    for en in SKINNY_N:
                        for ek in SKINNY_K:
                            all_points.append((em, en, ek, layout, dclass))
    points = [pt for pt in all_points if pt[4] in classes]
    if args.skinny_only:
        points = [pt for pt in points if pt[0] in SKINNY_M]
    if args.k_exps:
        kx = {int(x) for x in args.k_exps.split(",") if x}
        points = [pt for pt in points if pt[2] in kx]
    if args.quick:
        points = points[::37]

    rows, winners = [], []
    t0 = time.time()
    for (em, en, ek, layout, dclass) in points:
        M, N, K = 1 << em, 1 << en, 1 << ek
        tin, tout = CLASS_TYPES[dclass]
        ein, eout = tg_size(tin), tg_size(tout)
        bytes_ = ein * (M * K + K * N) + eout * M * N
        reps = max(1, -(-3 * L2 // bytes_))
        reps = min(reps, 64)
        flops = 2.0 * M * N * K
        iters = int(min(200, max(10, 2e13 / flops)))
        copies = []
        tdt = {0: torch.float16, 1: torch.bfloat16, 2: torch.float32, 3: torch.float8_e4m3fn}
        for _ in range(reps):
            A = torch.randn(M, K, device=dev).to(tdt[tin])
            B = torch.randn(*((N, K) if layout == tg.B_NK else (K, N)), device=dev).to(tdt[tin])
            Cc = torch.empty(M, N, device=dev, dtype=tdt[tout])
            copies.append((A, B, Cc))
        best = None
        # Two passes, the second in reverse order, each candidate keeping its
        # better time: the GPU warms up (and its power-capped clock drops)
        # through a point's candidates, which otherwise favours whichever is
        # timed first.
        cands = candidates(tg, M, N, dclass)
        times = {}
        for order in (cands, cands[::-1]):
            for kind, cfg in order:
                us = time_config(torch, tg, M, N, K, layout, cfg, copies, stream, iters, sustained=flops >= 2e11,
                                 types=(tin, tout))
                if us is not None and (kind not in times or us < times[kind]):
                    times[kind] = us
        for kind, cfg in cands:
            if kind not in times:
                continue
            us = times[kind]
            rows.append(dict(em=em, en=en, ek=ek, layout=layout, dclass=dclass, kind=kind, us=round(us, 3),
                             tflops=round(flops / us / 1e6, 1)))
            if best is None or us < best[0]:
                best = (us, kind, cfg)
        del copies
        if best:
            winners.append((em, en, ek, layout, dclass, best))
        print("%5d %5d %5d %s class %d -> %s %.2f us" % (M, N, K, "nk" if layout else "kn", dclass,
                                                          best[1] if best else None, best[0] if best else -1),
              flush=True)
    print("sweep took %.0f s" % (time.time() - t0))

    lines = {}
    for em, en, ek, layout, dclass, (us, kind, c) in winners:
        lines[(em, en, ek, layout, dclass)] = "{%d, %d, %d, %d, %d, {%d, %d, %d, %d, %d, %d, %d}, %.3ff},  // %s\n" % (
            em, en, ek, layout, dclass, c.bm, c.bn, c.stages, c.cluster_m, c.group_m, c.split_k, c.swap_ab, us,
            kind)
    # keep the measurements and winners of every grid point not measured now
    measured = set(points)
    if os.path.exists(args.csv):
        rows = [r for r in read_rows(args.csv) if point_key(r) not in measured] + rows
    if os.path.exists(args.inc):
        with open(args.inc) as f:
            for line in f:
                if line.startswith("{"):
                    key = tuple(int(x) for x in line[1:].split(",")[:5])
                    if key not in measured and key in set(all_points):
                        lines[key] = line
    order = {pt: i for i, pt in enumerate(all_points)}
    rows.sort(key=lambda r: order.get(point_key(r), -1))
    with open(args.csv, "w", newline="") as f:
        w = csv.DictWriter(f, fieldnames=["em", "en", "ek", "layout", "dclass", "kind", "us", "tflops"])
        w.writeheader()
        w.writerows(rows)
    gpu = torch.cuda.get_device_name(dev)
    with open(args.inc, "w") as f:
        f.write("// Generated by dense_tiled_gemm_persistent_gb300/tune_picker.py on %s.\n" % gpu)
        f.write("// log2 M, log2 N, log2 K, B layout (0 = KxN, 1 = NxK), operand class (0 = FP16/BF16, 1 = FP8, "
                "2 = TF32)\n")
        f.write("// -> fastest measured configuration {bm, bn, stages, cluster_m, group_m, split_k, swap_ab}, "
                "and its time in us.\n")
        for pt in all_points:
            if pt in lines:
                f.write(lines[pt])
    print("wrote", args.csv, "and", args.inc)


def tg_size(t):
    return {0: 2, 1: 2, 2: 4, 3: 1}[t]


if __name__ == "__main__":
    main()
