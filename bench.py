"""Benchmark: device-timed TFLOPS of the tiled GEMM on one GB300.

Workload: C = A * B with M = N = K = 8192, A (M x K) and B stored N x K, both
FP16 drawn uniform on [-0.5, 0.5) from seed 3, FP32 accumulation, FP16
output -- the 8192^3 FP16 problem of the pages' headline table (the Croqtile
tutorial, "Performance at a glance").  A step is one tgemm_run call on the
whole problem; the operands (128 MiB each) and C (128 MiB) together exceed
the 129 MB L2, so back-to-back steps do not run from L2.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle (the
plain FP64 triple loop) on a bounded sample of the same workload instead.
Several GPUs under torchrun run independent replicas (no collective on the
data path); value is the FLOPs of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import signal
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "gemm_8192x8192x8192_f16_nk_f16"
METRIC = "GEMM TFLOPS (device-timed) and fraction of GB300 dense FP16/BF16 tensor peak"
PUBLISHED_TFLOPS = 489.9      # Croqtile v4 on H800 PCIe, same shape and B layout (context, other GPU)
FALLBACK_TENSOR_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1000 * 1000
GRAPH_FLOPS = 1e11
KERNEL_SOURCES = ["tgemm_kernel.cuh", "tgemm_kernel_pair.cuh", "tgemm_kernel_quad.cuh",
                  "tgemm_kernel_skinny.cuh", "tgemm_kernel_splitk_cluster.cuh", "tgemm_ptx.cuh", "tgemm_wait.cuh",
                  "tgemm_sched.h", "tgemm_params.h"]


def tflops(M: int, N: int, K: int, ms: float) -> float:
    """2*M*N*K floating-point operations over `ms` milliseconds, in TFLOP/s."""
    return 2.0 * M * N * K / (ms * 1e-3) / 1e12


def aggregate(total_ms_local: float, steps: int, flops_per_step: float, world: int, device="cpu"):
    """Whole-job throughput of `world` replicas: every rank ran `steps` steps
    of `flops_per_step`; the job's time is the slowest rank's.  Returns
    (max_ms, ms_per_step, TFLOPS over all ranks)."""
    total = float(total_ms_local)
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([total], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total = float(t.item())
    ms_per_step = total / steps
    return total, ms_per_step, flops_per_step * world / (ms_per_step * 1e-3) / 1e12


def kernel_digest() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "dense_tiled_gemm_persistent_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return None


def recorded_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    digest = kernel_digest()
    for ln in lines:
        parts = ln.split()
        if len(parts) == 3 and not ln.startswith("#") and parts[0] == workload and parts[1] == digest:
            return int(parts[2])
    return None


# ---- clocks --------------------------------------------------------------------

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_uuid=None):
        self.proc = None
        self.path = None
        self.gpu_uuid = gpu_uuid

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", "--query-gpu=" + CLOCK_FIELDS, "--format=csv,noheader,nounits", "-lms", "100"]
        if self.gpu_uuid:
            cmd += ["-i", self.gpu_uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.send_signal(signal.SIGTERM)
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ln in open(self.path).read().splitlines():
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), max=float(f[2]), power=float(f[3]), hw=f[5], hw_th=f[6],
                                 sw_th=f[7], pcap=f[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        smax = max(r["max"] for r in rows)
        loaded = [r for r in rows if r["power"] > 200] or rows
        reasons = set()
        for r in loaded:
            for key, name in (("hw", "hw_slowdown"), ("hw_th", "hw_thermal_slowdown"),
                              ("sw_th", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": max(r["power"] for r in rows)}


# ---- workload --------------------------------------------------------------------

def workload(name=WORKLOAD):
    from dense_tiled_gemm_persistent_gb300 import inputs as gen
    return gen.WORKLOADS[name]


def oracle_input(in_dtype: int) -> int:
    """The oracle's code for an input type: FP32 operands are multiplied as
    TF32, which the oracle names separately; the other codes coincide."""
    import oracle
    from dense_tiled_gemm_persistent_gb300 import inputs as gen
    return oracle.TF32 if in_dtype == gen.F32 else in_dtype


def cpu_oracle_sample(wl, a, b, budget_s: float, threads: int):
    """Time the oracle on rows [0, r) of C, r a multiple of the thread count
    chosen to fill about budget_s seconds; returns (TFLOPS, seconds, rows)."""
    import oracle
    lda, ldb = a.shape[1], b.shape[1]
    dt_in = oracle_input(wl.in_dtype)
    t0 = time.perf_counter()
    oracle.gemm_rows(a, b, wl.M, wl.N, wl.K, lda, ldb, wl.b_layout, dt_in, 0, threads, False, threads)
    t_wave = time.perf_counter() - t0                     # one row per thread
    rows = min(wl.M, max(1, int(budget_s / max(t_wave, 1e-9))) * threads)
    t0 = time.perf_counter()
    oracle.gemm_rows(a, b, wl.M, wl.N, wl.K, lda, ldb, wl.b_layout, dt_in, 0, rows, False, threads)
    dt = time.perf_counter() - t0
    return tflops(rows, wl.N, wl.K, dt * 1e3), dt, rows


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle as it stands, rank 0 only."""
    if rank != 0:
        return
    wl = workload(getattr(args, "workload", WORKLOAD))
    a, b = wl.operands()
    threads = os.cpu_count() or 1
    dt_in = oracle_input(wl.in_dtype)
    total_budget = 120.0
    per_step = max(0.05, min(20.0, total_budget / max(args.steps + args.warmup, 1)))
    import oracle
    oracle.build()
    # rows per step: calibrate on one row per thread
    t0 = time.perf_counter()
    oracle.gemm_rows(a, b, wl.M, wl.N, wl.K, a.shape[1], b.shape[1], wl.b_layout, dt_in, 0,
                     threads, False, threads)
    t_wave = time.perf_counter() - t0
    rows = max(1, min(wl.M, int(per_step / max(t_wave, 1e-9)) * threads))
    if rows < threads:
        rows = max(1, int(per_step / max(t_wave, 1e-9) * threads))
    used = min(threads, rows)
    times = []
    for step in range(args.warmup + args.steps):
        r0 = (step * rows) % max(wl.M - rows + 1, 1)
        t0 = time.perf_counter()
        oracle.gemm_rows(a, b, wl.M, wl.N, wl.K, a.shape[1], b.shape[1], wl.b_layout, dt_in, r0,
                         r0 + rows, False, threads)
        if step >= args.warmup:
            times.append(time.perf_counter() - t0)
    total = sum(times)
    value = tflops(rows * len(times), wl.N, wl.K, total * 1e3)
    sample = "%d rows of C per step (%d x %d outputs, K = %d), FP64 dot products on %d threads" % (
        rows, rows, wl.N, wl.K, used)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total * 1e3 / max(len(times), 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_dict(wl, world),
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": used, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_dict(wl, world):
    from dense_tiled_gemm_persistent_gb300 import inputs as gen
    reps = -(-3 * L2_BYTES // wl.algorithmic_bytes) if wl.algorithmic_bytes < 3 * L2_BYTES else 1
    return {"workload": wl.name, "M": wl.M, "N": wl.N, "K": wl.K,
            "in_dtype": gen.DTYPE_NAME[wl.in_dtype], "out_dtype": gen.DTYPE_NAME[wl.out_dtype],
            "accumulate": "f32", "b_layout": "NxK" if wl.b_layout == gen.B_NK else "KxN",
            "values": "A %s, B %s, seed %d" % (wl.dist_a.describe(), wl.dist_b.describe(), wl.seed),
            "l2": ("back to back over %d copies of A, B, C (%.0f MB > 3 x 129 MB L2)"
                   % (reps, reps * wl.algorithmic_bytes / 1e6)) if reps > 1 else
                  ("operands+output %.0f MB > 129 MB L2, back to back" % (wl.algorithmic_bytes / 1e6)),
            "parallelism": "replicas%d" % world if world > 1 else "single-gpu"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="tgemm", choices=["tgemm", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--config", default="auto",
                    choices=["auto", "pair", "pairsk", "quad", "quadsk", "1cta256", "1cta128", "workspace"],
                    help="tile shape: the library's pick, or a forced one (tuning)")
    ap.add_argument("--group-m", type=int, default=0, help="GROUP_SIZE_M override (0: library default)")
    ap.add_argument("--epilogue", default="none", choices=["none", "bias_gelu", "residual"],
                    help="fused epilogue (timing of a widened row; the headline line uses none)")
    ap.add_argument("--split-k", type=int, default=0, help="split count override for the swap-AB path (tuning)")
    ap.add_argument("--stages", type=int, default=0,
                    help="ring depth override for the swap-AB path (tuning; selects the in-cluster ring budget)")
    ap.add_argument("--graph", default="auto", choices=["auto", "on", "off"],
                    help="replay the timed launches from a CUDA graph (auto: problems under 1e11 FLOP)")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="another named workload (parity-test configurations; not the headline line)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    import torch.distributed as dist
    from dense_tiled_gemm_persistent_gb300 import build as libbuild
    from dense_tiled_gemm_persistent_gb300 import inputs as gen
    from dense_tiled_gemm_persistent_gb300 import tgemm
    import ctypes

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    libbuild.build()
    tgemm.load()

    wl = workload(args.workload)
    a_cpu, b_cpu = wl.operands()
    A, B = a_cpu.to(dev), b_cpu.to(dev)
    C = torch.empty((wl.M, wl.N), dtype=gen.TORCH_DTYPE[wl.out_dtype], device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = ctypes.c_void_p(stream.cuda_stream)
    lda, ldb, ldc = A.shape[1], B.shape[1], wl.N

    rc, picked = tgemm.tgemm_query_config(wl.M, wl.N, wl.K, wl.b_layout, wl.in_dtype, wl.out_dtype)
    if rc != 0:
        raise RuntimeError("tgemm_query_config: " + tgemm.status_string(rc))
    forced = None
    if args.config == "workspace" and picked.swap_ab:
        forced = tgemm.Config(bm=picked.bm, bn=picked.bn, bk=64, stages=4, cluster_m=1, group_m=1,
                              split_k=args.split_k or picked.split_k, swap_ab=1, grid=0)
        picked = forced
    elif (args.split_k or args.stages) and picked.swap_ab:
        sk = args.split_k or picked.split_k
        forced = tgemm.Config(bm=picked.bm, bn=picked.bn, bk=64, stages=args.stages or picked.stages,
                              cluster_m=sk if picked.swap_ab == 2 else 1, group_m=1,
                              split_k=sk, swap_ab=picked.swap_ab, grid=0)
        picked = forced
    elif args.config != "auto" or args.group_m:
        shapes = {"pair": (256, 256, 6, 2, 1), "pairsk": (256, 256, 6, 2, 0), "quad": (256, 256, 6, 4, 1),
                  "quadsk": (256, 256, 6, 4, 0), "1cta256": (128, 256, 4, 1, 1),
                  "1cta128": (128, 128, 6, 1, 1)}
        bm, bn, st, cl, sk = shapes[args.config] if args.config != "auto" else (
            picked.bm, picked.bn, picked.stages, picked.cluster_m, picked.split_k)
        forced = tgemm.Config(bm=bm, bn=bn, bk=64, stages=st, cluster_m=cl,
                              group_m=args.group_m or picked.group_m, split_k=sk, swap_ab=0, grid=0)
        picked = forced

    ep = None
    if args.epilogue != "none":
        g_ep = torch.Generator().manual_seed(11)
        bias_t = torch.randn(wl.N, generator=g_ep).to(gen.TORCH_DTYPE[wl.out_dtype]).to(dev)
        cin_t = torch.randn(wl.M, wl.N, generator=g_ep).to(gen.TORCH_DTYPE[wl.out_dtype]).to(dev)
        if args.epilogue == "bias_gelu":
            ep = tgemm.Epilogue(alpha=1.0, beta=0.0, c_in=None, ldc_in=wl.N, bias=bias_t.data_ptr(),
                                bias_dtype=wl.out_dtype, act=tgemm.ACT_GELU_TANH)
        else:   # residual: D = A*B + C_in
            ep = tgemm.Epilogue(alpha=1.0, beta=1.0, c_in=cin_t.data_ptr(), ldc_in=wl.N, bias=None,
                                bias_dtype=wl.out_dtype, act=tgemm.ACT_NONE)

    def step(c_ptr=None, a_ptr=None, b_ptr=None, stream_handle=None):
        args_ = (wl.M, wl.N, wl.K, a_ptr or A.data_ptr(), lda, b_ptr or B.data_ptr(), ldb,
                 wl.b_layout, c_ptr or C.data_ptr(), ldc, wl.in_dtype, wl.out_dtype, stream_handle or sh)
        if ep is not None:
            rc = tgemm.tgemm_run_ex(*args_, ep, forced)
        else:
            rc = tgemm.tgemm_run(*args_) if forced is None else tgemm.tgemm_run_config(*args_, forced)
        if rc != 0:
            raise RuntimeError("tgemm_run: " + tgemm.status_string(rc))

    for _ in range(args.warmup):
        step()
    rc = tgemm.tgemm_check(sh)
    if rc != 0:
        raise RuntimeError("warm-up failed: " + tgemm.status_string(rc))

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    sampler = ClockSampler(uuid)
    sampler.start()

    # Workloads whose operands fit in L2 cycle through R copies of A, B and C
    # (R * bytes > 3 x L2), so every launch streams its operands from HBM;
    # launches run back to back either way.
    reps = 1
    if wl.algorithmic_bytes < 3 * L2_BYTES:
        reps = -(-3 * L2_BYTES // wl.algorithmic_bytes)
    copies = [(A, B, C)] + [(A.clone(), B.clone(), torch.empty_like(C)) for _ in range(reps - 1)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    # Two events bracket the whole timed loop: the average launch duration is
    # the loop time over the launch count (an event after every launch would
    # add its own overhead to kernels of a few microseconds).  Small problems
    # replay the loop from a captured CUDA graph so that the host's per-call
    # cost does not starve the GPU; the graph holds the same launches.
    use_graph = args.graph == "on" or (args.graph == "auto" and wl.flops < GRAPH_FLOPS)
    graph = None
    if use_graph:
        cap = torch.cuda.Stream(dev)
        cap_h = ctypes.c_void_p(cap.cuda_stream)
        with torch.cuda.stream(cap):
            for i in range(reps):                      # per-stream set-up outside capture
                a_, b_, c_ = copies[i]
                step(c_.data_ptr(), a_.data_ptr(), b_.data_ptr(), cap_h)
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            for i in range(args.steps):
                a_, b_, c_ = copies[i % reps]
                step(c_.data_ptr(), a_.data_ptr(), b_.data_ptr(), cap_h)
        graph.replay()
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i in range(args.steps):
            a_, b_, c_ = copies[i % reps]
            step(c_.data_ptr(), a_.data_ptr(), b_.data_ptr())
    e_end.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    rc = tgemm.tgemm_check(sh)
    if rc != 0:
        raise RuntimeError("timed region failed: " + tgemm.status_string(rc))
    total_ms = e_start.elapsed_time(e_end)
    local_ms = total_ms
    total_ms, ms_per_step, value = aggregate(local_ms, args.steps, wl.flops, world, dev)
    avg_launch = local_ms / args.steps

    peaks = measured_peaks()
    # nominal dense rates relative to FP16/BF16 (2.25 PFLOP/s): FP8 4.5, TF32 1.1
    rate = {1: 2.0, 2: 1.0, 4: 1.1 / 2.25}[gen.DTYPE_SIZE[wl.in_dtype]]
    if peaks and peaks.get("bf16_tflops"):
        peak_t, src_t = rate * float(peaks["bf16_tflops"]), "measured (cuBLAS bf16 burst; fp16 dense rate equals bf16)"
        if rate != 1.0:
            src_t = "measured cuBLAS bf16 burst x %.3g (nominal %s/BF16 dense ratio)" % (
                rate, "FP8" if rate > 1 else "TF32")
    else:
        peak_t, src_t = rate * FALLBACK_TENSOR_TFLOPS, "fallback" + (" x %.3g" % rate if rate != 1.0 else "")
    if peaks and peaks.get("hbm_gbs"):
        peak_h, src_h = float(peaks["hbm_gbs"]), "measured (copy)"
    else:
        peak_h, src_h = FALLBACK_HBM_GBS, "fallback"
    ridge = peak_t * 1e12 / (peak_h * 1e9)          # FLOP per byte where the two roofs meet
    ai = wl.flops / wl.algorithmic_bytes
    if ai >= ridge:
        achieved = tflops(wl.M, wl.N, wl.K, avg_launch)
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak_t, "unit": "TFLOP/s",
                    "frac": achieved / peak_t, "peak_source": src_t}
        if peaks and peaks.get("bf16_tflops_sustained"):
            roofline["frac_of_sustained"] = achieved / (rate * float(peaks["bf16_tflops_sustained"]))
    else:
        achieved = wl.algorithmic_bytes / (avg_launch * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peak_h, "unit": "GB/s",
                    "frac": achieved / peak_h, "peak_source": src_h}
    roofline.update({"traffic": recorded_traffic(wl.name), "algorithmic_bytes": wl.algorithmic_bytes,
                     "flops_per_launch": wl.flops, "arithmetic_intensity": ai})

    # End to end through the C ABI with host buffers: every step copies its A
    # and B in from pinned host memory, runs the GEMM and copies its C out to
    # pinned host memory.  Steps are pipelined over three streams with two
    # device buffer sets: the H2D copy of step i+1 and the D2H copy of step i-1
    # overlap the GEMM of step i (events order each buffer's reuse).
    e2e = None
    if not args.no_e2e:
        ha = a_cpu.pin_memory()
        hb = b_cpu.pin_memory()
        hcs = [torch.empty((wl.M, wl.N), dtype=gen.TORCH_DTYPE[wl.out_dtype]).pin_memory() for _ in range(2)]
        bufs = [(torch.empty_like(A), torch.empty_like(B), torch.empty_like(C)) for _ in range(2)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        s_comp = stream
        comp_h = ctypes.c_void_p(s_comp.cuda_stream)
        in_done = [torch.cuda.Event() for _ in range(2)]
        comp_done = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]
        for ev in comp_done + out_done:
            ev.record(s_comp)

        def e2e_step(i):
            bi = i % 2
            A2, B2, C2 = bufs[bi]
            s_in.wait_event(comp_done[bi])          # the GEMM two steps back is done reading A2, B2
            with torch.cuda.stream(s_in):
                A2.copy_(ha, non_blocking=True)
                B2.copy_(hb, non_blocking=True)
            in_done[bi].record(s_in)
            s_comp.wait_event(in_done[bi])
            s_comp.wait_event(out_done[bi])         # C2 from two steps back is on the host
            step(C2.data_ptr(), A2.data_ptr(), B2.data_ptr(), comp_h)
            comp_done[bi].record(s_comp)
            s_out.wait_event(comp_done[bi])
            with torch.cuda.stream(s_out):
                hcs[bi].copy_(C2, non_blocking=True)
            out_done[bi].record(s_out)

        for i in range(4):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_comp)
        s_in.wait_event(e0)
        for i in range(args.e2e_steps):
            e2e_step(i)
        s_comp.wait_event(out_done[(args.e2e_steps - 1) % 2])
        s_comp.wait_event(out_done[args.e2e_steps % 2])
        e1.record(s_comp)
        torch.cuda.synchronize(dev)
        e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
        e2e = {"value": tflops(wl.M, wl.N, wl.K, e2e_ms) * world, "unit": "TFLOPS",
               "h2d_bytes_per_step": a_cpu.numel() * a_cpu.element_size() + b_cpu.numel() * b_cpu.element_size(),
               "d2h_bytes_per_step": hcs[0].numel() * hcs[0].element_size(), "ms_per_step": e2e_ms,
               "pipelined": "H2D of step i+1 and D2H of step i-1 overlap the GEMM of step i (two buffer sets)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.workload == WORKLOAD:
        import oracle
        oracle.build()
        threads = os.cpu_count() or 1
        v, dt, rows = cpu_oracle_sample(wl, a_cpu, b_cpu, 15.0, threads)
        cpu = {"value": v, "unit": "TFLOPS", "cores": min(threads, rows), "kind": "oracle",
               "sample": "rows 0..%d of C (%d x %d outputs, K = %d), FP64 dot products, %.1f s" % (
                   rows - 1, rows, wl.N, wl.K, dt)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": value / PUBLISHED_TFLOPS if wl.name == WORKLOAD else None,
            "dtype": gen.DTYPE_NAME[wl.in_dtype], "data": "synthetic",
            "config": dict(config_dict(wl, world), kernel=picked.as_dict(),
                           launch="cuda_graph" if graph is not None else "stream", epilogue=args.epilogue),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "clocks": clocks, "gpu_launches": args.steps,
            "kernel_ms": {"mean": avg_launch},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
