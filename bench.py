"""Benchmark: device-timed TFLOPS of the tiled GEMM on one GB300.

Workload: C = A * B with M = N = K = 8192, A (M x K) and B stored N x K, both
FP16 drawn uniform on [-0.5, 0.5) from seed 3, FP32 accumulation, FP16
output -- the 8192^3 FP16 problem of the pages' headline table (the Croqtile
tutorial, "Performance at a glance").  A step is one tgemm_run call on the
whole problem; the operands (128 MiB each) and C (128 MiB) together exceed
the 129 MB L2, so back-to-back steps do not run from L2.

Prints one JSON line.  `--impl reference` times the CPU oracle (the plain
FP64 triple loop) on a bounded sample of the same workload instead.  The
library is single-GPU: with more than one GPU (`--gpus N`, or WORLD_SIZE > 1
under torchrun) the GEMM arm prints a line saying so and does no work.  One
of its kernels shares operand tiles between the CTAs of a cluster with TMA
multicast, which is only allowed in code that runs on one GPU alone.

Besides the timed K steps (whose mean is the headline value) the line
carries the median and the best of K individually event-bracketed launches,
the SM clock the GEMM launches measured themselves (tgemm_debug_clock_record)
beside NVML samples of the timed region and probes just before and after it,
a steady-state window of about a second after it (the GB300 settles at its
power limit within a few hundred milliseconds of dense GEMMs), and, from the
CPU-baseline leg, the oracle's check of sampled output elements.
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
# The pages' only figure for this shape: the Croqtile tutorial's tuned kernel,
# 8192^3 FP16, B stored N x K, on an H800 PCIe with FP16 accumulation.  Another
# GPU and another accumulator width: context, not a baseline.
PAGE_CONTEXT = {"tflops": 489.9, "what": "Croqtile tutorial v4 kernel, 8192^3 FP16 N x K, H800 PCIe, "
                                         "FP16 accumulation (another GPU and accumulator: context only)"}
# Dense tensor FLOP per clock per SM of one tcgen05.mma issue stream, by
# operand size in bytes (16-bit 8192; FP8 twice; TF32 half).
FLOP_PER_CLK_SM = {2: 8192, 1: 16384, 4: 4096}
STEADY_STATE_S = 1.0
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


def launch_stats(ms_list):
    """Median and best of per-launch times (milliseconds)."""
    if not ms_list:
        return None
    return {"median": statistics.median(ms_list), "best": min(ms_list), "launches": len(ms_list)}


def per_clock_efficiency(tflops_value: float, sms: int, flop_per_clk: int, sm_mhz):
    """Achieved FLOP/s over what `sms` SMs issue at `sm_mhz` (None without a clock)."""
    if not sm_mhz:
        return None
    return tflops_value * 1e12 / (sms * flop_per_clk * sm_mhz * 1e6)


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

# Clock-event reason bits of NVML's public header (nvml.h).
_REASON_BITS = (("sw_power_cap", 0x4), ("hw_slowdown", 0x8), ("sw_thermal_slowdown", 0x20),
                ("hw_thermal_slowdown", 0x40), ("hw_power_brake_slowdown", 0x80))
_NVML_CLOCK_SM = 1


class ClockSampler:
    """Polls the GPU's SM clock, board power and clock-event reasons in a
    background thread: through NVML (libnvidia-ml, every `period_s`) where
    it loads, else through `nvidia-smi -lms 100`.  Samples carry host
    timestamps (time.perf_counter), so a window can be cut out afterwards."""

    def __init__(self, gpu_uuid=None, period_s=0.002):
        self.gpu_uuid = gpu_uuid
        self.period_s = period_s
        self.samples = []          # (t, sm_mhz, power_w, reasons frozenset)
        self.max_mhz = None
        self.source = None
        self._stop = None
        self._thread = None
        self._proc = None
        self._path = None

    def _nvml(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return None
        if lib.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        rc = -1
        if self.gpu_uuid:
            rc = lib.nvmlDeviceGetHandleByUUID(self.gpu_uuid.encode(), ctypes.byref(h))
        if rc != 0:
            rc = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(0), ctypes.byref(h))
        if rc != 0:
            return None
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, _NVML_CLOCK_SM, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        return lib, h

    def start(self):
        import threading
        nv = self._nvml()
        if nv is not None:
            import ctypes
            lib, h = nv
            self.source = "nvml every %g ms" % (self.period_s * 1e3)
            self._stop = threading.Event()

            def poll():
                clk, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
                while not self._stop.is_set():
                    t = time.perf_counter()
                    if lib.nvmlDeviceGetClockInfo(h, _NVML_CLOCK_SM, ctypes.byref(clk)) == 0:
                        p = mw.value / 1000.0 if lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw)) == 0 else 0.0
                        r = rs.value if lib.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(rs)) == 0 else 0
                        self.samples.append((t, float(clk.value), p,
                                             frozenset(n for n, bit in _REASON_BITS if r & bit)))
                    time.sleep(self.period_s)

            self._thread = threading.Thread(target=poll, daemon=True)
            self._thread.start()
        else:
            fd, self._path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                   "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                   "clocks_event_reasons.sw_power_cap", "--format=csv,noheader,nounits", "-lms", "100"]
            if self.gpu_uuid:
                cmd += ["-i", self.gpu_uuid]
            try:
                self._t0 = time.perf_counter()
                self._proc = subprocess.Popen(cmd, stdout=open(self._path, "w"), stderr=subprocess.DEVNULL)
                self.source = "nvidia-smi every 100 ms (timestamps approximate)"
            except OSError:
                self._proc = None
        time.sleep(0.05)

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
        if self._proc is not None:
            t1 = time.perf_counter()
            self._proc.send_signal(signal.SIGTERM)
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
            rows = []
            for ln in open(self._path).read().splitlines():
                f = [x.strip() for x in ln.split(",")]
                try:
                    rows.append((float(f[0]), float(f[1]), float(f[2]),
                                 frozenset(n for n, v in zip(("hw_slowdown", "hw_thermal_slowdown",
                                                              "sw_thermal_slowdown", "sw_power_cap"), f[3:7])
                                           if v.lower() == "active")))
                except (ValueError, IndexError):
                    continue
            os.unlink(self._path)
            # nvidia-smi prints no timestamps: spread its rows evenly
            n = max(len(rows), 1)
            self.samples = [(self._t0 + (t1 - self._t0) * (i + 0.5) / n, r[0], r[2], r[3])
                            for i, r in enumerate(rows)]
            self.max_mhz = max((r[1] for r in rows), default=None)

    def window(self, t0: float, t1: float):
        """Summary of the samples taken in [t0, t1] (host perf_counter seconds)."""
        inside = [x for x in self.samples if t0 <= x[0] <= t1]
        out = {"samples": len(inside), "source": self.source, "sm_max_mhz": self.max_mhz}
        if len(inside) < 3:
            out.update(sm_mhz=None, reasons=sorted(set().union(*[x[3] for x in inside])) if inside else [],
                       note="fewer than 3 samples inside the window: no median")
            return out
        out.update(sm_mhz=statistics.median(x[1] for x in inside),
                   sm_mhz_min=min(x[1] for x in inside),
                   power_w_median=statistics.median(x[2] for x in inside),
                   power_w_max=max(x[2] for x in inside),
                   reasons=sorted(set().union(*[x[3] for x in inside])))
        return out


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


def sample_points(M: int, N: int, seed: int, n_random: int = 4096):
    """Seeded random output positions plus the first and last row and column
    and the rows/columns at multiples of 128 and 256 minus one and zero."""
    import numpy as np
    rng = np.random.default_rng(seed)
    ii, jj = [rng.integers(0, M, n_random)], [rng.integers(0, N, n_random)]
    for r in sorted({0, 127, 128, 255, 256, M - 1} & set(range(M))):
        ii.append(np.full(N, r))
        jj.append(np.arange(N))
    for c in sorted({0, 127, 128, 255, 256, N - 1} & set(range(N))):
        ii.append(np.arange(M))
        jj.append(np.full(M, c))
    return np.concatenate(ii).astype(np.int64), np.concatenate(jj).astype(np.int64)


def oracle_check(wl, a, b, c_gpu, threads: int):
    """The oracle on sampled elements of the timed run's C: the worst error
    as a fraction of the acceptance bound 1e-3 * sum|A||B| + ulp_out(C_ref)."""
    import numpy as np
    import oracle
    ii, jj = sample_points(wl.M, wl.N, seed=wl.seed)
    ref, bound = oracle.gemm_elements(a, b, wl.M, wl.N, wl.K, a.shape[1], b.shape[1], wl.b_layout,
                                      oracle_input(wl.in_dtype), ii, jj, threads)
    got = c_gpu[ii, jj].double().numpy()
    tol = 1e-3 * bound + oracle.ulp(ref, wl.out_dtype)
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    return {"elements": int(len(ii)), "outside_bound": int(bad.sum()),
            "max_err_over_tol": float(np.max(np.where(bad, np.inf, err / tol))),
            "max_err_over_sum_abs": float(np.max(err / np.maximum(bound, 1e-300))),
            "sample": "4096 seeded random elements plus rows and columns 0, 127, 128, 255, 256 and the last"}


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
        "data": "synthetic", "config": config_dict(wl),
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": used, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_dict(wl):
    """The workload's description; the same dictionary on both arms."""
    from dense_tiled_gemm_persistent_gb300 import inputs as gen
    reps = -(-3 * L2_BYTES // wl.algorithmic_bytes) if wl.algorithmic_bytes < 3 * L2_BYTES else 1
    return {"workload": wl.name, "M": wl.M, "N": wl.N, "K": wl.K,
            "in_dtype": gen.DTYPE_NAME[wl.in_dtype], "out_dtype": gen.DTYPE_NAME[wl.out_dtype],
            "accumulate": "f32", "b_layout": "NxK" if wl.b_layout == gen.B_NK else "KxN",
            "values": "A %s, B %s, seed %d" % (wl.dist_a.describe(), wl.dist_b.describe(), wl.seed),
            "l2": ("back to back over %d copies of A, B, C (%.0f MB > 3 x 129 MB L2)"
                   % (reps, reps * wl.algorithmic_bytes / 1e6)) if reps > 1 else
                  ("operands+output %.0f MB > 129 MB L2, back to back" % (wl.algorithmic_bytes / 1e6)),
            "parallelism": "single-gpu"}


def multi_gpu_line(args, world: int) -> dict:
    """What the GEMM arm prints when asked for more than one GPU."""
    return {"metric": METRIC, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "unavailable": "single-GPU library: one of its kernels shares operand tiles within a cluster by "
                           "TMA multicast, which may only run where one GPU alone is in use; no multi-GPU "
                           "path is built"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="tgemm", choices=["tgemm", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-steady-state", action="store_true")
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
    world = max(int(os.environ.get("WORLD_SIZE", "1")), 1)
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1 or args.gpus > 1:
        if rank == 0:
            print(json.dumps(multi_gpu_line(args, max(world, args.gpus))), flush=True)
        return

    import ctypes

    import torch
    from dense_tiled_gemm_persistent_gb300 import build as libbuild
    from dense_tiled_gemm_persistent_gb300 import inputs as gen
    from dense_tiled_gemm_persistent_gb300 import tgemm

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    libbuild.build()
    tgemm.load()

    wl = workload(args.workload)
    a_cpu, b_cpu = wl.operands()
    A, B = a_cpu.to(dev), b_cpu.to(dev)
    C = torch.empty((wl.M, wl.N), dtype=gen.TORCH_DTYPE[wl.out_dtype], device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = ctypes.c_void_p(stream.cuda_stream)
    lda, ldb, ldc = A.shape[1], B.shape[1], wl.N
    sms = torch.cuda.get_device_properties(dev).multi_processor_count

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
    torch.cuda.synchronize(dev)
    # Two events bracket the whole timed loop: the average launch duration is
    # the loop time over the launch count (an event after every launch would
    # add its own overhead to kernels of a few microseconds).  Small problems
    # replay the loop from a captured CUDA graph so that the host's per-call
    # cost does not starve the GPU; the graph holds the same launches.
    use_graph = args.graph == "on" or (args.graph == "auto" and wl.flops < GRAPH_FLOPS)
    # The kernels' own SM-clock record (tgemm_debug_clock_record): set before
    # any graph is captured, so the captured launches carry it too.
    clock_rec = torch.zeros(8, dtype=torch.int64, device=dev)
    rc = tgemm.tgemm_debug_clock_record(clock_rec.data_ptr())
    if rc != 0:
        raise RuntimeError("tgemm_debug_clock_record: " + tgemm.status_string(rc))

    def kernel_clock():
        torch.cuda.synchronize(dev)
        ns, cyc, n = clock_rec[0].item(), clock_rec[1].item(), clock_rec[2].item()
        clock_rec.zero_()
        torch.cuda.synchronize(dev)
        return {"sm_mhz": cyc * 1e3 / ns if ns > 0 else None, "launches": n,
                "how": "clock64 cycles over globaltimer time inside every GEMM launch (its first CTA, from the "
                       "dependency wait to exit)"}

    cap = torch.cuda.Stream(dev)
    cap_h = ctypes.c_void_p(cap.cuda_stream)

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for i in range(n):
                a_, b_, c_ = copies[i % reps]
                step(c_.data_ptr(), a_.data_ptr(), b_.data_ptr(), cap_h)
        return g

    graph = None
    if use_graph:
        with torch.cuda.stream(cap):
            for i in range(reps):                      # per-stream set-up outside capture
                a_, b_, c_ = copies[i]
                step(c_.data_ptr(), a_.data_ptr(), b_.data_ptr(), cap_h)
        torch.cuda.synchronize(dev)
        graph = capture(args.steps)
        graph.replay()
        torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    kernel_clock()                                     # drop what warm-up and capture recorded
    # SM-clock probes (tgemm_debug_sm_clock: clock64 cycles over globaltimer
    # time on one SM) just before and just after the timed region, outside
    # its events, on the same stream.
    probe_buf = torch.zeros(8, dtype=torch.int64, device=dev)

    def probe(slot):
        rc_ = tgemm.tgemm_debug_sm_clock(probe_buf.data_ptr() + 16 * slot, 20, sh)
        if rc_ != 0:
            raise RuntimeError("tgemm_debug_sm_clock: " + tgemm.status_string(rc_))

    def probe_mhz(slot):
        ns, cyc = probe_buf[2 * slot].item(), probe_buf[2 * slot + 1].item()
        return cyc * 1e3 / ns if ns > 0 else None

    probe(0)
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_host0 = time.perf_counter()
    e_start.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i in range(args.steps):
            a_, b_, c_ = copies[i % reps]
            step(c_.data_ptr(), a_.data_ptr(), b_.data_ptr())
    e_end.record(stream)
    probe(1)
    torch.cuda.synchronize(dev)
    t_host1 = time.perf_counter()
    rc = tgemm.tgemm_check(sh)
    if rc != 0:
        raise RuntimeError("timed region failed: " + tgemm.status_string(rc))
    total_ms = e_start.elapsed_time(e_end)
    ms_per_step = total_ms / args.steps
    value = tflops(wl.M, wl.N, wl.K, ms_per_step)
    avg_launch = ms_per_step
    flop_clk = FLOP_PER_CLK_SM[gen.DTYPE_SIZE[wl.in_dtype]]
    clocks = sampler.window(t_host0, t_host1)
    clocks["window"] = "the timed region (%.1f ms of host time)" % ((t_host1 - t_host0) * 1e3)
    # NVML's clock and power readings trail the hardware by tens of
    # milliseconds (a 12 ms dense-GEMM burst reads as ~170 W on a board that
    # draws 1.4 kW in it), so inside a region that short they show the state
    # before it: they are reported, but no per-clock efficiency is derived
    # from them.  The steady-state window below is long enough.
    in_kernel = kernel_clock()
    mhz0, mhz1 = probe_mhz(0), probe_mhz(1)
    clocks["sm_mhz_probe"] = {"before": mhz0, "after": mhz1,
                              "how": "clock64 cycles over 20 us of globaltimer on one SM, just before and just "
                                     "after the timed region"}
    clocks["sm_mhz_in_kernels"] = in_kernel
    if (t_host1 - t_host0) < 0.25:
        clocks["note"] = ("timed region shorter than NVML's update interval: its NVML samples show the clock "
                          "before the region; sm_mhz_in_kernels is the clock the GEMM launches themselves "
                          "measured, and steady_state holds a second of clocks under load")
    clocks["per_clock_efficiency"] = per_clock_efficiency(value, sms, flop_clk, in_kernel["sm_mhz"])
    clocks["per_clock_basis"] = "sm_mhz_in_kernels"

    # Per-launch distribution: K more launches (graph mode: blocks of up to
    # 10 replayed launches), each bracketed by its own pair of events.
    per = []
    if graph is not None:
        blk = max(1, min(10, args.steps))
        g_blk = capture(blk)
        for _ in range(max(1, args.steps // blk)):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g_blk.replay()
            e1.record(stream)
            e1.synchronize()
            per.append(e0.elapsed_time(e1) / blk)
    else:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for i, (e0, e1) in enumerate(evs):
            a_, b_, c_ = copies[i % reps]
            e0.record(stream)
            step(c_.data_ptr(), a_.data_ptr(), b_.data_ptr())
            e1.record(stream)
        torch.cuda.synchronize(dev)
        per = [e0.elapsed_time(e1) for e0, e1 in evs]
    kernel_clock()
    kstats = launch_stats(per) or {}
    kernel_ms = {"mean": avg_launch, "median": kstats.get("median"), "best": kstats.get("best"),
                 "distribution": "%d %s, an event pair around each" % (
                     len(per), "blocks of %d graph-replayed launches" % blk if graph is not None
                     else "launches")}

    # Steady state: about a second of back-to-back steps after the timed
    # region, with the clocks sampled inside it.  The GPU reaches its power
    # limit there; the timed K steps may still run at burst clocks.
    steady = None
    if not args.no_steady_state:
        n_ss = max(args.steps, int(STEADY_STATE_S * 1e3 / max(avg_launch, 1e-4)))
        if graph is not None:
            n_rep = max(1, n_ss // args.steps)
            n_ss = n_rep * args.steps
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        e0.record(stream)
        if graph is not None:
            for _ in range(n_rep):
                graph.replay()
        else:
            for i in range(n_ss):
                a_, b_, c_ = copies[i % reps]
                step(c_.data_ptr(), a_.data_ptr(), b_.data_ptr())
        e1.record(stream)
        probe(2)
        torch.cuda.synchronize(dev)
        t1 = time.perf_counter()
        ss_ms = e0.elapsed_time(e1) / n_ss
        ss_val = tflops(wl.M, wl.N, wl.K, ss_ms)
        # skip the first quarter: the clock falls from burst to its power-limited level
        ss_clk = sampler.window(t0 + 0.25 * (t1 - t0), t1)
        ss_clk["sm_mhz_probe_after"] = probe_mhz(2)
        ss_clk["sm_mhz_in_kernels"] = kernel_clock()
        steady = {"steps": n_ss, "seconds": (t1 - t0), "ms_per_step": ss_ms, "value": ss_val, "unit": "TFLOPS",
                  "clocks": ss_clk,
                  "per_clock_efficiency": per_clock_efficiency(ss_val, sms, flop_clk,
                                                               ss_clk["sm_mhz_in_kernels"]["sm_mhz"])}
    sampler.stop()
    tgemm.tgemm_debug_clock_record(None)
    rc = tgemm.tgemm_check(sh)
    if rc != 0:
        raise RuntimeError("distribution/steady-state launches failed: " + tgemm.status_string(rc))

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
            sus = rate * float(peaks["bf16_tflops_sustained"])
            roofline["frac_of_sustained"] = achieved / sus
            if steady is not None:
                steady["frac_of_sustained"] = steady["value"] / sus
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
        e2e = {"value": tflops(wl.M, wl.N, wl.K, e2e_ms), "unit": "TFLOPS",
               "h2d_bytes_per_step": a_cpu.numel() * a_cpu.element_size() + b_cpu.numel() * b_cpu.element_size(),
               "d2h_bytes_per_step": hcs[0].numel() * hcs[0].element_size(), "ms_per_step": e2e_ms,
               "pipelined": "H2D of step i+1 and D2H of step i-1 overlap the GEMM of step i (two buffer sets)"}
        rc = tgemm.tgemm_check(sh)
        if rc != 0:
            raise RuntimeError("end-to-end launches failed: " + tgemm.status_string(rc))

    # CPU-baseline leg: the oracle timed on a row sample of the headline
    # workload, and the oracle's check of sampled elements of the C that the
    # timed launches wrote (any workload).
    cpu = None
    parity = None
    if not args.no_cpu_baseline:
        import oracle
        oracle.build()
        threads = os.cpu_count() or 1
        parity = oracle_check(wl, a_cpu, b_cpu, C.cpu(), threads)
        if args.workload == WORKLOAD:
            v, dt, rows = cpu_oracle_sample(wl, a_cpu, b_cpu, 15.0, threads)
            cpu = {"value": v, "unit": "TFLOPS", "cores": min(threads, rows), "kind": "oracle",
                   "sample": "rows 0..%d of C (%d x %d outputs, K = %d), FP64 dot products, %.1f s" % (
                       rows - 1, rows, wl.N, wl.K, dt)}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": gen.DTYPE_NAME[wl.in_dtype], "data": "synthetic",
        "config": config_dict(wl),
        "kernel": dict(picked.as_dict(), launch="cuda_graph" if graph is not None else "stream",
                       epilogue=args.epilogue),
        "roofline": roofline, "cpu_baseline": cpu, "parity": parity, "e2e": e2e,
        "clocks": clocks, "steady_state": steady, "gpu_launches": args.steps,
        "kernel_ms": kernel_ms,
        "page_context": dict(PAGE_CONTEXT, ratio=value / PAGE_CONTEXT["tflops"]) if wl.name == WORKLOAD else None,
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
