"""Python binding of the C ABI in include/tgemm.h (libtgemm.so).

Argument marshalling only: every element of C is computed by the library's
CUDA kernels.  There is no CPU fallback; if the library is missing, every
call raises.  The raw functions mirror the C names and take integer device
pointers and a stream handle; ``matmul`` is a thin convenience that derives
sizes and leading dimensions from torch tensors.
"""
from __future__ import annotations

import ctypes
import os
import threading

F16, BF16, F32, E4M3, E5M2 = 0, 1, 2, 3, 4   # FP8 inputs only; FP8/FP32 inputs: B stored N x K
B_KN, B_NK = 0, 1

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_MISALIGNED, ERR_ARCH, ERR_CUDA, ERR_OOM, ERR_TIMEOUT = range(8)

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libtgemm.so")

# Every symbol include/tgemm.h declares.
EXPORTS = ("tgemm_run", "tgemm_query_config", "tgemm_query_config_sms", "tgemm_run_config", "tgemm_check",
           "tgemm_last_fault_code", "tgemm_status_string", "tgemm_shutdown", "tgemm_tile_coord",
           "tgemm_debug_wait_timeout", "tgemm_debug_tile_order", "tgemm_stream_k_plan", "tgemm_group_size",
           "tgemm_run_noalloc",
           "tgemm_run_ex", "tgemm_run_strided_batched", "tgemm_debug_noalloc_wait_timeout",
           "tgemm_debug_sm_clock", "tgemm_debug_clock_record")

ACT_NONE, ACT_RELU, ACT_GELU_TANH = 0, 1, 2


class TgemmError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s failed: %s (status %d)" % (where, status_string(code), code))


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("bm", "bn", "bk", "stages", "cluster_m", "group_m", "split_k", "swap_ab", "grid")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class Epilogue(ctypes.Structure):
    """D = act(alpha * (A*B) + beta * C_in + bias), FP32 before the cast."""
    _fields_ = [("alpha", ctypes.c_float), ("beta", ctypes.c_float), ("c_in", ctypes.c_void_p),
                ("ldc_in", ctypes.c_int64), ("bias", ctypes.c_void_p), ("bias_dtype", ctypes.c_int),
                ("act", ctypes.c_int)]


_lock = threading.Lock()
_lib = None
_i64, _p, _i = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int


def load(path: str = LIB_PATH):
    """Load libtgemm.so (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError("libtgemm.so is not built (%s); run "
                               "dense_tiled_gemm_persistent_gb300.build.build()" % path)
        lib = ctypes.CDLL(path)
        run_args = [_i64, _i64, _i64, _p, _i64, _p, _i64, _i, _p, _i64, _i, _i, _p]
        lib.tgemm_run.argtypes = run_args
        lib.tgemm_run.restype = _i
        lib.tgemm_run_config.argtypes = run_args + [ctypes.POINTER(Config)]
        lib.tgemm_run_config.restype = _i
        lib.tgemm_query_config.argtypes = [_i64, _i64, _i64, _i, _i, _i, ctypes.POINTER(Config)]
        lib.tgemm_query_config.restype = _i
        lib.tgemm_check.argtypes = [_p]
        lib.tgemm_check.restype = _i
        lib.tgemm_last_fault_code.argtypes = []
        lib.tgemm_last_fault_code.restype = ctypes.c_uint32
        lib.tgemm_status_string.argtypes = [_i]
        lib.tgemm_status_string.restype = ctypes.c_char_p
        lib.tgemm_shutdown.argtypes = []
        lib.tgemm_shutdown.restype = None
        lib.tgemm_tile_coord.argtypes = [_i64, _i64, _i, _i, _i, _i64, ctypes.POINTER(_i64),
                                         ctypes.POINTER(_i64)]
        lib.tgemm_tile_coord.restype = _i
        lib.tgemm_run_ex.argtypes = run_args + [ctypes.POINTER(Epilogue), ctypes.POINTER(Config)]
        lib.tgemm_run_ex.restype = _i
        lib.tgemm_run_strided_batched.argtypes = [_i64, _i64, _i64, _i64, _p, _i64, _i64, _p, _i64, _i64, _i, _p,
                                                  _i64, _i64, _i, _i, _p, ctypes.POINTER(Epilogue),
                                                  ctypes.POINTER(Config)]
        lib.tgemm_run_strided_batched.restype = _i
        lib.tgemm_run_noalloc.argtypes = run_args
        lib.tgemm_run_noalloc.restype = _i
        lib.tgemm_debug_wait_timeout.argtypes = [ctypes.c_uint32, _p]
        lib.tgemm_debug_wait_timeout.restype = _i
        lib.tgemm_debug_noalloc_wait_timeout.argtypes = [ctypes.c_uint32, _p]
        lib.tgemm_debug_noalloc_wait_timeout.restype = _i
        lib.tgemm_debug_sm_clock.argtypes = [_p, ctypes.c_uint32, _p]
        lib.tgemm_debug_sm_clock.restype = _i
        lib.tgemm_debug_clock_record.argtypes = [_p]
        lib.tgemm_debug_clock_record.restype = _i
        lib.tgemm_debug_tile_order.argtypes = [_i64, _i64, _i, _i, _i, _p, _p, _p]
        lib.tgemm_debug_tile_order.restype = _i
        lib.tgemm_stream_k_plan.argtypes = [_i64, _i64, _i, _i, ctypes.POINTER(_i64), ctypes.POINTER(_i64),
                                            ctypes.POINTER(_i64)]
        lib.tgemm_stream_k_plan.restype = _i
        lib.tgemm_query_config_sms.argtypes = [_i64, _i64, _i64, _i, _i, _i, _i, ctypes.POINTER(Config)]
        lib.tgemm_query_config_sms.restype = _i
        lib.tgemm_group_size.argtypes = [_i64, _i64, _i64, _i, _i, _i, _i, _i, ctypes.POINTER(_i)]
        lib.tgemm_group_size.restype = _i
        _lib = lib
        return lib


# ---- raw C ABI ---------------------------------------------------------------

def tgemm_run(M, N, K, A, lda, B, ldb, b_layout, C, ldc, in_dtype, out_dtype, stream=None) -> int:
    return load().tgemm_run(M, N, K, A, lda, B, ldb, b_layout, C, ldc, in_dtype, out_dtype, stream)


def tgemm_run_ex(M, N, K, A, lda, B, ldb, b_layout, C, ldc, in_dtype, out_dtype, stream=None, ep=None,
                 cfg=None) -> int:
    """tgemm_run with a fused epilogue (Epilogue or None) and an optional Config."""
    return load().tgemm_run_ex(M, N, K, A, lda, B, ldb, b_layout, C, ldc, in_dtype, out_dtype, stream,
                               None if ep is None else ctypes.byref(ep), None if cfg is None else ctypes.byref(cfg))


def tgemm_run_strided_batched(batch, M, N, K, A, lda, stride_a, B, ldb, stride_b, b_layout, C, ldc, stride_c,
                              in_dtype, out_dtype, stream=None, ep=None, cfg=None) -> int:
    return load().tgemm_run_strided_batched(batch, M, N, K, A, lda, stride_a, B, ldb, stride_b, b_layout, C, ldc,
                                            stride_c, in_dtype, out_dtype, stream,
                                            None if ep is None else ctypes.byref(ep),
                                            None if cfg is None else ctypes.byref(cfg))


def tgemm_run_noalloc(M, N, K, A, lda, B, ldb, b_layout, C, ldc, in_dtype, out_dtype, stream=None) -> int:
    """tgemm_run for at most 64 rows of A without any device allocation (a
    fixed scratch array inside the library; calls that overlap on the GPU race)."""
    return load().tgemm_run_noalloc(M, N, K, A, lda, B, ldb, b_layout, C, ldc, in_dtype, out_dtype, stream)


def tgemm_run_config(M, N, K, A, lda, B, ldb, b_layout, C, ldc, in_dtype, out_dtype, stream,
                     cfg: Config) -> int:
    return load().tgemm_run_config(M, N, K, A, lda, B, ldb, b_layout, C, ldc, in_dtype, out_dtype,
                                   stream, ctypes.byref(cfg))


def tgemm_query_config(M, N, K, b_layout, in_dtype, out_dtype):
    cfg = Config()
    rc = load().tgemm_query_config(M, N, K, b_layout, in_dtype, out_dtype, ctypes.byref(cfg))
    return rc, cfg


def tgemm_query_config_sms(M, N, K, b_layout, in_dtype, out_dtype, sm_count):
    """(status, Config) tgemm_run would choose on a GPU with sm_count SMs (no device touched)."""
    cfg = Config()
    rc = load().tgemm_query_config_sms(M, N, K, b_layout, in_dtype, out_dtype, sm_count, ctypes.byref(cfg))
    return rc, cfg


def tgemm_check(stream=None) -> int:
    return load().tgemm_check(stream)


def tgemm_last_fault_code() -> int:
    return load().tgemm_last_fault_code()


def status_string(code: int) -> str:
    return load().tgemm_status_string(code).decode()


def tgemm_shutdown() -> None:
    load().tgemm_shutdown()


def tgemm_tile_coord(M, N, bm, bn, group_m, bid):
    r, c = _i64(), _i64()
    rc = load().tgemm_tile_coord(M, N, bm, bn, group_m, bid, ctypes.byref(r), ctypes.byref(c))
    return rc, r.value, c.value


def tgemm_group_size(M, N, K, bm, unit_bn, in_dtype, out_dtype, resident):
    """(status, group_m) the library picks for a single problem on the tile kernels."""
    g = _i()
    rc = load().tgemm_group_size(M, N, K, bm, unit_bn, in_dtype, out_dtype, resident, ctypes.byref(g))
    return rc, g.value


def tgemm_stream_k_plan(items, k_blocks, units, tiles_per_item=1):
    """(status, whole items, shared items, sharing units) of a stream-K launch."""
    dp, sk, u = _i64(), _i64(), _i64()
    rc = load().tgemm_stream_k_plan(items, k_blocks, units, tiles_per_item, ctypes.byref(dp), ctypes.byref(sk),
                                    ctypes.byref(u))
    return rc, dp.value, sk.value, u.value


def tgemm_debug_wait_timeout(timeout_us: int, stream=None) -> int:
    return load().tgemm_debug_wait_timeout(timeout_us, stream)


def tgemm_debug_noalloc_wait_timeout(timeout_us: int, stream=None) -> int:
    return load().tgemm_debug_noalloc_wait_timeout(timeout_us, stream)


def tgemm_debug_sm_clock(out, duration_us: int, stream=None) -> int:
    """out: device address of two uint64 (elapsed ns, SM cycles)."""
    return load().tgemm_debug_sm_clock(out, duration_us, stream)


def tgemm_debug_clock_record(rec) -> int:
    """rec: device address of eight uint64 (rec[0..2] zeroed), or None to stop."""
    return load().tgemm_debug_clock_record(rec)


def tgemm_debug_tile_order(M, N, bm, bn, group_m, rows, cols, stream=None) -> int:
    """The scheduler's tile order computed on the GPU into two int32 device
    arrays (pointers) of ceil(M/bm) * ceil(N/bn) elements."""
    return load().tgemm_debug_tile_order(M, N, bm, bn, group_m, rows, cols, stream)


# ---- torch convenience ------------------------------------------------------

def _dtype_code(t):
    import torch
    return {torch.float16: F16, torch.bfloat16: BF16, torch.float32: F32,
            torch.float8_e4m3fn: E4M3, torch.float8_e5m2: E5M2}[t]


def _ld(t) -> int:
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("operands must be 2-D with unit column stride (row-major)")
    return t.stride(0) if t.shape[0] > 1 else max(t.stride(0), t.shape[1])


def _stream_handle(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def matmul(A, B, b_layout: int = B_NK, out_dtype=None, C=None, stream=None, config: Config = None):
    """C = A @ B on the GPU through tgemm_run (or tgemm_run_config).

    A: (M, K) row-major CUDA tensor, FP16, BF16, FP8 (float8_e4m3fn,
    float8_e5m2) or FP32 (multiplied as TF32).  B: (K, N) for B_KN or (N, K)
    for B_NK, same dtype (FP8 and FP32: B_NK only).  C: optional (M, N) output (allocated with torch.empty when
    omitted, dtype out_dtype, else BF16 for FP8 inputs and A.dtype otherwise).
    """
    import torch
    if not (A.is_cuda and B.is_cuda):
        raise ValueError("operands must be CUDA tensors")
    if A.dtype != B.dtype:
        raise ValueError("A and B must have the same dtype")
    M, K = A.shape
    N = B.shape[1] if b_layout == B_KN else B.shape[0]
    kb = B.shape[0] if b_layout == B_KN else B.shape[1]
    if kb != K:
        raise ValueError("inner dimensions differ")
    if C is None:
        default = torch.bfloat16 if A.element_size() == 1 else A.dtype
        C = torch.empty((M, N), dtype=out_dtype or default, device=A.device)
    args = (M, N, K, A.data_ptr(), _ld(A), B.data_ptr(), _ld(B), b_layout, C.data_ptr(), _ld(C),
            _dtype_code(A.dtype), _dtype_code(C.dtype), _stream_handle(stream))
    rc = tgemm_run(*args) if config is None else tgemm_run_config(*args, config)
    if rc != OK:
        raise TgemmError(rc, "tgemm_run")
    return C
