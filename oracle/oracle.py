"""ctypes front end of the plain-C FP64 oracle (tgemm_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, the package smoke entry and the
benchmark's CPU-baseline leg, never by the product path.  It shares no code
with the CUDA library.

Inputs are bit patterns: numpy uint16 (FP16/BF16), uint8 (FP8) or uint32
(FP32 storage read as TF32) arrays, or torch tensors of those dtypes; outputs
are float64 numpy arrays.  Each wrapper states the passage it follows
in the C file's header: the defining sum C[i][j] = sum_k A[i][k] B[k][j] from
"Writing high-performance matrix multiplication with NVIDIA CUDA Tile"
(juejin.cn, "What is matrix multiplication?").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F16, BF16, F32, E4M3, E5M2, TF32 = 0, 1, 2, 3, 4, 5
B_KN, B_NK = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tgemm_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_p = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile tgemm_oracle.c with gcc into oracle/_build/liboracle.so."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if stale:
        tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lpthread", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # A test may point the wrapper at a deliberately broken build of the
            # same source to show that the pins catch the mistake.
            override = os.environ.get("TGEMM_ORACLE_LIB")
            lib = ctypes.CDLL(override if override else build())
            lib.oracle_gemm_rows.argtypes = [_i64, _i64, _i64, _p, _i64, _p, _i64, ctypes.c_int,
                                             ctypes.c_int, _i64, _i64, _p, _i64, _p, _i64, ctypes.c_int]
            lib.oracle_gemm_rows.restype = ctypes.c_int
            lib.oracle_gemm_elements.argtypes = [_i64, _i64, _i64, _p, _i64, _p, _i64, ctypes.c_int,
                                                 ctypes.c_int, _i64, _p, _p, _p, _p, ctypes.c_int]
            lib.oracle_gemm_elements.restype = ctypes.c_int
            lib.oracle_round_bits_n.argtypes = [_p, _i64, ctypes.c_int, _p]
            lib.oracle_ulp_n.argtypes = [_p, _i64, ctypes.c_int, _p]
            lib.oracle_decode_n.argtypes = [_p, _i64, ctypes.c_int, _p]
            lib.oracle_epilogue.argtypes = [_i64, _i64, _p, _i64, ctypes.c_double, ctypes.c_double, _p, _i64,
                                            _p, ctypes.c_int]
            lib.oracle_epilogue.restype = None
            _lib = lib
    return _lib


def _u16(x) -> np.ndarray:
    """An input pattern array: numpy uint16/int16/uint8/uint32/float32, or a
    torch tensor (FP16/BF16 -> 16-bit patterns, FP8 -> 8-bit patterns, FP32
    -> 32-bit patterns)."""
    if hasattr(x, "detach"):  # torch tensor: reinterpret its bits
        import torch
        t = x.detach().cpu().contiguous()
        if t.element_size() == 1:
            return np.ascontiguousarray(t.view(torch.uint8).numpy())
        if t.element_size() == 4:
            return np.ascontiguousarray(t.view(torch.int32).numpy().view(np.uint32))
        x = t.view(torch.int16).numpy()
    x = np.ascontiguousarray(x)
    if x.dtype in (np.uint8, np.uint32):
        return x
    if x.dtype in (np.float32, np.int32):
        return x.view(np.uint32)
    if x.dtype != np.uint16:
        x = x.view(np.uint16)
    return x


def _default_threads() -> int:
    return os.cpu_count() or 1


def gemm_rows(A, B, M, N, K, lda, ldb, b_layout, in_dtype, row_begin, row_end,
              with_bound=True, threads=None):
    """Rows [row_begin, row_end) of C and of sum_k |A_ik||B_kj|, float64.

    A holds M x lda patterns (row-major), B holds K x ldb (KN) or N x ldb (NK).
    Returns (C, bound) with shape (row_end - row_begin, N); bound is None when
    with_bound is False.
    """
    lib = _load()
    a, b = _u16(A), _u16(B)
    rows = row_end - row_begin
    C = np.zeros((max(rows, 0), max(N, 1)), dtype=np.float64)
    Bd = np.zeros_like(C) if with_bound else None
    ldc = max(N, 1)
    c_ptr = C.ctypes.data
    b_ptr = Bd.ctypes.data if with_bound else None
    rc = lib.oracle_gemm_rows(M, N, K, a.ctypes.data, lda, b.ctypes.data, ldb, b_layout, in_dtype,
                              row_begin, row_end, c_ptr, ldc, b_ptr, ldc,
                              threads or _default_threads())
    if rc != 0:
        raise ValueError("oracle_gemm_rows: bad arguments")
    C = C[:, :N]
    return C, (Bd[:, :N] if with_bound else None)


def gemm(A, B, M, N, K, lda, ldb, b_layout, in_dtype, threads=None):
    """The full product C (M x N, float64) and the bound sum_k |A_ik||B_kj|."""
    return gemm_rows(A, B, M, N, K, lda, ldb, b_layout, in_dtype, 0, M, True, threads)


def gemm_elements(A, B, M, N, K, lda, ldb, b_layout, in_dtype, ii, jj, threads=None):
    """C[ii[t], jj[t]] and its bound for each t, float64."""
    lib = _load()
    a, b = _u16(A), _u16(B)
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    out = np.zeros(len(ii), dtype=np.float64)
    bound = np.zeros(len(ii), dtype=np.float64)
    rc = lib.oracle_gemm_elements(M, N, K, a.ctypes.data, lda, b.ctypes.data, ldb, b_layout,
                                  in_dtype, len(ii), ii.ctypes.data, jj.ctypes.data,
                                  out.ctypes.data, bound.ctypes.data, threads or _default_threads())
    if rc != 0:
        raise ValueError("oracle_gemm_elements: bad arguments")
    return out, bound


def round_bits(x, dtype) -> np.ndarray:
    """Round-to-nearest-even of float64 values into the output format's bits."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.uint32)
    lib.oracle_round_bits_n(x.ctypes.data, x.size, dtype, out.ctypes.data)
    return out


def ulp(x, dtype) -> np.ndarray:
    """Spacing of the output format at |x| (subnormal spacing near zero)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.float64)
    lib.oracle_ulp_n(x.ctypes.data, x.size, dtype, out.ctypes.data)
    return out


ACT_NONE, ACT_RELU, ACT_GELU_TANH = 0, 1, 2


def epilogue(C, alpha=1.0, beta=0.0, cin=None, bias=None, act=ACT_NONE) -> np.ndarray:
    """act(alpha * C + beta * cin + bias[None, :]) in float64 (a new array).

    C and cin are float64 (rows x cols); bias float64 (cols,) or None."""
    lib = _load()
    D = np.ascontiguousarray(C, dtype=np.float64).copy()
    rows, cols = D.shape
    cin_a = None if cin is None else np.ascontiguousarray(cin, dtype=np.float64)
    bias_a = None if bias is None else np.ascontiguousarray(bias, dtype=np.float64)
    lib.oracle_epilogue(rows, cols, D.ctypes.data, cols, float(alpha), float(beta),
                        None if cin_a is None else cin_a.ctypes.data, cols,
                        None if bias_a is None else bias_a.ctypes.data, act)
    return D


def decode(bits, dtype) -> np.ndarray:
    """Value of 16-bit (F16/BF16), 8-bit (E4M3/E5M2) or 32-bit (F32, or TF32:
    the FP32 pattern with its low 13 fraction bits dropped) patterns as float64."""
    lib = _load()
    b = np.ascontiguousarray(bits, dtype=np.uint32)
    out = np.zeros(b.shape, dtype=np.float64)
    lib.oracle_decode_n(b.ctypes.data, b.size, dtype, out.ctypes.data)
    return out
