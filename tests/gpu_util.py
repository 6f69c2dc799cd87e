"""Helpers shared by the GPU parity tests (not collected by pytest).

The acceptance bound for every floating-point element is
    |C_gpu - C_ref| <= 1e-3 * sum_k |A_ik||B_kj| + ulp_out(C_ref)
with C_ref and the bound from the FP64 oracle and ulp_out the spacing of the
output format at C_ref.  Integer-valued cases compare bit patterns with the
oracle's round-to-nearest-even of the exact result.  An infinite GPU element
passes the tolerance check only where a value within the bound, on the far
side of the oracle's value from zero, rounds to the same infinity in the
output format (the cast overflows to +-Inf under round-to-nearest-even).
"""
import numpy as np
import torch

import oracle
from dense_tiled_gemm_persistent_gb300 import build as libbuild
from dense_tiled_gemm_persistent_gb300 import inputs as gen
from dense_tiled_gemm_persistent_gb300 import tgemm

TOL_REL = 1e-3
DEV = "cuda:0"


def ensure_built():
    libbuild.build()
    tgemm.load()


def round_up(x, m):
    return -(-x // m) * m


def operands(M, N, K, in_dtype, layout, dist, seed, dist_b=None):
    """Seeded operands with leading dimensions rounded up to 8 elements (the
    16-byte row rule), the pad poisoned with NaN."""
    b_cols = N if layout == gen.B_KN else K
    return gen.make_operands(M, N, K, in_dtype, layout, dist, dist_b, seed,
                             lda=round_up(max(K, 1), 8), ldb=round_up(max(b_cols, 1), 8),
                             pad_value=float("nan"))


def run_gpu(a, b, M, N, K, layout, in_dtype, out_dtype, ldc=None, c_fill=None, config=None, stream=None):
    """Copy seeded CPU operands to the GPU, run tgemm through the C ABI, and
    return C's storage (M x ldc) back on the CPU."""
    A, B = a.to(DEV), b.to(DEV)
    ldc = round_up(max(N, 1), 16 // gen.DTYPE_SIZE[out_dtype]) if ldc is None else ldc
    C = torch.empty((max(M, 1), max(ldc, 1)), dtype=gen.TORCH_DTYPE[out_dtype], device=DEV)
    if c_fill is not None:
        C.fill_(c_fill)
    args = (M, N, K, A.data_ptr(), a.shape[1], B.data_ptr(), b.shape[1], layout, C.data_ptr(), ldc,
            in_dtype, out_dtype, None if stream is None else tgemm.ctypes.c_void_p(stream.cuda_stream))
    rc = tgemm.tgemm_run(*args) if config is None else tgemm.tgemm_run_config(*args, config)
    assert rc == tgemm.OK, tgemm.status_string(rc)
    rc = tgemm.tgemm_check(args[-1])
    assert rc == tgemm.OK, tgemm.status_string(rc)
    return C.cpu()


def values(C_cpu, out_dtype):
    return C_cpu.double().numpy()


def bits(C_cpu, out_dtype):
    if out_dtype == gen.F32:
        return C_cpu.view(torch.int32).numpy().view(np.uint32)
    return C_cpu.view(torch.int16).numpy().view(np.uint16).astype(np.uint32)


def overflow_ok(got, ref, tol, out_dtype):
    """Where the GPU wrote +-Inf: right when a value within the tolerance of
    the oracle's, on the far side from zero, rounds (RNE) to that same
    infinity in the output format."""
    with np.errstate(invalid="ignore"):
        far = ref + np.sign(ref) * tol
    edge = oracle.decode(oracle.round_bits(far, out_dtype), out_dtype)
    return np.isinf(got) & np.isinf(edge) & (np.sign(got) == np.sign(edge))


def assert_close(got, ref, bound, out_dtype, what=""):
    tol = TOL_REL * bound + oracle.ulp(ref, out_dtype)
    with np.errstate(invalid="ignore"):
        err = np.abs(got - ref)
    bad = ~((err <= tol) | overflow_ok(got, ref, tol, out_dtype))     # NaN counts as bad
    if bad.any():
        idx = np.argwhere(bad)
        i = tuple(idx[0])
        raise AssertionError("%s: %d of %d elements outside the bound; first at %s: got %r, "
                             "oracle %r, bound %r" % (what, bad.sum(), bad.size, i, got[i], ref[i], tol[i]))
    fin = np.isfinite(err)
    return float(np.max(err[fin] / np.maximum(bound[fin], 1e-300))) if fin.any() else 0.0


def check_full(a, b, M, N, K, layout, in_dtype, out_dtype, exact=False, config=None, what=""):
    C = run_gpu(a, b, M, N, K, layout, in_dtype, out_dtype, config=config)
    ref, bound = oracle.gemm(a, b, M, N, K, a.shape[1], b.shape[1], layout, in_dtype)
    if exact:
        want = oracle.round_bits(ref, out_dtype)
        got = bits(C[:M, :N], out_dtype)
        mism = got != want
        assert not mism.any(), "%s: %d bit mismatches, first at %s" % (
            what, mism.sum(), tuple(np.argwhere(mism)[0]))
        return 0.0
    return assert_close(values(C[:M, :N], out_dtype), ref, bound, out_dtype, what)


def boundary_indices(extent, tile, extra=()):
    """Rows/columns at tile boundaries: 0, tile-1, tile, 2*tile-1, 2*tile,
    the first index of the last (possibly partial) tile, and the last."""
    cand = {0, tile - 1, tile, 2 * tile - 1, 2 * tile, ((extent - 1) // tile) * tile, extent - 1}
    cand |= set(extra)
    return sorted(i for i in cand if 0 <= i < extent)


def sampled_points(M, N, seed, n_random=4096, row_tile=128, col_tiles=(64, 128, 256)):
    rng = np.random.default_rng(seed)
    ii = [rng.integers(0, M, n_random)]
    jj = [rng.integers(0, N, n_random)]
    for r in boundary_indices(M, row_tile):
        ii.append(np.full(N, r))
        jj.append(np.arange(N))
    cols = set()
    for t in col_tiles:
        cols |= set(boundary_indices(N, t))
    for c in sorted(cols):
        ii.append(np.arange(M))
        jj.append(np.full(M, c))
    return np.concatenate(ii).astype(np.int64), np.concatenate(jj).astype(np.int64)
