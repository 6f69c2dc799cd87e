"""tgemm_run_noalloc: the skinny GEMM without device allocation.

Callers whose device memory is owned by a pool or a fixed budget cannot let
the library cudaMalloc a workspace behind their back; tgemm_run_noalloc
serves them from a scratch array built into the library.  These tests call it
through the C ABI and check it against the FP64 oracle within the acceptance
bound the other tests use (1e-3 * sum|A||B| + one unit in the last place of
the output type at the oracle's value), on two calls in a row -- the second
call finds the scratch array holding the first call's leftovers -- and, as a
second check, against tgemm_run.

The cases reach every branch of the entry point's split choice: the natural
split count, the count capped by what the array's partial-sum region holds,
no room at all (one split, C written directly), and K = 0 (the empty sum).

This file is collected last so that a failing run stopped at the first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
from dense_tiled_gemm_persistent_gb300 import inputs as gen
from dense_tiled_gemm_persistent_gb300 import tgemm

from gpu_util import ensure_built, operands

pytestmark = pytest.mark.gpu

# Sizes of the built-in array's regions (tgemm_noalloc.cu): 4 MiB in all,
# a 256-byte head, 16 KiB of counters, the rest FP32 partial sums.
PARTIAL_BYTES = (4 << 20) - 256 - (16 << 10)


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def splits_that_fit(M, N):
    npad = 16 if M <= 16 else (32 if M <= 32 else 64)
    return PARTIAL_BYTES // (-(-N // 128) * 128 * npad * 4)


CASES = [
    # M, N, K, layout, in, out
    (16, 4096, 4096, gen.B_NK, gen.BF16, gen.BF16),   # the 16-token projection shape: natural split count
    (5, 300, 1000, gen.B_KN, gen.F16, gen.F32),
    (64, 1000, 2048, gen.B_NK, gen.F16, gen.F16),     # 15 splits fit, fewer than the natural count
    (64, 20000, 512, gen.B_NK, gen.BF16, gen.F32),    # no split fits: one split writes C directly
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "%dx%dx%d" % c[:3])
def test_noalloc_matches_the_oracle_on_two_calls(case):
    M, N, K, layout, ind, outd = case
    if (M, N) == (64, 1000):
        assert 1 <= splits_that_fit(M, N) < 2 * 152 // 8
    if (M, N) == (64, 20000):
        assert splits_that_fit(M, N) == 0
    a, b = operands(M, N, K, ind, layout, gen.normal(0, 1), seed=M * 7 + N, dist_b=gen.normal(0, 0.02))
    A, B = a.to("cuda:0"), b.to("cuda:0")
    ldc = -(-N // 8) * 8
    tdt = gen.TORCH_DTYPE[outd]
    args = (M, N, K, A.data_ptr(), A.shape[1], B.data_ptr(), B.shape[1], layout)
    ref, bound = oracle.gemm(a, b, M, N, K, a.shape[1], b.shape[1], layout, ind)
    tol = 1e-3 * bound + oracle.ulp(ref, outd)
    C_run = torch.empty((M, ldc), dtype=tdt, device="cuda:0")
    assert tgemm.tgemm_run(*args, C_run.data_ptr(), ldc, ind, outd, None) == 0
    assert tgemm.tgemm_check() == 0
    run = C_run[:, :N].double().cpu().numpy()
    for call in range(2):
        C = torch.full((M, ldc), float("nan"), dtype=tdt, device="cuda:0")
        assert tgemm.tgemm_run_noalloc(*args, C.data_ptr(), ldc, ind, outd, None) == 0
        torch.cuda.synchronize()
        assert tgemm.tgemm_check() == 0
        got = C[:, :N].double().cpu().numpy()
        bad = ~(np.abs(got - ref) <= tol)
        assert not bad.any(), "call %d: %d elements outside the bound, first at %s" % (
            call, bad.sum(), tuple(np.argwhere(bad)[0]))
        # and the same result as tgemm_run's kernel, within the same bound
        assert np.all(np.abs(got - run) <= tol + oracle.ulp(run, outd)), "call %d: differs from tgemm_run" % call


def test_noalloc_empty_sum_writes_zeros_and_leaves_the_padding():
    M, N, ldc = 40, 100, 128
    C = torch.full((M, ldc), 5.0, dtype=torch.float16, device="cuda:0")
    x = torch.empty(64, dtype=torch.float16, device="cuda:0")
    for _ in range(2):
        assert tgemm.tgemm_run_noalloc(M, N, 0, x.data_ptr(), 8, x.data_ptr(), 8, gen.B_NK, C.data_ptr(), ldc,
                                       gen.F16, gen.F16, None) == 0
        assert tgemm.tgemm_check() == 0
        c = C.cpu()
        assert torch.count_nonzero(c[:, :N]).item() == 0      # the empty sum
        assert torch.all(c[:, N:] == 5.0)                      # columns beyond N untouched


def test_noalloc_timeout_is_reported_by_check_and_the_next_call_is_right():
    """A wait that gives up records its fault in the status word kept in the
    built-in array; tgemm_check reports TGEMM_ERR_TIMEOUT once and clears it,
    and the next allocation-free call is correct."""
    assert tgemm.tgemm_check() == 0
    assert tgemm.tgemm_debug_noalloc_wait_timeout(1000) == 0
    assert tgemm.tgemm_check() == tgemm.ERR_TIMEOUT
    assert tgemm.tgemm_last_fault_code() >> 28 == 7
    assert tgemm.tgemm_check() == 0
    M, N, K = 16, 512, 1024
    a, b = operands(M, N, K, gen.BF16, gen.B_NK, gen.ints(-2, 2), seed=3)
    A, B = a.to("cuda:0"), b.to("cuda:0")
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda:0")
    assert tgemm.tgemm_run_noalloc(M, N, K, A.data_ptr(), A.shape[1], B.data_ptr(), B.shape[1], gen.B_NK,
                                   C.data_ptr(), N, gen.BF16, gen.F32, None) == 0
    assert tgemm.tgemm_check() == 0
    ref, _ = oracle.gemm(a, b, M, N, K, a.shape[1], b.shape[1], gen.B_NK, gen.BF16)
    assert np.array_equal(C.cpu().double().numpy(), ref)       # small integers: exact


def test_noalloc_rejects_sizes_beyond_its_limits():
    x = torch.empty(64, dtype=torch.float16, device="cuda:0")
    p = x.data_ptr()
    # more than 64 rows of A
    assert tgemm.tgemm_run_noalloc(65, 128, 64, p, 64, p, 64, gen.B_NK, p, 128, gen.F16, gen.F16, None) \
        == tgemm.ERR_UNSUPPORTED
    # more than 4096 column tiles of 128
    assert tgemm.tgemm_run_noalloc(16, 4096 * 128 + 1, 64, p, 64, p, 64, gen.B_NK, p, 4096 * 128 + 8, gen.F16,
                                   gen.F16, None) == tgemm.ERR_UNSUPPORTED
    assert tgemm.tgemm_debug_noalloc_wait_timeout(0) == tgemm.ERR_INVALID_ARG
