"""tgemm_run_noalloc: the skinny GEMM without device allocation.

Callers whose device memory is owned by a pool or a fixed budget cannot let
the library cudaMalloc a workspace behind their back; tgemm_run_noalloc
serves them from a scratch array built into the library.  These tests call it
through the C ABI and check that it gives what tgemm_run gives, within the
acceptance bound the other tests use (1e-3 * sum|A||B| + one unit in the last
place of the output type), on two calls in a row -- the second call finds
the scratch array holding the first call's leftovers.

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


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


CASES = [
    # M, N, K, layout, in, out
    (16, 4096, 4096, gen.B_NK, gen.BF16, gen.BF16),   # the 16-token projection shape
    (5, 300, 1000, gen.B_KN, gen.F16, gen.F32),
    (64, 1000, 2048, gen.B_NK, gen.F16, gen.F16),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "%dx%dx%d" % c[:3])
def test_noalloc_matches_tgemm_run_on_two_calls(case):
    M, N, K, layout, ind, outd = case
    a, b = operands(M, N, K, ind, layout, gen.normal(0, 1), seed=M * 7 + N, dist_b=gen.normal(0, 0.02))
    A, B = a.to("cuda:0"), b.to("cuda:0")
    ldc = -(-N // 8) * 8
    tdt = gen.TORCH_DTYPE[outd]
    C_run = torch.empty((M, ldc), dtype=tdt, device="cuda:0")
    args = (M, N, K, A.data_ptr(), A.shape[1], B.data_ptr(), B.shape[1], layout)
    assert tgemm.tgemm_run(*args, C_run.data_ptr(), ldc, ind, outd, None) == 0
    assert tgemm.tgemm_check() == 0
    ref, bound = oracle.gemm(a, b, M, N, K, a.shape[1], b.shape[1], layout, ind)
    want = C_run[:, :N].double().cpu().numpy()
    tol = 1e-3 * bound + oracle.ulp(want, outd)
    for call in range(2):
        C = torch.full((M, ldc), float("nan"), dtype=tdt, device="cuda:0")
        assert tgemm.tgemm_run_noalloc(*args, C.data_ptr(), ldc, ind, outd, None) == 0
        torch.cuda.synchronize()
        assert tgemm.tgemm_check() == 0
        got = C[:, :N].double().cpu().numpy()
        bad = ~(np.abs(got - want) <= tol)
        assert not bad.any(), "call %d: %d elements differ from tgemm_run" % (call, bad.sum())


def test_noalloc_rejects_sizes_beyond_its_limits():
    x = torch.empty(64, dtype=torch.float16, device="cuda:0")
    p = x.data_ptr()
    # more than 64 rows of A
    assert tgemm.tgemm_run_noalloc(65, 128, 64, p, 64, p, 64, gen.B_NK, p, 128, gen.F16, gen.F16, None) \
        == tgemm.ERR_UNSUPPORTED
    # more than 4096 column tiles of 128
    assert tgemm.tgemm_run_noalloc(16, 4096 * 128 + 1, 64, p, 64, p, 64, gen.B_NK, p, 4096 * 128 + 8, gen.F16,
                                   gen.F16, None) == tgemm.ERR_UNSUPPORTED
