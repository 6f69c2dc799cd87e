"""Host-side tests of the stream-K plan (no GPU needed).

The pair and quad kernels deal the last one or two waves of work items out
by k-block iterations instead of whole items: unit u of U takes iterations
[u*I//U, (u+1)*I//U) of the I shared ones.  These tests check the plan the
library computes (tgemm_stream_k_plan, the same function tgemm_run uses)
against that definition and against the rules the kernels rely on, over a
grid of shapes, and pin the plans of the measured workloads.
"""
import pytest

from dense_tiled_gemm_persistent_gb300 import build as libbuild
from dense_tiled_gemm_persistent_gb300 import tgemm

MAX_SEGMENTS = 3      # items one unit's share may touch (workspace slots per unit)
MIN_ITERS = 8         # smallest share worth a partial-sum hand-off
COUNTERS = 16384      # arrival counters in the workspace (two per tile)


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return tgemm.load()


def shares(sk_items, k_blocks, units):
    total = sk_items * k_blocks
    return [(u * total // units, (u + 1) * total // units) for u in range(units)]


def check_plan(T, KB, P, tpi):
    rc, dp, sk, units = tgemm.tgemm_stream_k_plan(T, KB, P, tpi)
    assert rc == 0
    if units == 0:
        assert (dp, sk) == (T, 0)
        return dp, sk, units
    assert dp + sk == T and dp % P == 0 and 2 <= units <= P
    assert 2 * tpi * sk <= COUNTERS
    full, rem = divmod(T, P)
    if full >= 1 and 2 * rem <= P:
        # leftover wave at most half full: every full wave stays whole
        assert dp == full * P and sk == rem
    else:
        # otherwise the last full wave is shared as well (the pair), or every
        # item when there are fewer items than units
        assert (tpi == 1 or full == 0) and dp == max(full - 1, 0) * P
    sh = shares(sk, KB, units)
    assert sh[0][0] == 0 and sh[-1][1] == sk * KB
    assert all(a[1] == b[0] for a, b in zip(sh, sh[1:]))              # contiguous: each iteration once
    lens = [b - a for a, b in sh]
    assert min(lens) >= MIN_ITERS and max(lens) - min(lens) <= 1        # equal shares, none too small
    for a, b in sh:
        assert (b - 1) // KB - a // KB + 1 <= MAX_SEGMENTS             # items one unit touches
    # never slower than whole items: the busiest unit's iterations
    busiest = (dp // P) * KB + max(lens)
    assert busiest <= -(-T // P) * KB
    return dp, sk, units


@pytest.mark.parametrize("tpi", [1, 2], ids=["pair", "quad"])
@pytest.mark.parametrize("P", [1, 2, 3, 7, 36, 38, 76])
def test_plans_follow_the_definition(lib, tpi, P):
    for T in list(range(1, 200)) + [255, 256, 257, 512, 1023, 1024, 1025, 7168]:
        for KB in (1, 4, 7, 8, 16, 40, 64, 79, 128, 256):
            check_plan(T, KB, P, tpi)


def test_plans_of_the_measured_workloads(lib):
    # 8192^3 on 76 CTA pairs: 1024 tiles of 128 k-blocks; 13 whole waves, the
    # 36 leftover tiles each cut in two
    assert tgemm.tgemm_stream_k_plan(1024, 128, 76, 1)[1:] == (988, 36, 72)
    # 4096^3: 256 tiles of 64 k-blocks, 28 left over, two units each
    assert tgemm.tgemm_stream_k_plan(256, 64, 76, 1)[1:] == (228, 28, 56)
    # 4000 x 3000 x 5000 on 36 quads: 96 blocks, the leftover wave two thirds
    # full, so whole blocks
    assert tgemm.tgemm_stream_k_plan(96, 79, 36, 2)[1:] == (96, 0, 0)
    # 2000 x 3000 x 5000 on 36 quads: 48 blocks, the 12 left over in thirds
    assert tgemm.tgemm_stream_k_plan(48, 79, 36, 2)[1:] == (36, 12, 36)
    # fewer blocks than quads: all of them shared
    assert tgemm.tgemm_stream_k_plan(15, 24, 36, 2)[1:] == (0, 15, 36)
    # shallow K: shares below MIN_ITERS are not worth the hand-off
    assert tgemm.tgemm_stream_k_plan(4, 2, 36, 2)[1:] == (4, 0, 0)
    # whole waves need no tail
    assert tgemm.tgemm_stream_k_plan(152, 64, 76, 1)[1:] == (152, 0, 0)


def test_plan_rejects_bad_arguments(lib):
    assert tgemm.tgemm_stream_k_plan(-1, 8, 4, 1)[0] == tgemm.ERR_INVALID_ARG
    assert tgemm.tgemm_stream_k_plan(10, 0, 4, 1)[0] == tgemm.ERR_INVALID_ARG
    assert tgemm.tgemm_stream_k_plan(10, 8, 0, 1)[0] == tgemm.ERR_INVALID_ARG
    assert tgemm.tgemm_stream_k_plan(10, 8, 4, 3)[0] == tgemm.ERR_INVALID_ARG
    assert tgemm.tgemm_stream_k_plan(0, 8, 4, 1)[1:] == (0, 0, 0)
