"""GPU parity: the tcgen05 kernels against the FP64 CPU oracle, element by
element, through the C ABI.

Sizes span several tiles and ragged tails in M, N and K (the tail rules of
the CUDA Programming Guide 13.4.2, section 2.4.9.1: zero-padded partial K
tile, out-of-range M/N elements dropped at the store).
"""
import numpy as np
import pytest
import torch

import oracle
from dense_tiled_gemm_persistent_gb300 import inputs as gen
from dense_tiled_gemm_persistent_gb300 import tgemm

from gpu_util import check_full, ensure_built, run_gpu, bits, values, assert_close, operands

pytestmark = pytest.mark.gpu

LAYOUTS = [gen.B_NK, gen.B_KN]
LNAME = {gen.B_NK: "nk", gen.B_KN: "kn"}
DEV_ = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def cfg(bn, stages=None, group_m=8, grid=0, pair=False, quad=False):
    if pair or quad:
        return tgemm.Config(bm=256, bn=256, bk=64, stages=stages or 6, cluster_m=4 if quad else 2, group_m=group_m,
                            split_k=1, swap_ab=0, grid=grid)
    return tgemm.Config(bm=128, bn=bn, bk=64, stages=stages or (4 if bn == 256 else 6), cluster_m=1,
                        group_m=group_m, split_k=1, swap_ab=0, grid=grid)


# every compiled tile shape: 128 x 256 and 128 x 128 on one CTA, 256 x 256 on a CTA pair, and two
# 256 x 256 pairs sharing A in a cluster of four
SHAPE_CFGS = [("1cta_128x256", dict(bn=256)), ("1cta_128x128", dict(bn=128)),
              ("1cta_128x128_2stage", dict(bn=128, stages=2)), ("pair_256x256", dict(bn=256, pair=True)),
              ("quad_256x512", dict(bn=256, quad=True))]


# ---- one tile, exact integers: descriptor and layout sanity ------------------

@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("name,kw", SHAPE_CFGS, ids=[n for n, _ in SHAPE_CFGS])
def test_one_tile_integers_exact(layout, name, kw):
    M, N, K = (256 if kw.get("pair") or kw.get("quad") else 128), kw["bn"], 64
    a, b = operands(M, N, K, gen.F16, layout, gen.ints(-2, 2), seed=1)
    check_full(a, b, M, N, K, layout, gen.F16, gen.F32, exact=True, config=cfg(**kw),
               what="one tile %s %s" % (LNAME[layout], name))


@pytest.mark.parametrize("layout", LAYOUTS)
def test_one_hot_products_land_in_place(layout):
    """A single 1 in A at (i, k) and in B at (k, j): C is zero except C[i, j] = 1."""
    M, N, K = 256, 512, 192
    rng = np.random.default_rng(3)
    for _ in range(4):
        i, k, j = int(rng.integers(M)), int(rng.integers(K)), int(rng.integers(N))
        a = torch.zeros(M, K, dtype=torch.bfloat16)
        a[i, k] = 1
        b = torch.zeros((K, N) if layout == gen.B_KN else (N, K), dtype=torch.bfloat16)
        if layout == gen.B_KN:
            b[k, j] = 1
        else:
            b[j, k] = 1
        C = run_gpu(a, b, M, N, K, layout, gen.BF16, gen.F32)
        v = values(C, gen.F32)
        want = np.zeros((M, N))
        want[i, j] = 1
        assert np.array_equal(v, want), "one-hot (%d,%d,%d) misplaced: nonzeros at %s" % (
            i, k, j, np.argwhere(v != 0)[:4].tolist())


# ---- full comparisons over shapes, layouts, dtypes and tile widths --------------

SHAPES = [(256, 256, 256), (300, 520, 200), (129, 257, 65), (1, 1, 1), (640, 384, 1000), (17, 700, 130)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("layout", LAYOUTS, ids=["nk", "kn"])
@pytest.mark.parametrize("in_dtype", [gen.F16, gen.BF16], ids=["f16", "bf16"])
@pytest.mark.parametrize("out_dtype", [gen.F32, gen.F16, gen.BF16], ids=["o32", "o16", "obf16"])
def test_full_compare(shape, layout, in_dtype, out_dtype):
    M, N, K = shape
    seed = hash((M, N, K, layout, in_dtype, out_dtype)) % 1000
    a, b = operands(M, N, K, in_dtype, layout, gen.normal(0, 1), seed=seed)
    for name, kw in SHAPE_CFGS:
        check_full(a, b, M, N, K, layout, in_dtype, out_dtype, config=cfg(**kw),
                   what="%s %s %s" % (shape, LNAME[layout], name))


@pytest.mark.parametrize("layout", LAYOUTS, ids=["nk", "kn"])
@pytest.mark.parametrize("out_dtype", [gen.F32, gen.F16, gen.BF16], ids=["o32", "o16", "obf16"])
def test_integers_bit_exact_all_outputs(layout, out_dtype):
    M, N, K = 384, 640, 520
    a, b = operands(M, N, K, gen.BF16, layout, gen.ints(-2, 2), seed=5)
    for name, kw in SHAPE_CFGS:
        check_full(a, b, M, N, K, layout, gen.BF16, out_dtype, exact=True, config=cfg(**kw),
                   what="ints %s %s" % (LNAME[layout], name))


@pytest.mark.parametrize("K", [1, 15, 16, 63, 64, 65, 127, 129, 1000])
def test_k_tails(K):
    M, N = 200, 300
    for layout in LAYOUTS:
        a, b = operands(M, N, K, gen.F16, layout, gen.uniform(-1, 1), seed=K)
        for name, kw in SHAPE_CFGS:
            check_full(a, b, M, N, K, layout, gen.F16, gen.F32, config=cfg(**kw),
                       what="K=%d %s %s" % (K, LNAME[layout], name))


# ---- the persistent loop: many tiles per CTA -----------------------------------

@pytest.mark.parametrize("grid", [4, 8, 0])
@pytest.mark.parametrize("group_m", [1, 3, 8])
def test_quad_persistent_block_loop(grid, group_m):
    """Quads walk several 256 x 512 blocks each (odd tile columns: the last
    block's second pair computes past N and stores nothing)."""
    M, N, K = 1100, 1300, 700
    for layout in LAYOUTS:
        a, b = operands(M, N, K, gen.BF16, layout, gen.ints(-2, 2), seed=61 + group_m)
        check_full(a, b, M, N, K, layout, gen.BF16, gen.F32, exact=True,
                   config=cfg(256, quad=True, group_m=group_m, grid=grid),
                   what="quad grid=%d group_m=%d %s" % (grid, group_m, LNAME[layout]))


@pytest.mark.parametrize("grid", [2, 6, 0])
@pytest.mark.parametrize("group_m", [1, 3, 8, 16])
def test_persistent_tile_loop(grid, group_m):
    """More tiles than CTAs, so each CTA runs the stage ring and both
    accumulator buffers through several phases; the result may not depend on
    the grid size or the tile order."""
    M, N, K = 1100, 1300, 300
    for layout in LAYOUTS:
        a, b = operands(M, N, K, gen.BF16, layout, gen.ints(-2, 2), seed=9)
        for name, kw in SHAPE_CFGS:
            check_full(a, b, M, N, K, layout, gen.BF16, gen.BF16, exact=True,
                       config=cfg(group_m=group_m, grid=grid, **kw),
                       what="grid=%d group=%d %s %s" % (grid, group_m, LNAME[layout], name))


@pytest.mark.parametrize("name,kw", SHAPE_CFGS + [("default", None)], ids=[n for n, _ in SHAPE_CFGS] + ["default"])
def test_more_tiles_than_sms(name, kw):
    M, N, K = 4096, 2304 + 256 * 12, 256
    a, b = operands(M, N, K, gen.F16, gen.B_KN, gen.uniform(-1, 1), seed=11)
    check_full(a, b, M, N, K, gen.B_KN, gen.F16, gen.F16, config=None if kw is None else cfg(**kw),
               what="%dx%dx%d %s" % (M, N, K, name))


# ---- padding, poison and degenerate sizes ---------------------------------------

@pytest.mark.parametrize("layout", LAYOUTS, ids=["nk", "kn"])
def test_poisoned_padding_is_never_read_or_written(layout):
    M, N, K = 300, 200, 150
    b_cols = N if layout == gen.B_KN else K
    lda, ldb, ldc = 152 + 24, -(-b_cols // 8) * 8 + 40, N + 56     # every row 16-byte aligned
    a, b = gen.make_operands(M, N, K, gen.F16, layout, gen.normal(0, 1), None, seed=13,
                             lda=lda, ldb=ldb, pad_value=float("nan"))
    A, B = a.to("cuda:0"), b.to("cuda:0")
    C = torch.full((M + 5, ldc), 12345.0, dtype=torch.float32, device="cuda:0")
    rc = tgemm.tgemm_run(M, N, K, A.data_ptr(), lda, B.data_ptr(), b.shape[1], layout, C.data_ptr(), ldc,
                         gen.F16, gen.F32, None)
    assert rc == 0
    assert tgemm.tgemm_check() == 0
    Cc = C.cpu().double().numpy()
    ref, bound = oracle.gemm(a, b, M, N, K, lda, b.shape[1], layout, gen.F16)
    assert_close(Cc[:M, :N], ref, bound, gen.F32, "padded")
    assert np.all(Cc[:M, N:] == 12345.0), "columns beyond N were written"
    assert np.all(Cc[M:, :] == 12345.0), "rows beyond M were written"


def test_k_zero_writes_the_empty_sum():
    M, N = 70, 96
    C = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda:0")
    A = torch.empty(16, device="cuda:0", dtype=torch.bfloat16)
    rc = tgemm.tgemm_run(M, N, 0, A.data_ptr(), 8, A.data_ptr(), 8, gen.B_NK, C.data_ptr(), N,
                         gen.BF16, gen.BF16, None)
    assert rc == 0 and tgemm.tgemm_check() == 0
    assert torch.count_nonzero(C).item() == 0


def test_empty_m_or_n_leaves_c_untouched():
    C = torch.full((8, 8), 3.0, dtype=torch.float16, device="cuda:0")
    assert tgemm.tgemm_run(0, 8, 8, 0, 8, 0, 8, gen.B_NK, C.data_ptr(), 8, gen.F16, gen.F16, None) == 0
    assert tgemm.tgemm_run(8, 0, 8, 0, 8, 0, 8, gen.B_NK, C.data_ptr(), 8, gen.F16, gen.F16, None) == 0
    assert tgemm.tgemm_check() == 0
    assert torch.all(C == 3.0)


# ---- streams, query and failure reporting -----------------------------------------

def test_runs_on_a_side_stream():
    M, N, K = 512, 768, 256
    a, b = operands(M, N, K, gen.F16, gen.B_NK, gen.ints(-2, 2), seed=17)
    s = torch.cuda.Stream()
    C = run_gpu(a, b, M, N, K, gen.B_NK, gen.F16, gen.F16, stream=s)
    ref, _ = oracle.gemm(a, b, M, N, K, a.shape[1], b.shape[1], gen.B_NK, gen.F16)
    assert np.array_equal(bits(C[:M, :N], gen.F16), oracle.round_bits(ref, gen.F16))


def test_misaligned_rows_pick_the_quad_kernel():
    # K = 5000 BF16 rows are 10000 bytes: not a multiple of 128
    rc, c = tgemm.tgemm_query_config(4000, 3000, 5000, gen.B_NK, gen.BF16, gen.BF16)
    assert rc == 0 and (c.cluster_m, c.bm, c.bn, c.split_k) == (4, 256, 256, 0)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert c.grid == 4 * (sms // 4)          # stream-K tail: every quad
    # FP8 rows of 1040 bytes (16-byte aligned, not 128) are misaligned too; 1024-byte rows are not.  At
    # 1024 x 8192 x 1024 the FP8 rows of the measured table pick the CTA pair; only misaligned rows turn
    # it into a quad.
    rc, c = tgemm.tgemm_query_config(1024, 8192, 1040, gen.B_NK, gen.E4M3, gen.BF16)
    assert rc == 0 and c.cluster_m == 4
    rc, c = tgemm.tgemm_query_config(1024, 8192, 1024, gen.B_NK, gen.E4M3, gen.BF16)
    assert rc == 0 and c.cluster_m == 2


def test_query_config_grid_is_the_launch_grid_for_quads():
    """A configuration returned by tgemm_query_config and passed back to
    tgemm_run_config launches what tgemm_run launches: for the quad, one
    cluster of four per 256 x 512 block (whole blocks)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for M, N, K in [(256, 14336, 4096), (192, 14336, 4096), (256, 16384, 4096)]:
        rc, c = tgemm.tgemm_query_config(M, N, K, gen.B_NK, gen.F16, gen.F16)
        assert rc == 0
        if c.cluster_m == 4 and c.split_k == 1:
            blocks = -(-M // 256) * -(-(-(-N // 256)) // 2)
            assert c.grid == 4 * min(blocks, sms // 4), (M, N, K, c.grid)


def test_query_config_matches_what_runs():
    rc, c = tgemm.tgemm_query_config(8192, 8192, 8192, gen.B_NK, gen.F16, gen.F16)
    assert rc == 0
    assert c.bk == 64 and c.bn in (128, 256) and c.grid >= 1
    assert (c.cluster_m, c.bm) in ((1, 128), (2, 256))
    assert c.grid % c.cluster_m == 0
    assert c.grid <= torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("group_m", [1, 2, 3, 4, 8, 16])
def test_device_tile_order_equals_host(group_m):
    """The kernels' tile order, computed on the GPU, equals the host mapping
    (tgemm_tile_coord) and is a bijection onto the tile grid, for grids up
    to 64 x 64 tiles including short last bands."""
    sizes = [1, 2, 3, 5, 7, 8, 13, 16, 31, 64]
    for tm in sizes:
        for tn in sizes:
            M, N = 128 * tm - 5, 256 * tn - 7
            n = tm * tn
            rows = torch.full((n,), -1, dtype=torch.int32, device="cuda")
            cols = torch.full((n,), -1, dtype=torch.int32, device="cuda")
            assert tgemm.tgemm_debug_tile_order(M, N, 128, 256, group_m, rows.data_ptr(), cols.data_ptr()) == 0
            assert tgemm.tgemm_check() == 0
            r, c = rows.cpu().numpy(), cols.cpu().numpy()
            host = [tgemm.tgemm_tile_coord(M, N, 128, 256, group_m, bid) for bid in range(n)]
            assert all(h[0] == 0 for h in host)
            assert np.array_equal(r, [h[1] for h in host]) and np.array_equal(c, [h[2] for h in host]), \
                "grid %dx%d group %d" % (tm, tn, group_m)
            assert len(set(zip(r.tolist(), c.tolist()))) == n


def test_device_tile_order_rejects_bad_arguments():
    x = torch.empty(4, dtype=torch.int32, device="cuda")
    assert tgemm.tgemm_debug_tile_order(0, 10, 128, 128, 8, x.data_ptr(), x.data_ptr()) == tgemm.ERR_INVALID_ARG
    assert tgemm.tgemm_debug_tile_order(10, 10, 128, 128, 0, x.data_ptr(), x.data_ptr()) == tgemm.ERR_INVALID_ARG
    assert tgemm.tgemm_debug_tile_order(10, 10, 128, 128, 8, None, x.data_ptr()) == tgemm.ERR_INVALID_ARG
    assert tgemm.tgemm_debug_tile_order(1 << 20, 1 << 20, 1, 1, 8, x.data_ptr(), x.data_ptr()) == \
        tgemm.ERR_UNSUPPORTED


def test_bounded_wait_reports_timeout_and_context_survives():
    """A wait on a barrier nothing signals gives up after ~1 ms; the host sees
    TGEMM_ERR_TIMEOUT and the next GEMM still runs correctly."""
    assert tgemm.tgemm_check() == 0
    assert tgemm.tgemm_debug_wait_timeout(1000) == 0
    assert tgemm.tgemm_check() == tgemm.ERR_TIMEOUT
    code = tgemm.tgemm_last_fault_code()
    assert code >> 28 == 7 and (code >> 20) & 0xff == 7
    assert tgemm.tgemm_check() == 0
    M, N, K = 256, 256, 128
    a, b = operands(M, N, K, gen.F16, gen.B_NK, gen.ints(-2, 2), seed=19)
    check_full(a, b, M, N, K, gen.B_NK, gen.F16, gen.F32, exact=True, what="after timeout")


# ---- the swap-AB split-K path (at most 64 rows of A) -------------------------------

def skinny_cfg(npad, splits):
    return tgemm.Config(bm=128, bn=npad, bk=64, stages=4, cluster_m=1, group_m=1, split_k=splits, swap_ab=1,
                        grid=0)


@pytest.mark.parametrize("M", [1, 7, 16, 17, 33, 64])
@pytest.mark.parametrize("layout", LAYOUTS, ids=["nk", "kn"])
def test_skinny_default_pick(M, layout):
    rc, c = tgemm.tgemm_query_config(M, 4096, 512, layout, gen.BF16, gen.BF16)
    assert rc == 0 and c.swap_ab in (1, 2) and c.bn >= M
    for (N, K) in [(300, 1000), (4096, 512), (129, 4160)]:
        for out in (gen.F32, gen.BF16):
            a, b = operands(M, N, K, gen.BF16, layout, gen.normal(0, 1), seed=M + N + K, dist_b=gen.normal(0, 0.02))
            check_full(a, b, M, N, K, layout, gen.BF16, out, what="skinny M=%d N=%d K=%d" % (M, N, K))


@pytest.mark.parametrize("layout", LAYOUTS, ids=["nk", "kn"])
@pytest.mark.parametrize("splits", [1, 2, 3, 7, 32])
def test_skinny_forced_splits_integers_exact(layout, splits):
    M, N, K = 16, 640, 2048
    a, b = operands(M, N, K, gen.F16, layout, gen.ints(-2, 2), seed=23)
    for npad in (16, 32, 64):
        check_full(a, b, M, N, K, layout, gen.F16, gen.F16, exact=True, config=skinny_cfg(npad, splits),
                   what="splits=%d npad=%d" % (splits, npad))


CLUSTER_STAGES = {16: 12, 32: 10, 64: 9, 128: 6}
CLUSTER_MAX_SPLITS = {16: 8, 32: 8, 64: 7, 128: 4}
# the half-size ring: two CTAs per SM
HALF_STAGES = {16: 6, 32: 5, 64: 4}
HALF_MAX_SPLITS = {16: 8, 32: 7, 64: 4}


def cluster_cfg(npad, splits, half=False):
    return tgemm.Config(bm=128, bn=npad, bk=64, stages=(HALF_STAGES if half else CLUSTER_STAGES)[npad],
                        cluster_m=splits, group_m=1, split_k=splits, swap_ab=2, grid=0)


@pytest.mark.parametrize("layout", LAYOUTS, ids=["nk", "kn"])
@pytest.mark.parametrize("npad", [16, 32, 64, 128])
def test_cluster_split_k_integers_exact(layout, npad):
    """Split-K reduced through distributed shared memory inside a cluster, for
    every cluster size the leader can receive (128 rows: up to 4)."""
    M, N, K = (100 if npad == 128 else min(npad, 40)), 700, 1600
    a, b = operands(M, N, K, gen.BF16, layout, gen.ints(-2, 2), seed=41 + npad)
    for splits in range(1, CLUSTER_MAX_SPLITS[npad] + 1):
        check_full(a, b, M, N, K, layout, gen.BF16, gen.F32, exact=True, config=cluster_cfg(npad, splits),
                   what="cluster splits=%d npad=%d" % (splits, npad))


@pytest.mark.parametrize("layout", LAYOUTS, ids=["nk", "kn"])
@pytest.mark.parametrize("npad", [16, 32, 64])
def test_cluster_split_k_half_ring_integers_exact(layout, npad):
    """The half-size ring (two CTAs per SM, fewer stages, fewer partials the
    leader can receive), every cluster size it allows."""
    M, N, K = min(npad, 40), 700, 1600
    a, b = operands(M, N, K, gen.BF16, layout, gen.ints(-2, 2), seed=47 + npad)
    for splits in range(1, HALF_MAX_SPLITS[npad] + 1):
        check_full(a, b, M, N, K, layout, gen.BF16, gen.F32, exact=True, config=cluster_cfg(npad, splits, True),
                   what="half ring splits=%d npad=%d" % (splits, npad))


@pytest.mark.parametrize("npad", [16, 32, 64, 128])
def test_cluster_split_k_one_k_block_per_cta(npad):
    """K ranges of one k-block (ring stage 0 only: the second MMA issuer adds
    nothing) and of one or two (a ragged K), full and half rings."""
    M = 100 if npad == 128 else min(npad, 40)
    for splits in (2, 4):
        for K in (64 * splits, 64 * splits + 16):
            a, b = operands(M, 384, K, gen.BF16, gen.B_NK, gen.ints(-2, 2), seed=59 + npad + K)
            for half in ((False, True) if npad < 128 else (False,)):
                if splits > (HALF_MAX_SPLITS if half else CLUSTER_MAX_SPLITS)[npad]:
                    continue
                check_full(a, b, M, 384, K, gen.B_NK, gen.BF16, gen.F32, exact=True,
                           config=cluster_cfg(npad, splits, half),
                           what="one k-block per CTA npad=%d splits=%d K=%d half=%s" % (npad, splits, K, half))


def test_cluster_split_k_half_ring_two_ctas_per_sm():
    """More CTAs than SMs (128 tiles x 2 splits = 256), all resident two per
    SM, and a ragged last tile; sampled against the oracle."""
    M, N, K = 16, 16384 - 40, 4096
    a, b = operands(M, N, K, gen.BF16, gen.B_NK, gen.normal(0, 1), seed=53, dist_b=gen.normal(0, 0.02))
    for splits in (2, 3):
        check_full(a, b, M, N, K, gen.B_NK, gen.BF16, gen.BF16, config=cluster_cfg(16, splits, True),
                   what="half ring 16x16344x4096 splits=%d" % splits)


def test_cluster_split_k_rejects_too_many_splits():
    x = torch.empty(1 << 16, dtype=torch.bfloat16, device="cuda:0")
    p = x.data_ptr()
    for npad, too_many, half in ((16, 9, False), (64, 8, False), (16, 9, True), (64, 5, True)):
        rc = tgemm.tgemm_run_config(16, 256, 1024, p, 1024, p, 1024, gen.B_NK, p, 256, gen.BF16, gen.BF16, None,
                                    cluster_cfg(npad, too_many, half))
        assert rc == tgemm.ERR_UNSUPPORTED


def test_cluster_and_workspace_reductions_agree_bitwise():
    """Both reductions add the same partials in the same split order."""
    M, N, K = 16, 1024, 2048
    a, b = operands(M, N, K, gen.BF16, gen.B_NK, gen.normal(0, 1), seed=43, dist_b=gen.normal(0, 0.02))
    for splits in (2, 4, 8):
        c1 = run_gpu(a, b, M, N, K, gen.B_NK, gen.BF16, gen.F32, config=cluster_cfg(16, splits))
        c2 = run_gpu(a, b, M, N, K, gen.B_NK, gen.BF16, gen.F32, config=skinny_cfg(16, splits))
        assert torch.equal(c1, c2), "splits=%d" % splits


def test_skinny_repeated_calls_are_bitwise_identical():
    """The arrival counters return to zero after every call and the partials
    are summed in a fixed order, so repeating a call reproduces C exactly."""
    M, N, K = 16, 4096, 4096
    a, b = operands(M, N, K, gen.BF16, gen.B_NK, gen.normal(0, 1), seed=29, dist_b=gen.normal(0, 0.02))
    outs = [run_gpu(a, b, M, N, K, gen.B_NK, gen.BF16, gen.F32) for _ in range(3)]
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    ref, bound = oracle.gemm(a, b, M, N, K, a.shape[1], b.shape[1], gen.B_NK, gen.BF16)
    assert_close(values(outs[0][:M, :N], gen.F32), ref, bound, gen.F32, "16x4096x4096")


def test_skinny_concurrent_streams_do_not_share_partials():
    M, N, K = 32, 2048, 3072
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    ops = [operands(M, N, K, gen.BF16, gen.B_NK, gen.ints(-2, 2), seed=s) for s in (31, 37)]
    dev = [(a.to("cuda:0"), b.to("cuda:0")) for a, b in ops]
    Cs = [torch.empty((M, N), dtype=torch.float32, device="cuda:0") for _ in range(2)]
    torch.cuda.synchronize()
    for _ in range(5):
        for (A, B), C, s in zip(dev, Cs, (s1, s2)):
            rc = tgemm.tgemm_run(M, N, K, A.data_ptr(), A.shape[1], B.data_ptr(), B.shape[1], gen.B_NK,
                                 C.data_ptr(), N, gen.BF16, gen.F32, tgemm.ctypes.c_void_p(s.cuda_stream))
            assert rc == 0
    torch.cuda.synchronize()
    assert tgemm.tgemm_check() == 0
    for (a, b), C in zip(ops, Cs):
        ref, _ = oracle.gemm(a, b, M, N, K, a.shape[1], b.shape[1], gen.B_NK, gen.BF16)
        assert np.array_equal(C.cpu().double().numpy(), ref)


def test_query_config_follows_the_measured_table():
    # 8192^3 with B stored N x K is a grid point of the table: the CTA pair won there
    rc, c = tgemm.tgemm_query_config(8192, 8192, 8192, gen.B_NK, gen.F16, gen.F16)
    assert rc == 0 and (c.cluster_m, c.bm, c.bn) == (2, 256, 256)
    # 16 x 4096 x 4096: the in-cluster split-K path
    rc, c = tgemm.tgemm_query_config(16, 4096, 4096, gen.B_NK, gen.BF16, gen.BF16)
    assert rc == 0 and c.swap_ab == 2 and c.split_k == c.cluster_m


# ---- stream-K tail of the CTA-pair kernel -------------------------------------------

def sk_cfg(pairs=0, group_m=8):
    return tgemm.Config(bm=256, bn=256, bk=64, stages=6, cluster_m=2, group_m=group_m, split_k=0, swap_ab=0,
                        grid=2 * pairs)


@pytest.mark.parametrize("layout", LAYOUTS, ids=["nk", "kn"])
@pytest.mark.parametrize("pairs", [3, 4, 7, 13, 0])
def test_stream_k_tail_integers_exact(layout, pairs):
    """1100 x 1300 pair tiles (5 x 6 = 30) over 3, 4, 7, 13 or all pairs: the
    last waves' tiles are shared out by k-block and summed from partials."""
    M, N, K = 1100, 1300, 1500
    a, b = operands(M, N, K, gen.BF16, layout, gen.ints(-2, 2), seed=47)
    check_full(a, b, M, N, K, layout, gen.BF16, gen.F32, exact=True, config=sk_cfg(pairs),
               what="stream-K pairs=%d %s" % (pairs, LNAME[layout]))


@pytest.mark.parametrize("shape", [(256, 256, 8192), (300, 520, 4000), (1000, 700, 3000), (2304, 1280, 1024)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("out_dtype", [gen.F32, gen.BF16], ids=["o32", "obf16"])
def test_stream_k_random_values(shape, out_dtype):
    M, N, K = shape
    a, b = operands(M, N, K, gen.BF16, gen.B_NK, gen.normal(0, 1), seed=53)
    check_full(a, b, M, N, K, gen.B_NK, gen.BF16, out_dtype, config=sk_cfg(), what="stream-K %s" % (shape,))


def test_stream_k_is_deterministic_across_calls():
    M, N, K = 640, 1280, 6000
    a, b = operands(M, N, K, gen.F16, gen.B_NK, gen.normal(0, 1), seed=59)
    outs = [run_gpu(a, b, M, N, K, gen.B_NK, gen.F16, gen.F32, config=sk_cfg()) for _ in range(3)]
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


# ---- stream-K tail of the quad kernel ---------------------------------------------

def qsk_cfg(quads=0, group_m=8):
    return tgemm.Config(bm=256, bn=256, bk=64, stages=6, cluster_m=4, group_m=group_m, split_k=0, swap_ab=0,
                        grid=4 * quads)


@pytest.mark.parametrize("layout", LAYOUTS, ids=["nk", "kn"])
@pytest.mark.parametrize("n", [1300, 1100], ids=["even_cols", "odd_cols"])
@pytest.mark.parametrize("quads", [2, 3, 4, 6, 7, 0])
def test_quad_stream_k_integers_exact(layout, n, quads):
    """1100 x N blocks of 256 x 512 (5 x 3 = 15) over 2, 3, 4, 6, 7 or all
    resident quads.  Where the leftover wave is at most half full (2, 6, 7
    quads) its blocks are shared out by k-block; with more quads than blocks
    all of them are; 3 quads leave no leftover and 4 a more than half full
    one, which stay whole blocks.  Both pairs of a quad run the same k-range,
    and each tile half is summed from its partials.  N = 1100 has odd tile
    columns: the last block's second tile lies past N and stores nothing."""
    M, N, K = 1100, n, 1500
    a, b = operands(M, N, K, gen.BF16, layout, gen.ints(-2, 2), seed=83)
    check_full(a, b, M, N, K, layout, gen.BF16, gen.F32, exact=True, config=qsk_cfg(quads),
               what="quad stream-K quads=%d N=%d %s" % (quads, N, LNAME[layout]))


@pytest.mark.parametrize("shape", [(256, 512, 8192), (300, 520, 4000), (1000, 1500, 2500), (2304, 1280, 1024)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("out_dtype", [gen.F32, gen.BF16], ids=["o32", "obf16"])
def test_quad_stream_k_random_values(shape, out_dtype):
    """Random values, including rows that are not 128-byte multiples
    (K = 2500 BF16: 5000-byte rows), which is where the quad is chosen."""
    M, N, K = shape
    a, b = operands(M, N, K, gen.BF16, gen.B_NK, gen.normal(0, 1), seed=89)
    check_full(a, b, M, N, K, gen.B_NK, gen.BF16, out_dtype, config=qsk_cfg(), what="quad stream-K %s" % (shape,))


def test_quad_stream_k_is_deterministic_across_calls():
    M, N, K = 640, 1280, 6000
    a, b = operands(M, N, K, gen.F16, gen.B_NK, gen.normal(0, 1), seed=97)
    outs = [run_gpu(a, b, M, N, K, gen.B_NK, gen.F16, gen.F32, config=qsk_cfg()) for _ in range(3)]
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


# ---- back-to-back dependent launches ------------------------------------------

@pytest.mark.parametrize("kinds", [("pair", "pair", "pair"), ("pair", "cta128", "quad"), ("quad", "auto", "cta256")])
def test_chained_products_see_each_others_results(kinds):
    """C1 = A B, C2 = C1 D, C3 = C2 E launched back to back on one stream with
    no synchronisation in between: each launch may start early (programmatic
    dependent launch) and must still read the previous product complete.
    Small integers keep every intermediate exact in FP16, so C3 is compared bit
    for bit with the oracle's chain."""
    M, K1, N1, N2, N3 = 256, 16, 128, 512, 256
    g = torch.Generator().manual_seed(77)
    A = torch.randint(-1, 2, (M, K1), generator=g).half()
    B = torch.randint(-1, 2, (N1, K1), generator=g).half()       # N x K
    D = torch.randint(-1, 2, (N2, N1), generator=g).half()
    E = torch.randint(-1, 2, (N3, N2), generator=g).half()
    configs = {
        "pair": cfg(256, pair=True), "quad": cfg(256, quad=True), "cta128": cfg(128), "cta256": cfg(256),
        "auto": None,
    }
    dev = "cuda:0"
    Ad, Bd, Dd, Ed = A.to(dev), B.to(dev), D.to(dev), E.to(dev)
    C1 = torch.empty(M, N1, dtype=torch.float16, device=dev)
    C2 = torch.empty(M, N2, dtype=torch.float16, device=dev)
    C3 = torch.empty(M, N3, dtype=torch.float32, device=dev)
    steps = [(Ad, Bd, C1, K1, N1, gen.F16), (C1, Dd, C2, N1, N2, gen.F16), (C2, Ed, C3, N2, N3, gen.F32)]
    for (x, w, c, k, n, out), kind in zip(steps, kinds):
        args = (M, n, k, x.data_ptr(), k, w.data_ptr(), k, gen.B_NK, c.data_ptr(), n, gen.F16, out, None)
        conf = configs[kind]
        rc = tgemm.tgemm_run(*args) if conf is None else tgemm.tgemm_run_config(*args, conf)
        assert rc == tgemm.OK, tgemm.status_string(rc)
    assert tgemm.tgemm_check() == tgemm.OK
    # the oracle's chain, each intermediate rounded to FP16 as the GPU stores it
    r1, _ = oracle.gemm(A, B, M, N1, K1, K1, K1, gen.B_NK, gen.F16)
    c1 = torch.from_numpy(oracle.round_bits(r1, gen.F16).astype(np.uint16).view(np.int16)).view(torch.float16)
    r2, _ = oracle.gemm(c1, D, M, N2, N1, N1, N1, gen.B_NK, gen.F16)
    c2 = torch.from_numpy(oracle.round_bits(r2, gen.F16).astype(np.uint16).view(np.int16)).view(torch.float16)
    r3, _ = oracle.gemm(c2, E, M, N3, N2, N2, N2, gen.B_NK, gen.F16)
    assert np.abs(r2).max() <= 2048                                 # every intermediate exact in FP16
    assert np.array_equal(bits(C3.cpu(), gen.F32), oracle.round_bits(r3, gen.F32))


@pytest.mark.parametrize("graph", [False, True], ids=["stream", "graph"])
def test_chained_skinny_products_see_each_others_results(graph):
    """Eight 16-row projections X_{i+1} = X_i W_i^T launched back to back (the
    in-cluster swap-AB kernel and its reduce-scatter exchange): each launch
    may start early and must read the previous launch's owners' stores
    complete.  Small integers keep every intermediate exact in BF16, so the
    last product is compared bit for bit with the oracle's chain."""
    M, N = 16, 1024
    g = torch.Generator().manual_seed(79)
    x0 = torch.randint(-1, 2, (M, N), generator=g).to(torch.bfloat16)
    # weights with one +-1 per row, so every intermediate stays in {-1, 0, 1} x small
    W = []
    for i in range(8):
        w = torch.zeros(N, N)
        cols = torch.randperm(N, generator=g)[:N]
        w[torch.arange(N), cols] = torch.randint(0, 2, (N,), generator=g).float() * 2 - 1
        W.append(w.to(torch.bfloat16))
    dev = "cuda:0"
    Wd = [w.to(dev) for w in W]
    X = [x0.to(dev)] + [torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev) for _ in W]
    s = torch.cuda.Stream()
    sh = tgemm.ctypes.c_void_p(s.cuda_stream)
    cfg = tgemm.Config(bm=128, bn=16, bk=64, stages=6, cluster_m=4, group_m=1, split_k=4, swap_ab=2, grid=0)

    def launch_all():
        for i, w in enumerate(Wd):
            rc = tgemm.tgemm_run_config(M, N, N, X[i].data_ptr(), N, w.data_ptr(), N, gen.B_NK, X[i + 1].data_ptr(),
                                        N, gen.BF16, gen.BF16, sh, cfg)
            assert rc == tgemm.OK, tgemm.status_string(rc)

    torch.cuda.synchronize()
    if graph:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            launch_all()
        for t in X[1:]:
            t.fill_(float("nan"))
        gr.replay()
    else:
        with torch.cuda.stream(s):
            launch_all()
    torch.cuda.synchronize()
    assert tgemm.tgemm_check(sh) == tgemm.OK
    ref = x0
    for w in W:
        r, _ = oracle.gemm(ref, w, M, N, N, N, N, gen.B_NK, gen.BF16)
        ref = torch.from_numpy(oracle.round_bits(r, gen.BF16).astype(np.uint16).view(np.int16)).view(torch.bfloat16)
    assert np.array_equal(bits(X[-1].cpu(), gen.BF16), bits(ref, gen.BF16))


LOG_RUN = r"""
import sys, torch
sys.path.insert(0, %r)
from dense_tiled_gemm_persistent_gb300 import tgemm
for M, N, K in [(1024, 1024, 1024), (16, 4096, 4096), (4000, 3000, 5000)]:
    A = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda:0")
    B = torch.zeros(N, K, dtype=torch.bfloat16, device="cuda:0")
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda:0")
    assert tgemm.tgemm_run(M, N, K, A.data_ptr(), K, B.data_ptr(), K, tgemm.B_NK, C.data_ptr(), N, tgemm.BF16,
                           tgemm.BF16, None) == 0
    assert tgemm.tgemm_check() == 0
    rc, c = tgemm.tgemm_query_config(M, N, K, tgemm.B_NK, tgemm.BF16, tgemm.BF16)
    print("%%d %%d %%d %%d %%d %%d %%d %%d" %% (c.bm, c.bn, c.stages, c.cluster_m, c.group_m, c.split_k, c.swap_ab, c.grid))
"""


def test_log_line_shows_what_tgemm_query_config_returns():
    """With TGEMM_LOG=1 every call prints the configuration it launched; for
    the library's own choice that is tgemm_query_config's answer."""
    import os
    import re
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", LOG_RUN % root], env=dict(os.environ, TGEMM_LOG="1"),
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    logged = [ln for ln in r.stderr.splitlines() if ln.startswith("tgemm: tgemm_run ")]
    queried = r.stdout.split("\n")
    assert len(logged) == 3
    for ln, q in zip(logged, queried):
        m = re.search(r"bm=(\d+) bn=(\d+) bk=64 stages=(\d+) cluster_m=(\d+) group_m=(\d+) split_k=(\d+) "
                      r"swap_ab=(\d+) grid=(\d+)", ln)
        assert m and ln.endswith("; ok") and "config=library" in ln, ln
        got = [int(x) for x in m.groups()]
        want = [int(x) for x in q.split()]
        assert got[:7] == want[:7], (ln, q)


def test_sm_clock_probe_reads_a_plausible_clock():
    """tgemm_debug_sm_clock: cycles over at least the asked time, at a clock
    between 300 MHz and the device's maximum (with 5 % slack)."""
    out = torch.zeros(2, dtype=torch.int64, device="cuda:0")
    assert tgemm.tgemm_debug_sm_clock(out.data_ptr(), 50) == 0
    assert tgemm.tgemm_check() == 0
    ns, cyc = out.tolist()
    assert ns >= 50_000
    mhz = cyc * 1e3 / ns
    assert 300 <= mhz <= 2070 * 1.05, mhz


def test_clock_record_counts_launches_and_reads_a_plausible_clock():
    """tgemm_debug_clock_record: every GEMM kernel launched while it is set
    adds its elapsed time and SM cycles; none after it is cleared."""
    rec = torch.zeros(8, dtype=torch.int64, device="cuda:0")
    assert tgemm.tgemm_debug_clock_record(rec.data_ptr()) == 0
    try:
        M, N, K = 512, 512, 512
        a, b = operands(M, N, K, gen.F16, gen.B_NK, gen.ints(-2, 2), seed=3)
        for name, kw in SHAPE_CFGS:
            check_full(a, b, M, N, K, gen.B_NK, gen.F16, gen.F32, exact=True, config=cfg(**kw), what=name)
        a16, b16 = operands(16, 4096, 4096, gen.BF16, gen.B_NK, gen.normal(0, 1), seed=4)
        run_gpu(a16, b16, 16, 4096, 4096, gen.B_NK, gen.BF16, gen.BF16)    # a skinny kernel
    finally:
        assert tgemm.tgemm_debug_clock_record(None) == 0
    ns, cyc, n = rec[:3].tolist()
    assert n == len(SHAPE_CFGS) + 1
    mhz = cyc * 1e3 / ns
    assert 300 <= mhz <= 2070 * 1.05, mhz
    run_gpu(a, b, M, N, K, gen.B_NK, gen.F16, gen.F32)
    assert rec[2].item() == n


@pytest.mark.parametrize("M", [65, 100, 128])
@pytest.mark.parametrize("layout", LAYOUTS, ids=["nk", "kn"])
def test_swap_ab_128_rows(M, layout):
    """65-128 rows of A on the in-cluster kernel padded to 128 (MMA N = 128):
    the library's own pick on a weight whose column tiles alone do not fill
    the GPU, random values against the oracle, both output widths."""
    N, K = 4096, 2048
    rc, c = tgemm.tgemm_query_config(M, N, K, layout, gen.BF16, gen.BF16)
    assert rc == 0 and c.swap_ab == 2 and c.bn == 128 and 1 <= c.split_k <= 4
    a, b = operands(M, N, K, gen.BF16, layout, gen.normal(0, 1), seed=M + 3, dist_b=gen.normal(0, 0.02))
    for out in (gen.F32, gen.BF16):
        check_full(a, b, M, N, K, layout, gen.BF16, out, what="swap-AB 128 rows M=%d" % M)


def test_swap_ab_128_rows_with_epilogue_and_ragged_n():
    """The fused epilogue (alpha, bias, GELU) on the 128-row kernel, with a
    ragged last column tile."""
    M, N, K = 96, 1000, 1024
    a, b = operands(M, N, K, gen.F16, gen.B_NK, gen.normal(0, 1), seed=9, dist_b=gen.normal(0, 0.05))
    A, B = a.to("cuda:0"), b.to("cuda:0")
    ldc = 1000
    Cd = torch.full((M, ldc), float("nan"), dtype=torch.float32, device="cuda:0")
    bias = torch.randn(N).to("cuda:0")
    ep = tgemm.Epilogue(alpha=0.5, beta=0.0, c_in=None, ldc_in=ldc, bias=bias.data_ptr(), bias_dtype=gen.F32,
                        act=tgemm.ACT_GELU_TANH)
    for splits in (1, 2, 4):
        rc = tgemm.tgemm_run_ex(M, N, K, A.data_ptr(), A.shape[1], B.data_ptr(), B.shape[1], gen.B_NK, Cd.data_ptr(),
                                ldc, gen.F16, gen.F32, None, ep, cluster_cfg(128, splits))
        assert rc == 0, tgemm.status_string(rc)
        assert tgemm.tgemm_check() == 0
        acc, bound = oracle.gemm(a, b, M, N, K, a.shape[1], b.shape[1], gen.B_NK, gen.F16)
        bias64 = bias.double().cpu().numpy()
        ref = oracle.epilogue(acc, 0.5, 0.0, None, bias64, oracle.ACT_GELU_TANH)
        mag = np.abs(0.5 * acc) + np.abs(bias64)[None, :]
        tol = 1.13 * (0.5 * 1e-3 * bound + 2.0 ** -20 * mag) + oracle.ulp(ref, gen.F32)
        got = Cd.double().cpu().numpy()
        assert np.all(np.abs(got - ref) <= tol), "splits=%d" % splits


def test_swap_ab_128_rows_rejects_five_splits_and_the_workspace_kernel():
    x = torch.empty(1 << 16, dtype=torch.bfloat16, device="cuda:0")
    p = x.data_ptr()
    rc = tgemm.tgemm_run_config(100, 256, 1024, p, 1024, p, 1024, gen.B_NK, p, 256, gen.BF16, gen.BF16, None,
                                cluster_cfg(128, 5))
    assert rc == tgemm.ERR_UNSUPPORTED
    rc = tgemm.tgemm_run_config(100, 256, 1024, p, 1024, p, 1024, gen.B_NK, p, 256, gen.BF16, gen.BF16, None,
                                skinny_cfg(128, 4))
    assert rc == tgemm.ERR_UNSUPPORTED


# ---- maximum sizes ----------------------------------------------------------------

@pytest.mark.parametrize("name,kw", SHAPE_CFGS + [("default", None)], ids=[n for n, _ in SHAPE_CFGS] + ["default"])
def test_long_k_integers_exact(name, kw):
    """K = 2^17: 2048 k-blocks, so the stage ring and its barrier phases wrap
    hundreds of times inside one tile; small integers keep every partial sum
    exact in FP32, so the result is bit-exact."""
    M, N, K = 256, 256, 1 << 17
    a, b = operands(M, N, K, gen.BF16, gen.B_NK, gen.ints(-2, 2), seed=101)
    check_full(a, b, M, N, K, gen.B_NK, gen.BF16, gen.F32, exact=True, config=None if kw is None else cfg(**kw),
               what="K=2^17 %s" % name)


def test_output_beyond_2_31_elements():
    """C of 65536 x 65536 FP16 elements (8 GiB, 2^32 elements): offsets past
    2^31 elements in every addressing path of the chosen kernel; sampled
    elements (the last row and column included) against the oracle."""
    M = N = 65536
    K = 64
    a, b = operands(M, N, K, gen.F16, gen.B_NK, gen.ints(-2, 2), seed=103)
    A, B = a.to(DEV_), b.to(DEV_)
    C = torch.empty((M, N), dtype=torch.float16, device=DEV_)
    rc = tgemm.tgemm_run(M, N, K, A.data_ptr(), K, B.data_ptr(), K, gen.B_NK, C.data_ptr(), N, gen.F16, gen.F16, None)
    assert rc == 0 and tgemm.tgemm_check() == 0
    rng = np.random.default_rng(7)
    ii = np.concatenate([rng.integers(0, M, 8192), np.full(N, M - 1), np.arange(M), [M - 1, 0, M - 1]])
    jj = np.concatenate([rng.integers(0, N, 8192), np.arange(N), np.full(M, N - 1), [0, N - 1, N - 1]])
    got = C[torch.from_numpy(ii).to(DEV_), torch.from_numpy(jj).to(DEV_)].cpu()
    del C
    ref, _ = oracle.gemm_elements(a, b, M, N, K, K, K, gen.B_NK, gen.F16, ii, jj)
    want = oracle.round_bits(ref, gen.F16)
    assert np.array_equal(bits(got, gen.F16), want)


def test_skinny_widest_n():
    """16 rows against a 524288 x 256 weight (4096 column tiles), on the
    library's pick and on the workspace kernel; full comparison."""
    M, N, K = 16, 1 << 19, 256
    a, b = operands(M, N, K, gen.BF16, gen.B_NK, gen.normal(0, 1), seed=107, dist_b=gen.normal(0, 0.02))
    for conf in (None, skinny_cfg(16, 2)):
        check_full(a, b, M, N, K, gen.B_NK, gen.BF16, gen.BF16, config=conf, what="16 x 2^19 x 256")
