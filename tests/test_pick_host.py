"""Host-side tests of the automatic configuration choice (no GPU needed).

tgemm_query_config_sms runs the steps tgemm_run takes to choose a
configuration: the measured table, the wave model off its grid, the quad for
misaligned rows, the band height. It takes the SM count from the caller
instead of the device. These tests pin its choice on every named workload
for a 152-SM GB300, and check over a grid of shapes that each choice passes
the library's own legality checks. On a GPU they check that it agrees with
tgemm_query_config.
"""
import itertools

import pytest

from dense_tiled_gemm_persistent_gb300 import build as libbuild
from dense_tiled_gemm_persistent_gb300 import inputs as gen
from dense_tiled_gemm_persistent_gb300 import tgemm

SMS = 152
FAKE = 1 << 20   # a 16-byte aligned non-null address, never dereferenced by host checks


@pytest.fixture(scope="module", autouse=True)
def lib():
    libbuild.build()
    return tgemm.load()


def pick(M, N, K, layout, ind, outd, sms=SMS):
    rc, c = tgemm.tgemm_query_config_sms(M, N, K, layout, ind, outd, sms)
    assert rc == 0, tgemm.status_string(rc)
    return c


def fields(c):
    return dict(bm=c.bm, bn=c.bn, stages=c.stages, cluster_m=c.cluster_m, group_m=c.group_m, split_k=c.split_k,
                swap_ab=c.swap_ab)


# The choices the bench's measurements were taken with (kernel families in the
# measurement tables: 1-CTA, pair and quad tiles with or without a stream-K
# tail, in-cluster swap-AB split-K), on the current picker table.
PINNED = {
    "gemm_256x256x256_f16_kn_f32": dict(bm=128, bn=128, stages=6, cluster_m=1, group_m=8, split_k=1, swap_ab=0),
    "gemm_4000x3000x5000_bf16_nk_bf16": dict(bm=256, bn=256, stages=6, cluster_m=4, group_m=8, split_k=0,
                                             swap_ab=0),
    "gemm_4096x4096x4096_f16_kn_f16": dict(bm=256, bn=256, stages=6, cluster_m=2, group_m=8, split_k=0, swap_ab=0),
    "gemm_8192x4864x1024_f16_nk_f16": dict(bm=256, bn=256, stages=6, cluster_m=2, group_m=8, split_k=1, swap_ab=0),
    "gemm_8192x8192x8192_f16_nk_f16": dict(bm=256, bn=256, stages=6, cluster_m=2, group_m=11, split_k=0,
                                           swap_ab=0),
    "gemm_8192x8192x8192_e4m3_nk_bf16": dict(bm=256, bn=256, stages=6, cluster_m=2, group_m=16, split_k=1,
                                             swap_ab=0),
    "gemm_8192x8192x8192_tf32_nk_f32": dict(bm=256, bn=256, stages=6, cluster_m=4, group_m=11, split_k=0,
                                            swap_ab=0),
    "proj_16384x14336x4096_bf16_nk_bf16": dict(bm=256, bn=256, stages=6, cluster_m=2, group_m=16, split_k=1,
                                               swap_ab=0),
    "proj_16x4096x4096_bf16_nk_bf16": dict(bm=128, bn=16, stages=6, cluster_m=8, group_m=1, split_k=8, swap_ab=2),
    "proj_16x4096x4096_e4m3_nk_bf16": dict(bm=128, bn=16, stages=6, cluster_m=4, group_m=1, split_k=4, swap_ab=2),
    "proj_128x4096x4096_bf16_nk_bf16": dict(bm=128, bn=128, stages=6, cluster_m=3, group_m=1, split_k=3,
                                            swap_ab=2),
}


@pytest.mark.parametrize("name", sorted(PINNED))
def test_named_workloads_pick_the_measured_configuration(name):
    wl = gen.WORKLOADS[name]
    assert fields(pick(wl.M, wl.N, wl.K, wl.b_layout, wl.in_dtype, wl.out_dtype)) == PINNED[name]


def test_every_named_workload_is_pinned():
    assert set(PINNED) | {"gemm_256x256x256_f16_kn_f32_ints"} == set(gen.WORKLOADS)


def _accepted(M, N, K, layout, ind, outd, cfg):
    # FAKE pointers: an accepted configuration stops at the device query
    # (no GPU here) instead of launching
    ldb = N if layout == gen.B_KN else K
    rc = tgemm.tgemm_run_config(M, N, K, FAKE, K, FAKE, ldb, layout, FAKE, N, ind, outd, None, cfg)
    return rc in (tgemm.ERR_CUDA, tgemm.ERR_ARCH)


def test_every_choice_passes_the_legality_checks():
    import torch
    if torch.cuda.is_available():
        pytest.skip("host-path check with placeholder pointers; runs only without a GPU")
    ms = [1, 16, 17, 64, 65, 128, 129, 256, 1000, 4096, 16384]
    ns = [64, 512, 4096, 14336]
    ks = [64, 128, 1024, 4096, 16384]
    kinds = [(gen.F16, gen.F16, gen.B_NK), (gen.BF16, gen.BF16, gen.B_KN), (gen.F16, gen.F32, gen.B_KN),
             (gen.E4M3, gen.BF16, gen.B_NK), (gen.F32, gen.F32, gen.B_NK)]
    n = 0
    for (M, N, K), (ind, outd, layout) in itertools.product(itertools.product(ms, ns, ks), kinds):
        c = pick(M, N, K, layout, ind, outd)
        c.grid = 0
        assert _accepted(M, N, K, layout, ind, outd, c), (M, N, K, ind, outd, layout, fields(c))
        if c.swap_ab:
            assert M <= 128 and c.bn >= M and c.bm == 128
        else:
            assert c.bm in (128, 256) and c.group_m >= 1
        n += 1
    assert n == len(ms) * len(ns) * len(ks) * len(kinds)


def test_sm_count_shapes_the_grid_not_the_tile_choice_on_the_table():
    # the table's measured tile shape stays; the persistent grid follows the SMs
    a = pick(8192, 8192, 8192, gen.B_NK, gen.F16, gen.F16, 152)
    b = pick(8192, 8192, 8192, gen.B_NK, gen.F16, gen.F16, 148)
    assert (a.bm, a.bn, a.cluster_m) == (b.bm, b.bn, b.cluster_m)
    assert a.grid == 152 and b.grid == 148


def test_rejects_bad_arguments():
    assert tgemm.tgemm_query_config_sms(64, 64, 64, gen.B_NK, gen.F16, gen.F16, 0)[0] == tgemm.ERR_INVALID_ARG
    assert tgemm.tgemm_query_config_sms(64, 64, 64, gen.B_NK, gen.F16, gen.F16, 5000)[0] == tgemm.ERR_INVALID_ARG
    assert tgemm.tgemm_query_config_sms(-1, 64, 64, gen.B_NK, gen.F16, gen.F16, 152)[0] == tgemm.ERR_INVALID_ARG
    assert tgemm.tgemm_query_config_sms(64, 64, 64, 7, gen.F16, gen.F16, 152)[0] == tgemm.ERR_INVALID_ARG
    assert tgemm.tgemm_query_config_sms(64, 64, 64, gen.B_KN, gen.E4M3, gen.F16, 152)[0] == tgemm.ERR_UNSUPPORTED
    assert tgemm.tgemm_query_config_sms(64, 64, 64, gen.B_NK, gen.F16, gen.E4M3, 152)[0] == tgemm.ERR_INVALID_ARG


@pytest.mark.gpu
def test_agrees_with_the_device_query():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for name, wl in sorted(gen.WORKLOADS.items()):
        rc, dev = tgemm.tgemm_query_config(wl.M, wl.N, wl.K, wl.b_layout, wl.in_dtype, wl.out_dtype)
        assert rc == 0
        host = pick(wl.M, wl.N, wl.K, wl.b_layout, wl.in_dtype, wl.out_dtype, sms)
        assert fields(host) == fields(dev) and host.grid == dev.grid, name
