"""Host-side tests of the C-ABI library (no GPU needed).

The library must load, export every entry point include/tgemm.h declares, and
reject bad arguments on the host before touching the device.  The scheduler's
tile mapping is checked against the pages' worked examples.
"""
import os
import re

import numpy as np
import pytest

from dense_tiled_gemm_persistent_gb300 import build as libbuild
from dense_tiled_gemm_persistent_gb300 import tgemm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return tgemm.load()


def read_golden(name):
    out = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, v = (s.strip() for s in line.split("=", 1))
        out[k] = [float(x) if "." in x else int(x) for x in v.split()]
    return out


def header_functions():
    src = open(os.path.join(ROOT, "include", "tgemm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tgemm_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    declared = header_functions()
    assert set(declared) == set(tgemm.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name
    nm = os.popen("nm -D --defined-only %s" % tgemm.LIB_PATH).read()
    exported = set(re.findall(r" T (tgemm_\w+)", nm))
    assert set(declared) <= exported
    # nothing else leaks out of the library under our prefix
    assert exported == set(declared)


def test_header_is_plain_c(tmp_path):
    """include/tgemm.h compiles as C99 on its own: plain pointers, sizes and
    enums, no C++ or torch types in the boundary."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    src = tmp_path / "use_header.c"
    src.write_text('#include "tgemm.h"\n'
                   "int main(void) {\n"
                   "    tgemm_config c = {0};\n"
                   "    tgemm_epilogue e = {1.0f, 0.0f, 0, 0, 0, TGEMM_F32, TGEMM_ACT_NONE};\n"
                   "    (void)c; (void)e;\n"
                   "    return tgemm_status_string(TGEMM_OK) == 0;\n"
                   "}\n")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only",
                        "-I" + os.path.join(ROOT, "include"), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_status_strings(lib):
    for code in range(8):
        s = tgemm.status_string(code)
        assert isinstance(s, str) and s
    assert tgemm.status_string(0) == "ok"
    assert "unknown" in tgemm.status_string(99)


FAKE = 1 << 20   # a 16-byte aligned non-null address, never dereferenced by host checks


@pytest.mark.parametrize("case,expect", [
    (dict(M=-1), tgemm.ERR_INVALID_ARG),
    (dict(K=-5), tgemm.ERR_INVALID_ARG),
    (dict(lda=63), tgemm.ERR_INVALID_ARG),            # lda < K
    (dict(ldb=63), tgemm.ERR_INVALID_ARG),            # NK: ldb < K
    (dict(ldc=95), tgemm.ERR_INVALID_ARG),            # ldc < N
    (dict(A=0), tgemm.ERR_INVALID_ARG),
    (dict(C=0), tgemm.ERR_INVALID_ARG),
    (dict(A=FAKE + 8), tgemm.ERR_MISALIGNED),
    (dict(C=FAKE + 4), tgemm.ERR_MISALIGNED),
    (dict(lda=68), tgemm.ERR_MISALIGNED),             # 68 * 2 bytes is not a multiple of 16
    (dict(ldc=98, out=tgemm.F32), tgemm.ERR_MISALIGNED),   # 392 bytes
    (dict(layout=7), tgemm.ERR_INVALID_ARG),
    (dict(ind=5), tgemm.ERR_INVALID_ARG),
    (dict(out=9), tgemm.ERR_INVALID_ARG),
    (dict(ind=tgemm.F32, layout=tgemm.B_KN, ldb=96), tgemm.ERR_UNSUPPORTED),    # TF32 operands: B N x K only
    (dict(ind=tgemm.E4M3, layout=tgemm.B_KN, ldb=96), tgemm.ERR_UNSUPPORTED),   # FP8 operands: B N x K only
    (dict(ind=tgemm.E5M2, lda=72), tgemm.ERR_MISALIGNED),                       # 72-byte FP8 rows
    (dict(M=1 << 31), tgemm.ERR_UNSUPPORTED),
])
def test_host_argument_checks(lib, case, expect):
    a = dict(M=128, N=96, K=64, A=FAKE, lda=64, B=FAKE, ldb=64, layout=tgemm.B_NK, C=FAKE, ldc=96,
             ind=tgemm.F16, out=tgemm.F16)
    a.update(case)
    rc = tgemm.tgemm_run(a["M"], a["N"], a["K"], a["A"], a["lda"], a["B"], a["ldb"], a["layout"],
                         a["C"], a["ldc"], a["ind"], a["out"], None)
    assert rc == expect, tgemm.status_string(rc)


def test_empty_output_is_a_noop_without_device(lib):
    # M = 0 or N = 0: nothing to do, not even a device query; NULL pointers are fine
    assert tgemm.tgemm_run(0, 10, 10, 0, 10, 0, 10, tgemm.B_NK, 0, 10, tgemm.F16, tgemm.F16, None) == 0
    assert tgemm.tgemm_run(10, 0, 10, 0, 10, 0, 10, tgemm.B_NK, 0, 0, tgemm.F16, tgemm.F16, None) == 0


def test_run_config_rejects_unknown_configuration(lib):
    cfg = tgemm.Config(bm=128, bn=200, bk=64, stages=4, cluster_m=1, group_m=8, split_k=1, swap_ab=0, grid=0)
    rc = tgemm.tgemm_run_config(128, 96, 64, FAKE, 64, FAKE, 64, tgemm.B_NK, FAKE, 96, tgemm.F16,
                                tgemm.F16, None, cfg)
    assert rc == tgemm.ERR_UNSUPPORTED


def test_tile_order_probe_checks_arguments_on_the_host(lib):
    # rejected before any device query: no GPU needed
    assert tgemm.tgemm_debug_tile_order(0, 10, 128, 128, 8, FAKE, FAKE) == tgemm.ERR_INVALID_ARG
    assert tgemm.tgemm_debug_tile_order(10, 10, 128, 0, 8, FAKE, FAKE) == tgemm.ERR_INVALID_ARG
    assert tgemm.tgemm_debug_tile_order(10, 10, 128, 128, 8, None, FAKE) == tgemm.ERR_INVALID_ARG
    assert tgemm.tgemm_debug_tile_order(1 << 20, 1 << 20, 1, 1, 8, FAKE, FAKE) == tgemm.ERR_UNSUPPORTED


def _cfg(bm=128, bn=256, bk=64, stages=4, cluster_m=1, group_m=8, split_k=1, swap_ab=0, grid=0):
    return tgemm.Config(bm=bm, bn=bn, bk=bk, stages=stages, cluster_m=cluster_m, group_m=group_m, split_k=split_k,
                        swap_ab=swap_ab, grid=grid)


LEGAL = [
    ("cta256", dict(), 256, tgemm.F16),
    ("cta128", dict(bn=128, stages=6), 256, tgemm.F16),
    ("cta128_2stage", dict(bn=128, stages=2), 256, tgemm.F16),
    ("pair", dict(bm=256, stages=6, cluster_m=2), 256, tgemm.F16),
    ("pair_streamk", dict(bm=256, stages=6, cluster_m=2, split_k=0), 256, tgemm.F16),
    ("quad", dict(bm=256, stages=6, cluster_m=4), 256, tgemm.F16),
    ("quad_streamk", dict(bm=256, stages=6, cluster_m=4, split_k=0), 256, tgemm.F16),
    ("fp8_quad_streamk", dict(bm=256, stages=6, cluster_m=4, split_k=0), 256, tgemm.E4M3),
    ("tf32_pair", dict(bm=256, stages=6, cluster_m=2), 256, tgemm.F32),
    ("skinny_workspace", dict(bn=16, group_m=1, split_k=5, swap_ab=1), 16, tgemm.F16),
    ("skinny_cluster", dict(bn=16, stages=12, cluster_m=3, group_m=1, split_k=3, swap_ab=2), 16, tgemm.F16),
    ("skinny_cluster_half_ring", dict(bn=16, stages=6, cluster_m=8, group_m=1, split_k=8, swap_ab=2), 16,
     tgemm.F16),
    ("skinny_cluster_64", dict(bn=64, stages=9, cluster_m=7, group_m=1, split_k=7, swap_ab=2), 64, tgemm.BF16),
    ("skinny_cluster_128", dict(bn=128, stages=6, cluster_m=4, group_m=1, split_k=4, swap_ab=2), 100, tgemm.BF16),
    ("fp8_skinny_cluster", dict(bn=16, stages=6, cluster_m=4, group_m=1, split_k=4, swap_ab=2), 16, tgemm.E4M3),
    ("fp8_skinny_cluster_128", dict(bn=128, stages=6, cluster_m=2, group_m=1, split_k=2, swap_ab=2), 100,
     tgemm.E5M2),
]

ILLEGAL = [
    ("bk_32", dict(bk=32), 256, tgemm.F16),
    ("group_0", dict(group_m=0), 256, tgemm.F16),
    ("negative_grid", dict(grid=-1), 256, tgemm.F16),
    ("cta_split_2", dict(split_k=2), 256, tgemm.F16),
    ("cta_streamk", dict(split_k=0), 256, tgemm.F16),                      # stream-K: pair and quad only
    ("cta_stages_5", dict(stages=5), 256, tgemm.F16),                      # no such ring depth compiled
    ("cta256_stages_2", dict(stages=2), 256, tgemm.F16),                   # two stages: 128 x 128 only
    ("fp8_cta128_stages_2", dict(bn=128, stages=2), 256, tgemm.E4M3),      # and 16-bit operands only
    ("cluster_3_tiles", dict(bm=256, stages=6, cluster_m=3), 256, tgemm.F16),
    ("pair_bn_128", dict(bm=256, bn=128, stages=6, cluster_m=2), 256, tgemm.F16),
    ("cluster_8_tiles", dict(bm=256, stages=6, cluster_m=8), 256, tgemm.F16),   # no cluster-of-eight tile kernel
    ("workspace_stages", dict(bn=16, stages=6, group_m=1, split_k=5, swap_ab=1), 16, tgemm.F16),
    ("workspace_bn_below_m", dict(bn=16, group_m=1, split_k=5, swap_ab=1), 32, tgemm.F16),
    ("cluster_mismatch", dict(bn=16, stages=12, cluster_m=2, group_m=1, split_k=3, swap_ab=2), 16, tgemm.F16),
    ("cluster_9_splits", dict(bn=16, stages=12, cluster_m=9, group_m=1, split_k=9, swap_ab=2), 16, tgemm.F16),
    ("half_ring_64_x5", dict(bn=64, stages=4, cluster_m=5, group_m=1, split_k=5, swap_ab=2), 64, tgemm.F16),
    ("cluster_128_x5", dict(bn=128, stages=6, cluster_m=5, group_m=1, split_k=5, swap_ab=2), 100, tgemm.F16),
    ("cluster_128_half_ring", dict(bn=128, stages=3, cluster_m=2, group_m=1, split_k=2, swap_ab=2), 100, tgemm.F16),
    ("workspace_128", dict(bn=128, group_m=1, split_k=5, swap_ab=1), 100, tgemm.F16),
    ("cluster_129_rows", dict(bn=128, stages=6, cluster_m=4, group_m=1, split_k=4, swap_ab=2), 129, tgemm.F16),
    ("swap_3", dict(bn=16, group_m=1, split_k=5, swap_ab=3), 16, tgemm.F16),
    ("fp8_swap", dict(bn=16, group_m=1, split_k=5, swap_ab=1), 16, tgemm.E4M3),   # workspace kernel: 16-bit only
    ("tf32_swap", dict(bn=16, stages=6, cluster_m=4, group_m=1, split_k=4, swap_ab=2), 16, tgemm.F32),
    ("fp8_cluster_5_splits_128", dict(bn=128, stages=6, cluster_m=5, group_m=1, split_k=5, swap_ab=2), 100,
     tgemm.E4M3),
    ("fp8_cta_split", dict(split_k=2), 256, tgemm.E4M3),
]


def _run_forced(cfg, M, ind):
    # FAKE pointers: only ever run where no device answers, so that an
    # accepted configuration stops at the device query instead of launching
    import torch
    if torch.cuda.is_available():
        pytest.skip("host-path check with placeholder pointers; runs only without a GPU")
    N, K = 512, 1024
    return tgemm.tgemm_run_config(M, N, K, FAKE, K, FAKE, K, tgemm.B_NK, FAKE, N, ind, tgemm.BF16, None, cfg)


@pytest.mark.parametrize("name,kw,M,ind", LEGAL, ids=[c[0] for c in LEGAL])
def test_legal_configurations_pass_the_host_checks(lib, name, kw, M, ind):
    # accepted: the call gets past every configuration check to the device query
    assert _run_forced(_cfg(**kw), M, ind) in (tgemm.ERR_CUDA, tgemm.ERR_ARCH)


@pytest.mark.parametrize("name,kw,M,ind", ILLEGAL, ids=[c[0] for c in ILLEGAL])
def test_illegal_configurations_are_rejected_on_the_host(lib, name, kw, M, ind):
    assert _run_forced(_cfg(**kw), M, ind) == tgemm.ERR_UNSUPPORTED


@pytest.mark.parametrize("case,expect", [
    (dict(batch=-1), tgemm.ERR_INVALID_ARG),
    (dict(sa=-64), tgemm.ERR_INVALID_ARG),
    (dict(sa=100), tgemm.ERR_INVALID_ARG),          # A batches overlap (64 rows x 64 need 4096)
    (dict(sb=1000), tgemm.ERR_INVALID_ARG),         # B batches overlap
    (dict(sc=64), tgemm.ERR_INVALID_ARG),           # C batches overlap (C may not be shared)
    (dict(sc=0), tgemm.ERR_INVALID_ARG),
    (dict(sa=4100), tgemm.ERR_MISALIGNED),          # 8200 bytes: rows of later batches off 16 bytes
    (dict(sc=4100), tgemm.ERR_MISALIGNED),
    (dict(batch=1 << 31), tgemm.ERR_UNSUPPORTED),
])
def test_batched_argument_checks_on_the_host(lib, case, expect):
    a = dict(batch=3, sa=4096, sb=0, sc=4096)
    a.update(case)
    rc = tgemm.tgemm_run_strided_batched(a["batch"], 64, 64, 64, FAKE, 64, a["sa"], FAKE, 64, a["sb"], tgemm.B_NK,
                                         FAKE, 64, a["sc"], tgemm.BF16, tgemm.BF16, None, None, None)
    assert rc == expect, tgemm.status_string(rc)


def test_zero_batches_and_empty_products_need_no_device(lib):
    args = (64, 64, 64, FAKE, 64, 4096, FAKE, 64, 0, tgemm.B_NK, FAKE, 64, 4096, tgemm.BF16, tgemm.BF16, None,
            None, None)
    assert tgemm.tgemm_run_strided_batched(0, *args) == tgemm.OK
    assert tgemm.tgemm_run_strided_batched(3, 0, 64, 64, 0, 64, 0, 0, 64, 0, tgemm.B_NK, 0, 64, 0, tgemm.BF16,
                                           tgemm.BF16, None, None, None) == tgemm.OK


# ---- tile space and grouped order ---------------------------------------------

def coords(M, N, bm, bn, g):
    rc, _, _ = tgemm.tgemm_tile_coord(M, N, bm, bn, g, 0)
    assert rc == 0
    tm, tn = -(-M // bm), -(-N // bn)
    out = []
    for bid in range(tm * tn):
        rc, r, c = tgemm.tgemm_tile_coord(M, N, bm, bn, g, bid)
        assert rc == 0
        out.append((r, c))
    assert tgemm.tgemm_tile_coord(M, N, bm, bn, g, tm * tn)[0] == tgemm.ERR_INVALID_ARG
    return out


def test_tile_space_of_figure_19(lib):
    """CUDA Programming Guide 13.4.2, section 2.4.6.1, Figure 19."""
    g = read_golden("tile_space_fig19.txt")
    rows, cols = g["array_shape"]
    th, tw = g["tile_shape"]
    tiles = coords(rows, cols, th, tw, 1)
    assert len(tiles) == g["tile_grid"][0] * g["tile_grid"][1]
    assert max(r for r, _ in tiles) + 1 == g["tile_grid"][0]
    assert max(c for _, c in tiles) + 1 == g["tile_grid"][1]
    ti, tj = g["tile_index"]
    assert (ti, tj) in tiles
    first = (ti * th, tj * tw)
    last = (min(ti * th + th, rows) - 1, min(tj * tw + tw, cols) - 1)
    assert list(first) == g["first_element"] and list(last) == g["last_element"]


def test_grouped_order_reads_of_figure_2(lib):
    """cuTile tutorial, "Performance optimisation: Swizzle", Figure 2: the
    first four tiles in row order touch 4 + 16 blocks, grouped 2 x 2 order
    touches 8 + 8."""
    g = read_golden("swizzle_fig2.txt")
    gm, gn = g["grid"]
    kb = g["k_blocks"][0]
    n_out = g["outputs"][0]

    def reads(group):
        first = coords(gm, gn, 1, 1, group)[:n_out]
        left = {(r, k) for r, _ in first for k in range(kb)}
        right = {(k, c) for _, c in first for k in range(kb)}
        return len(left), len(right)

    assert reads(1) == (g["linear_left"][0], g["linear_right"][0])
    assert sum(reads(1)) == g["linear_reads"][0]
    assert reads(g["group_size_m"][0]) == (g["grouped_left"][0], g["grouped_right"][0])
    assert sum(reads(g["group_size_m"][0])) == g["grouped_reads"][0]


@pytest.mark.parametrize("group", [1, 2, 3, 4, 8, 16])
def test_grouped_order_is_a_bijection(lib, group):
    rng = np.random.default_rng(group)
    shapes = [(1, 1), (5, 2), (7, 3), (64, 32), (33, 17)] + [tuple(rng.integers(1, 40, 2)) for _ in range(6)]
    for tm, tn in shapes:
        tiles = coords(int(tm), int(tn), 1, 1, group)
        assert sorted(tiles) == [(r, c) for r in range(tm) for c in range(tn)]


def test_grouped_order_within_full_bands(lib):
    # In a full band, consecutive tile numbers walk down the band's rows first.
    tiles = coords(16 * 128, 4 * 256, 128, 256, 8)
    assert tiles[:10] == [(0, 0), (1, 0), (2, 0), (3, 0), (4, 0), (5, 0), (6, 0), (7, 0), (0, 1), (1, 1)]
    assert tiles[32] == (8, 0)


def test_last_short_band_uses_the_tile_number(lib):
    # 5 x 2 tiles, bands of 3 rows: the last band has 2 rows.  The row inside
    # the band comes from the tile number (6 % 2 = 0), giving (3, 0) for tile 6.
    tiles = coords(5, 2, 1, 1, 3)
    assert tiles[6] == (3, 0)
    assert tiles[7] == (4, 0)


LOG_SCRIPT = r"""
import sys
sys.path.insert(0, %r)
from dense_tiled_gemm_persistent_gb300 import tgemm
F = 1 << 20
tgemm.tgemm_run(-1, 96, 64, F, 64, F, 64, tgemm.B_NK, F, 96, tgemm.F16, tgemm.F16, None)
tgemm.tgemm_run(0, 96, 64, 0, 64, 0, 64, tgemm.B_KN, 0, 96, tgemm.BF16, tgemm.F32, None)
cfg = tgemm.Config(bm=128, bn=200, bk=64, stages=4, cluster_m=1, group_m=8, split_k=1, swap_ab=0, grid=0)
tgemm.tgemm_run_config(128, 96, 64, F, 64, F, 64, tgemm.B_NK, F, 96, tgemm.F16, tgemm.F16, None, cfg)
"""


@pytest.mark.parametrize("value,lines", [("1", 3), ("0", 0), (None, 0)])
def test_log_prints_one_line_per_call(lib, value, lines):
    """TGEMM_LOG (set, not "0") prints one stderr line per GEMM call: the
    problem, whose configuration it was, what was launched and the status."""
    import subprocess
    import sys
    env = dict(os.environ)
    env.pop("TGEMM_LOG", None)
    if value is not None:
        env["TGEMM_LOG"] = value
    r = subprocess.run([sys.executable, "-c", LOG_SCRIPT % ROOT], env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stderr
    got = [ln for ln in r.stderr.splitlines() if ln.startswith("tgemm: ")]
    assert len(got) == lines, r.stderr
    if lines:
        assert got[0].startswith("tgemm: tgemm_run batch=1 M=-1 N=96 K=64 B=NxK in=f16 out=f16 epilogue=0 "
                                 "config=library -> no kernel; invalid argument")
        assert got[1].startswith("tgemm: tgemm_run batch=1 M=0 N=96 K=64 B=KxN in=bf16 out=f32 epilogue=0 "
                                 "config=library -> no kernel; ok")
        assert "tgemm_run_config" in got[2] and "config=caller" in got[2] and got[2].endswith(
            "unsupported dtype, size or configuration")


def test_sm_clock_probe_checks_arguments_on_the_host(lib):
    assert tgemm.tgemm_debug_sm_clock(None, 20) == tgemm.ERR_INVALID_ARG
    assert tgemm.tgemm_debug_sm_clock(FAKE, 0) == tgemm.ERR_INVALID_ARG
    assert tgemm.tgemm_debug_sm_clock(FAKE, 100001) == tgemm.ERR_INVALID_ARG
    assert tgemm.tgemm_debug_sm_clock(FAKE + 4, 20) == tgemm.ERR_MISALIGNED


def test_clock_record_checks_alignment_on_the_host(lib):
    assert tgemm.tgemm_debug_clock_record(FAKE + 4) == tgemm.ERR_MISALIGNED
