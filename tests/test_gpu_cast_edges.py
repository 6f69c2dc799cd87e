"""Bit-exact GPU tests of the FP32 -> FP16/BF16 output cast's edge cases, on
every kernel family that casts in its own code.

The cast is round-to-nearest-even with overflow to +-Inf (the reading of the
pages' `astype`: the cuTile tutorial's kernel walk-through and the CUDA
Programming Guide 13.4.2, section 2.4.9.1).  The operands come from
`inputs.cast_edge_operands`: every partial sum is exact in FP32 in any
order, so the kernel's result equals the oracle's exact sum rounded once,
bit for bit, and the outputs land on
  * FP16's largest finite value 65504, the tie at 65520 that rounds to
    infinity, and sums beyond it (FP16 inputs);
  * FP16 subnormals, half of them exactly half-way between two (FP16 inputs);
  * BF16's largest finite value, its tie to infinity and sums beyond it, up
    to just below FP32's largest finite value (BF16 inputs).
Each family rounds in its own code: the 1-CTA, pair and quad tile epilogues,
the pair and quad stream-K fix-ups, both swap-AB split-K reductions, the
fused epilogue (alpha scaling in FP32 before the cast) and the epilogue-only
kernel (K = 0).
"""
import numpy as np
import pytest
import torch

import oracle
from dense_tiled_gemm_persistent_gb300 import inputs as gen
from dense_tiled_gemm_persistent_gb300 import tgemm

from gpu_util import bits, ensure_built, round_up, run_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def C(**kw):
    base = dict(bm=128, bn=256, bk=64, stages=4, cluster_m=1, group_m=8, split_k=1, swap_ab=0, grid=0)
    base.update(kw)
    return tgemm.Config(**base)


# family -> (configuration, M, N, K)
FAMILIES = {
    "cta256": (C(), 300, 520, 1500),
    "cta128": (C(bn=128, stages=6), 300, 520, 1500),
    "cta128_2stage": (C(bn=128, stages=2), 300, 520, 1500),
    "pair": (C(bm=256, stages=6, cluster_m=2), 300, 520, 1500),
    "quad": (C(bm=256, stages=6, cluster_m=4), 300, 1100, 1500),
    # 5 x 6 pair tiles on 7 pairs: the 2 leftover tiles are shared by k-range
    "pair_streamk": (C(bm=256, stages=6, cluster_m=2, split_k=0, grid=14), 1100, 1300, 1500),
    # 5 x 3 quad blocks on 2 quads: the leftover block is shared by k-range
    "quad_streamk": (C(bm=256, stages=6, cluster_m=4, split_k=0, grid=8), 1100, 1300, 1500),
    "skinny_workspace": (C(bn=16, stages=4, group_m=1, split_k=4, swap_ab=1), 16, 640, 2048),
    "skinny_cluster": (C(bn=16, stages=12, cluster_m=4, group_m=1, split_k=4, swap_ab=2), 16, 640, 2048),
}


def check_exact(kind, family, layout, seed):
    cfg, M, N, K = FAMILIES[family]
    ind, outd = gen.cast_edge_in_dtype(kind), gen.cast_edge_out_dtype(kind)
    b_cols = N if layout == gen.B_KN else K
    a, b = gen.cast_edge_operands(kind, M, N, K, layout, seed, lda=round_up(K, 8), ldb=round_up(b_cols, 8))
    Cg = run_gpu(a, b, M, N, K, layout, ind, outd, config=cfg)
    ref, _ = oracle.gemm(a, b, M, N, K, a.shape[1], b.shape[1], layout, ind)
    want = oracle.round_bits(ref, outd)
    got = bits(Cg[:M, :N], outd)
    mism = got != want
    assert not mism.any(), "%s %s: %d of %d differ, first at %s: got 0x%04x, oracle 0x%04x (exact sum %r)" % (
        kind, family, mism.sum(), mism.size, tuple(np.argwhere(mism)[0]), got[mism][0], want[mism][0],
        ref[mism][0])
    return oracle.decode(want, outd)


@pytest.mark.parametrize("family", sorted(FAMILIES))
@pytest.mark.parametrize("kind", gen.CAST_EDGE_KINDS)
@pytest.mark.parametrize("layout", [gen.B_NK, gen.B_KN], ids=["nk", "kn"])
def test_cast_edges_bit_exact(family, kind, layout):
    vals = check_exact(kind, family, layout, seed=101 + len(family))
    # the case must exercise what it is named for
    if kind.endswith("overflow"):
        assert np.isinf(vals).any() and np.isfinite(vals).any()
    else:
        assert ((np.abs(vals) < 2.0 ** -14) & (vals != 0)).any()


EPI_FAMILIES = {
    "cta256": FAMILIES["cta256"],
    "pair": FAMILIES["pair"],
    "quad_streamk": FAMILIES["quad_streamk"],
    "skinny_cluster": FAMILIES["skinny_cluster"],
    "skinny_workspace": FAMILIES["skinny_workspace"],
}


@pytest.mark.parametrize("family", sorted(EPI_FAMILIES))
def test_fused_epilogue_scales_then_casts_to_inf(family):
    """alpha = 0.5 on sums of twice the size: 0.5 * (130944 + 8c) is exact in
    FP32 and lands on 65504, the tie at 65520 and beyond; one cast after the
    scaling, so the bits equal the oracle's epilogue rounded once."""
    cfg, M, N, K = EPI_FAMILIES[family]
    a, b = gen.cast_edge_operands("f16_overflow", M, N, K, gen.B_NK, seed=7, scale=2, lda=round_up(K, 8),
                                  ldb=round_up(K, 8))
    A, B = a.to(DEV), b.to(DEV)
    ldc = round_up(N, 8)
    Cd = torch.full((M, ldc), float("nan"), dtype=torch.float16, device=DEV)
    ep = tgemm.Epilogue(alpha=0.5, beta=0.0, c_in=None, ldc_in=ldc, bias=None, bias_dtype=gen.F32,
                        act=tgemm.ACT_NONE)
    rc = tgemm.tgemm_run_ex(M, N, K, A.data_ptr(), A.shape[1], B.data_ptr(), B.shape[1], gen.B_NK, Cd.data_ptr(),
                            ldc, gen.F16, gen.F16, None, ep, cfg)
    assert rc == 0, tgemm.status_string(rc)
    assert tgemm.tgemm_check() == 0
    acc, _ = oracle.gemm(a, b, M, N, K, a.shape[1], b.shape[1], gen.B_NK, gen.F16)
    want = oracle.round_bits(oracle.epilogue(acc, alpha=0.5), gen.F16)
    got = bits(Cd[:, :N].cpu(), gen.F16)
    assert np.array_equal(got, want), "%s: %d differ" % (family, (got != want).sum())
    v = oracle.decode(want, gen.F16)
    assert np.isinf(v).any() and (np.abs(v) == 65504).any()


def epilogue_only_inputs(out_dtype, M, N, seed=5):
    """C_in holds +-(the format's largest finite value), +-(the one below it)
    and, for FP16, +-5 times the smallest subnormal; the bias by column is 0,
    a quarter, just under a half, exactly a half or a whole spacing of the
    format's top binade (subnormals only in columns without bias).  Every
    sum is exact in FP32 or, for BF16's largest value plus a whole spacing
    (2^128), overflows FP32 to the infinity that BF16 rounds it to anyway."""
    tdt = gen.TORCH_DTYPE[out_dtype]
    big = float(torch.finfo(tdt).max)
    top = big - float(torch.tensor(big, dtype=tdt).nextafter(torch.tensor(0.0, dtype=tdt)))
    tiny = 5 * 2.0 ** -24 if out_dtype == gen.F16 else 0.0
    g = torch.Generator().manual_seed(seed)
    pick = torch.randint(0, 3, (M, N), generator=g)
    signs = torch.where(torch.rand((M, N), generator=g) < 0.5, -1.0, 1.0).double()
    pick = torch.where((torch.arange(N) % 5 == 0)[None, :], pick, pick % 2)   # subnormals only where bias = 0
    cin64 = torch.where(pick == 0, big, torch.where(pick == 1, big - top, tiny)).double() * signs
    cin = cin64.to(tdt)
    assert torch.equal(cin.double(), cin64)
    steps = torch.tensor([0.0, 0.25, 0.5 - 2.0 ** -10, 0.5, 1.0], dtype=torch.float64)
    bias64 = steps[torch.arange(N) % 5] * top
    bias = bias64.to(torch.float32)
    assert torch.equal(bias.double(), bias64)
    return cin, bias


@pytest.mark.parametrize("out_dtype", [gen.F16, gen.BF16], ids=["o16", "obf16"])
@pytest.mark.parametrize("beta", [1.0, 0.5])
def test_epilogue_only_kernel_cast_edges(out_dtype, beta):
    """K = 0: D = beta * C_in + bias, evaluated in FP32 and cast once.  With
    beta = 1 the bias pushes the largest finite values onto and past the tie
    that rounds to infinity; with beta = 0.5 the FP16 subnormals in columns
    without bias land half-way between two subnormals."""
    M, N = 64, 96
    tdt = gen.TORCH_DTYPE[out_dtype]
    cin, bias = epilogue_only_inputs(out_dtype, M, N)
    Cd = torch.full((M, N), float("nan"), dtype=tdt, device=DEV)
    cin_d, bias_d = cin.to(DEV), bias.to(DEV)
    ep = tgemm.Epilogue(alpha=1.0, beta=beta, c_in=cin_d.data_ptr(), ldc_in=N, bias=bias_d.data_ptr(),
                        bias_dtype=gen.F32, act=tgemm.ACT_NONE)
    x = torch.empty(16, dtype=torch.float16, device=DEV)
    rc = tgemm.tgemm_run_ex(M, N, 0, x.data_ptr(), 8, x.data_ptr(), 8, gen.B_NK, Cd.data_ptr(), N, gen.F16,
                            out_dtype, None, ep, None)
    assert rc == 0 and tgemm.tgemm_check() == 0
    ref = oracle.epilogue(np.zeros((M, N)), 1.0, beta, cin.double().numpy(), bias.double().numpy(),
                          oracle.ACT_NONE)
    # every term and sum is exact in FP32, so one rounding of the exact value is the answer
    want = oracle.round_bits(ref, out_dtype)
    got = bits(Cd.cpu(), out_dtype)
    assert np.array_equal(got, want), "beta=%g: %d differ" % (beta, (got != want).sum())
    v = oracle.decode(want, out_dtype)
    if beta == 1.0:
        assert np.isinf(v).any() and np.isfinite(v).any()
    elif out_dtype == gen.F16:
        assert ((np.abs(v) < 2.0 ** -14) & (v != 0)).any()
