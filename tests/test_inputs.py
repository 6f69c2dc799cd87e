"""The seeded operand generator and the named workloads (no GPU needed).

The generator holds no product arithmetic; these tests pin its recipe (draw
order, distributions, rounding, padding) and check that every named workload
carries the shape, types, layout, values, seed, FLOP count and algorithmic
byte count of the benchmark configuration it stands for.
"""
import math

import numpy as np
import pytest
import torch

from dense_tiled_gemm_persistent_gb300 import inputs as gen


def test_recipe_draws_a_first_then_b_in_storage_orientation():
    M, N, K = 5, 7, 3
    for layout, b_shape in ((gen.B_KN, (K, N)), (gen.B_NK, (N, K))):
        a, b = gen.make_operands(M, N, K, gen.F32, layout, gen.uniform(-1, 1), gen.normal(0, 2), seed=123)
        g = torch.Generator("cpu").manual_seed(123)
        a_ref = -1 + 2 * torch.rand((M, K), generator=g, dtype=torch.float32)
        b_ref = 0 + 2 * torch.randn(b_shape, generator=g, dtype=torch.float32)
        assert torch.equal(a, a_ref) and torch.equal(b, b_ref)


def test_same_seed_same_operands_other_seed_other_operands():
    args = (64, 48, 32, gen.BF16, gen.B_NK, gen.normal(0, 1), None)
    a1, b1 = gen.make_operands(*args, seed=4)
    a2, b2 = gen.make_operands(*args, seed=4)
    a3, _ = gen.make_operands(*args, seed=5)
    assert torch.equal(a1, a2) and torch.equal(b1, b2) and not torch.equal(a1, a3)


def test_distributions_stay_in_their_support():
    g = torch.Generator("cpu").manual_seed(0)
    u = gen.uniform(-0.5, 0.5).draw((200000,), g)
    assert u.min() >= -0.5 and u.max() < 0.5 and abs(float(u.mean())) < 0.01
    n = gen.normal(0, 0.02).draw((200000,), g)
    assert abs(float(n.mean())) < 0.001 and abs(float(n.std()) - 0.02) < 0.001
    i = gen.ints(-2, 2).draw((10000,), g)
    assert set(i.unique().tolist()) == {-2.0, -1.0, 0.0, 1.0, 2.0}


def test_rounding_to_the_operand_type_is_round_to_nearest_even():
    a, _ = gen.make_operands(16, 16, 16, gen.F16, gen.B_NK, gen.normal(0, 1), None, seed=9)
    g = torch.Generator("cpu").manual_seed(9)
    raw = torch.randn((16, 16), generator=g, dtype=torch.float32)
    assert a.dtype == torch.float16
    assert np.array_equal(a.numpy(), raw.numpy().astype(np.float16))   # numpy's cast is RNE


def test_leading_dimension_pads_rows_with_poison_only():
    a, b = gen.make_operands(4, 6, 5, gen.F16, gen.B_KN, gen.ints(-2, 2), None, seed=1, lda=8, ldb=16)
    assert a.shape == (4, 8) and b.shape == (5, 16)
    assert torch.isnan(a[:, 5:]).all() and not torch.isnan(a[:, :5]).any()
    assert torch.isnan(b[:, 6:]).all() and not torch.isnan(b[:, :6]).any()


def test_logical_b_is_a_view_of_the_stored_one():
    N, K = 6, 4
    _, b_nk = gen.make_operands(3, N, K, gen.F32, gen.B_NK, gen.uniform(-1, 1), None, seed=2)
    assert torch.equal(gen.b_logical(b_nk, N, K, gen.B_NK), b_nk.t())
    _, b_kn = gen.make_operands(3, N, K, gen.F32, gen.B_KN, gen.uniform(-1, 1), None, seed=2)
    assert torch.equal(gen.b_logical(b_kn, N, K, gen.B_KN), b_kn)


# name: (M, N, K, in, out, layout, A values, B values, seed, algorithmic bytes)
CONFIGS = {
    "gemm_256x256x256_f16_kn_f32": (256, 256, 256, gen.F16, gen.F32, gen.B_KN, "uniform[-1,1)", "uniform[-1,1)", 0,
                                    524_288),
    "gemm_256x256x256_f16_kn_f32_ints": (256, 256, 256, gen.F16, gen.F32, gen.B_KN, "ints{-2..2}", "ints{-2..2}", 0,
                                         524_288),
    "gemm_4000x3000x5000_bf16_nk_bf16": (4000, 3000, 5000, gen.BF16, gen.BF16, gen.B_NK, "normal(0,1)",
                                         "normal(0,1)", 1, 94_000_000),
    "gemm_4096x4096x4096_f16_kn_f16": (4096, 4096, 4096, gen.F16, gen.F16, gen.B_KN, "uniform[-1,1)",
                                       "uniform[-1,1)", 2, 100_663_296),
    "gemm_8192x8192x8192_f16_nk_f16": (8192, 8192, 8192, gen.F16, gen.F16, gen.B_NK, "uniform[-0.5,0.5)",
                                       "uniform[-0.5,0.5)", 3, 402_653_184),
    "proj_16384x14336x4096_bf16_nk_bf16": (16384, 14336, 4096, gen.BF16, gen.BF16, gen.B_NK, "normal(0,1)",
                                           "normal(0,0.02)", 4, 721_420_288),
    "proj_16x4096x4096_bf16_nk_bf16": (16, 4096, 4096, gen.BF16, gen.BF16, gen.B_NK, "normal(0,1)",
                                       "normal(0,0.02)", 4, 33_816_576),
}


def test_named_workloads_match_the_benchmark_configuration():
    for name, (M, N, K, ti, to, layout, da, db, seed, nbytes) in CONFIGS.items():
        w = gen.WORKLOADS[name]
        assert (w.M, w.N, w.K, w.in_dtype, w.out_dtype, w.b_layout, w.seed) == (M, N, K, ti, to, layout, seed), name
        assert (w.dist_a.describe(), w.dist_b.describe()) == (da, db), name
        assert w.flops == 2 * M * N * K
        assert w.algorithmic_bytes == nbytes, name


def test_arithmetic_intensity_classes():
    # ridge of the measured peaks: 1921.8 TFLOP/s / 6766 GB/s = 284 FLOP/B; only
    # the 16-token projection is below it (HBM-bound)
    ridge = 1921.8e12 / 6766e9
    for name, w in gen.WORKLOADS.items():
        ai = w.flops / w.algorithmic_bytes
        if name.startswith("gemm_256x"):
            assert math.isclose(ai, 64.0)          # launch-latency bound, reported only
        elif name == "proj_16x4096x4096_bf16_nk_bf16":
            assert 15 < ai < 16 and ai < ridge
        elif name == "proj_128x4096x4096_bf16_nk_bf16":
            assert 110 < ai < 125 and ai < ridge       # 128 tokens: still below the ridge
        elif name == "proj_16x4096x4096_e4m3_nk_bf16":
            assert 30 < ai < 32 and ai < ridge         # one byte per weight: twice the FLOP per byte
        else:
            assert ai > ridge, name


@pytest.mark.parametrize("kind", gen.CAST_EDGE_KINDS)
@pytest.mark.parametrize("layout", [gen.B_NK, gen.B_KN])
def test_cast_edge_operands_land_on_the_edges(orc, kind, layout):
    """The cast-edge operands are exact in their input type, and the oracle's
    exact sums round onto the edges they are named for."""
    import numpy as np
    M, N, K = 24, 40, 700
    a, b = gen.cast_edge_operands(kind, M, N, K, layout, seed=1)
    ind, outd = gen.cast_edge_in_dtype(kind), gen.cast_edge_out_dtype(kind)
    assert a.dtype == gen.TORCH_DTYPE[ind] and b.dtype == gen.TORCH_DTYPE[ind]
    ref, _ = orc.gemm(a, b, M, N, K, a.shape[1], b.shape[1], layout, ind)
    v = orc.decode(orc.round_bits(ref, outd), outd)
    if kind == "f16_overflow":
        assert set(np.unique(np.abs(v))) <= {65472.0, 65504.0, np.inf}
        assert np.isinf(v).any() and (np.abs(v) == 65504).any() and (np.abs(ref) == 65520).any()
    elif kind == "bf16_overflow":
        top = 255 * 2.0 ** 120
        assert set(np.unique(np.abs(v))) <= {top, np.inf}
        assert np.isinf(v).any() and (np.abs(v) == top).any()
        assert np.abs(ref).max() < (2 - 2.0 ** -23) * 2.0 ** 127          # FP32 never overflows
    else:
        sub = (np.abs(v) < 2.0 ** -14) & (v != 0)
        assert sub.mean() > 0.5
        assert ((np.abs(ref) / 2.0 ** -25) % 2 == 1).any()               # half-way cases
    # columns alternate in sign for the overflow kinds
    if kind != "f16_subnormal":
        assert (np.sign(ref[:, 0::2]) > 0).all() and (np.sign(ref[:, 1::2]) < 0).all()
