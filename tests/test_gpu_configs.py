"""GPU parity at the benchmark configuration's full sizes, in the launch
configuration tgemm_run picks (the one bench.py times).

Small problems are compared in full; the large ones on a seeded sample of
4096 outputs plus every element of the rows and columns at tile boundaries
(0, t-1, t, 2t-1, 2t, the first index of the last tile, the last index, for
row tile 128 and column tiles 64/128/256), each against the FP64 oracle with
|C_gpu - C_ref| <= 1e-3 * sum|A||B| + ulp_out(C_ref).
"""
import numpy as np
import pytest
import torch

import oracle
from dense_tiled_gemm_persistent_gb300 import inputs as gen
from dense_tiled_gemm_persistent_gb300 import tgemm

from gpu_util import assert_close, bits, ensure_built, operands, sampled_points

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def run_default(wl, a, b):
    A, B = a.to("cuda:0"), b.to("cuda:0")
    C = torch.empty((wl.M, wl.N), dtype=gen.TORCH_DTYPE[wl.out_dtype], device="cuda:0")
    rc = tgemm.tgemm_run(wl.M, wl.N, wl.K, A.data_ptr(), a.shape[1], B.data_ptr(), b.shape[1], wl.b_layout,
                         C.data_ptr(), wl.N, wl.in_dtype, wl.out_dtype, None)
    assert rc == 0, tgemm.status_string(rc)
    assert tgemm.tgemm_check() == 0
    return C


FULL = ["gemm_256x256x256_f16_kn_f32", "proj_16x4096x4096_bf16_nk_bf16", "proj_128x4096x4096_bf16_nk_bf16",
        "proj_16x4096x4096_e4m3_nk_bf16"]
SAMPLED = ["gemm_4000x3000x5000_bf16_nk_bf16", "gemm_4096x4096x4096_f16_kn_f16",
           "gemm_8192x8192x8192_f16_nk_f16", "proj_16384x14336x4096_bf16_nk_bf16",
           "gemm_8192x8192x8192_e4m3_nk_bf16", "gemm_8192x8192x8192_tf32_nk_f32", "gemm_8192x4864x1024_f16_nk_f16"]


def orc_in(wl):
    """The oracle's input code: FP32 operands are multiplied as TF32."""
    return oracle.TF32 if wl.in_dtype == gen.F32 else wl.in_dtype


@pytest.mark.parametrize("name", FULL)
def test_config_full_compare(name):
    wl = gen.WORKLOADS[name]
    a, b = wl.operands()
    C = run_default(wl, a, b).cpu()
    ref, bound = oracle.gemm(a, b, wl.M, wl.N, wl.K, a.shape[1], b.shape[1], wl.b_layout, wl.in_dtype)
    assert_close(C.double().numpy(), ref, bound, wl.out_dtype, name)


def test_config_256_integers_bit_exact():
    wl = gen.WORKLOADS["gemm_256x256x256_f16_kn_f32_ints"]
    a, b = wl.operands()
    C = run_default(wl, a, b).cpu()
    ref, _ = oracle.gemm(a, b, wl.M, wl.N, wl.K, a.shape[1], b.shape[1], wl.b_layout, wl.in_dtype)
    assert np.array_equal(bits(C, wl.out_dtype), oracle.round_bits(ref, wl.out_dtype))


@pytest.mark.parametrize("name", SAMPLED)
def test_config_sampled(name):
    wl = gen.WORKLOADS[name]
    a, b = wl.operands()
    C = run_default(wl, a, b)
    ii, jj = sampled_points(wl.M, wl.N, seed=wl.seed)
    got = C[torch.from_numpy(ii).to("cuda:0"), torch.from_numpy(jj).to("cuda:0")].double().cpu().numpy()
    ref, bound = oracle.gemm_elements(a, b, wl.M, wl.N, wl.K, a.shape[1], b.shape[1], wl.b_layout,
                                      orc_in(wl), ii, jj)
    assert len(ii) >= 4096
    assert_close(got, ref, bound, wl.out_dtype, name)
    # every boundary row/column of the sample is fully present
    assert set(gpu_boundary_rows(wl.M)).issubset(set(ii.tolist()))


def gpu_boundary_rows(M):
    from gpu_util import boundary_indices
    return boundary_indices(M, 128)


def test_taller_band_sampled():
    """16384 x 8192 x 8192 FP16: a shape whose default band of 8 tile rows the
    L2 footprint model makes 13 rows tall (bands 13, 13, 13, 13, 12 of the 64
    pair-tile rows), sampled against the oracle in tgemm_run's launch."""
    M, N, K = 16384, 8192, 8192
    rc, cfg = tgemm.tgemm_query_config(M, N, K, gen.B_NK, gen.F16, gen.F16)
    assert rc == 0 and cfg.cluster_m == 2 and cfg.group_m == 13
    a, b = operands(M, N, K, gen.F16, gen.B_NK, gen.uniform(-0.5, 0.5), seed=73)
    A, B = a.to("cuda:0"), b.to("cuda:0")
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda:0")
    rc = tgemm.tgemm_run(M, N, K, A.data_ptr(), a.shape[1], B.data_ptr(), b.shape[1], gen.B_NK, C.data_ptr(), N,
                         gen.F16, gen.F16, None)
    assert rc == 0 and tgemm.tgemm_check() == 0
    ii, jj = sampled_points(M, N, seed=73)
    got = C[torch.from_numpy(ii).to("cuda:0"), torch.from_numpy(jj).to("cuda:0")].double().cpu().numpy()
    ref, bound = oracle.gemm_elements(a, b, M, N, K, a.shape[1], b.shape[1], gen.B_NK, gen.F16, ii, jj)
    assert_close(got, ref, bound, gen.F16, "16384x8192x8192")
