"""GPU parity of FP32 operands multiplied as TF32 (B stored N x K) against the
FP64 oracle's TF32 reading: each element keeps sign, exponent and the top 10
fraction bits (the low 13 dropped), the products are summed in FP32.

Products of two TF32 values are exact in FP32 (at most 22 significant bits),
so against the oracle's sum of the same truncated values the only error is
the FP32 accumulation and the output rounding: the 16-bit cases' bound
    |C_gpu - C_ref| <= 1e-3 * sum_k |A_ik||B_kj| + ulp_out(C_ref)
holds unchanged.  Single-product and integer-valued cases are bit-exact; the
single-product case also pins the truncation reading on the hardware.
"""
import numpy as np
import pytest
import torch

import oracle
from dense_tiled_gemm_persistent_gb300 import inputs as gen
from dense_tiled_gemm_persistent_gb300 import tgemm

from gpu_util import assert_close, bits, ensure_built, round_up, sampled_points

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TF32 = oracle.TF32          # the oracle's name for FP32 storage read as TF32


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def C(**kw):
    base = dict(bm=128, bn=256, bk=64, stages=4, cluster_m=1, group_m=8, split_k=1, swap_ab=0, grid=0)
    base.update(kw)
    return tgemm.Config(**base)


CONFIGS = {
    "auto": None,
    "cta256": C(),
    "cta128": C(bn=128, stages=6),
    "pair": C(bm=256, stages=6, cluster_m=2),
    "pair_streamk": C(bm=256, stages=6, cluster_m=2, split_k=0),
    "quad": C(bm=256, stages=6, cluster_m=4),
    "quad_streamk": C(bm=256, stages=6, cluster_m=4, split_k=0),
}


def f32_operands(M, N, K, dist, seed, dist_b=None):
    """Seeded FP32 operands (B N x K), rows padded to 16 bytes with NaN."""
    return gen.make_operands(M, N, K, gen.F32, gen.B_NK, dist, dist_b, seed, lda=round_up(max(K, 1), 4),
                             ldb=round_up(max(K, 1), 4), pad_value=float("nan"))


def run(a, b, M, N, K, out_dtype, cfg=None, ep=None):
    A, B = a.to(DEV), b.to(DEV)
    ldc = round_up(max(N, 1), 16 // gen.DTYPE_SIZE[out_dtype])
    Cd = torch.full((max(M, 1), ldc), float("nan"), dtype=gen.TORCH_DTYPE[out_dtype], device=DEV)
    args = (M, N, K, A.data_ptr(), a.shape[1], B.data_ptr(), b.shape[1], gen.B_NK, Cd.data_ptr(), ldc, gen.F32,
            out_dtype, None)
    if ep is not None:
        rc = tgemm.tgemm_run_ex(*args, ep, cfg)
    elif cfg is None:
        rc = tgemm.tgemm_run(*args)
    else:
        rc = tgemm.tgemm_run_config(*args, cfg)
    assert rc == tgemm.OK, tgemm.status_string(rc)
    assert tgemm.tgemm_check() == tgemm.OK
    return Cd.cpu()


@pytest.mark.parametrize("name", sorted(CONFIGS))
def test_tf32_truncates_the_low_bits(name):
    """One product per output: C[i][j] = A[i][j mod K] * 1.  Full-mantissa A
    values in [1, 2) and [-2, -1) come back exactly as their TF32
    truncation (not rounded to nearest, not kept at FP32 precision)."""
    M, N, K = 300, 520, 72
    g = torch.Generator().manual_seed(21)
    a = (torch.rand(M, K, generator=g) + 1.0) * torch.where(torch.rand(M, K, generator=g) < 0.5, -1.0, 1.0)
    b = torch.zeros(N, K)
    b[torch.arange(N), torch.arange(N) % K] = 1.0
    out = run(a, b, M, N, K, gen.F32, CONFIGS[name])
    ref, _ = oracle.gemm(a, b, M, N, K, K, K, gen.B_NK, TF32)
    assert np.array_equal(bits(out[:M, :N], gen.F32), oracle.round_bits(ref, gen.F32))
    # and the truncation is visible: some inputs differ from their TF32 value
    assert (a.view(torch.int32) & 0x1FFF).ne(0).float().mean() > 0.99


@pytest.mark.parametrize("name", sorted(CONFIGS))
@pytest.mark.parametrize("out_dtype", [gen.F32, gen.BF16], ids=["f32", "bf16"])
def test_tf32_integers_bit_exact(name, out_dtype):
    M, N, K = 300, 520, 200
    a, b = f32_operands(M, N, K, gen.ints(-3, 3), seed=22)
    out = run(a, b, M, N, K, out_dtype, CONFIGS[name])
    ref, _ = oracle.gemm(a, b, M, N, K, a.shape[1], b.shape[1], gen.B_NK, TF32)
    got = bits(out[:M, :N], out_dtype)
    want = oracle.round_bits(ref, out_dtype)
    assert np.array_equal(got, want), "%d bit mismatches" % (got != want).sum()


@pytest.mark.parametrize("name", sorted(CONFIGS))
@pytest.mark.parametrize("out_dtype", [gen.F32, gen.F16, gen.BF16], ids=["f32", "f16", "bf16"])
def test_tf32_random_matches_oracle(name, out_dtype):
    M, N, K = 520, 777, 1036
    a, b = f32_operands(M, N, K, gen.normal(0, 1), seed=23, dist_b=gen.uniform(-2, 2))
    out = run(a, b, M, N, K, out_dtype, CONFIGS[name])
    ref, bound = oracle.gemm(a, b, M, N, K, a.shape[1], b.shape[1], gen.B_NK, TF32)
    assert_close(out[:M, :N].double().numpy(), ref, bound, out_dtype, name)


@pytest.mark.parametrize("M,N,K", [(1, 1, 4), (16, 4096, 4096), (64, 300, 2000), (129, 257, 4100),
                                   (1024, 1024, 16384)])
def test_tf32_shapes(M, N, K):
    a, b = f32_operands(M, N, K, gen.uniform(-1, 1), seed=24)
    out = run(a, b, M, N, K, gen.F32)
    if M * N * K <= 600 * 1000 * 1000:
        ref, bound = oracle.gemm(a, b, M, N, K, a.shape[1], b.shape[1], gen.B_NK, TF32)
        assert_close(out[:M, :N].double().numpy(), ref, bound, gen.F32)
    else:
        ii, jj = sampled_points(M, N, seed=6, n_random=2048)
        ref, bound = oracle.gemm_elements(a, b, M, N, K, a.shape[1], b.shape[1], gen.B_NK, TF32, ii, jj)
        assert_close(out[:M, :N].double().numpy()[ii, jj], ref, bound, gen.F32)


def test_tf32_epilogue_residual():
    """D = 0.5 * A*B + 1.0 * C_in, FP32 output, on the tile and pair kernels."""
    M, N, K = 300, 520, 1000
    a, b = f32_operands(M, N, K, gen.normal(0, 1), seed=25)
    g = torch.Generator().manual_seed(4)
    ldc = round_up(N, 4)
    cin = torch.randn(M, ldc, generator=g)
    cin_d = cin.to(DEV)
    ep = tgemm.Epilogue(alpha=0.5, beta=1.0, c_in=cin_d.data_ptr(), ldc_in=ldc, bias=None, bias_dtype=gen.F32,
                        act=tgemm.ACT_NONE)
    for name in ("cta256", "pair", "pair_streamk", "quad_streamk"):
        out = run(a, b, M, N, K, gen.F32, CONFIGS[name], ep=ep)
        acc, bound = oracle.gemm(a, b, M, N, K, a.shape[1], b.shape[1], gen.B_NK, TF32)
        c64 = cin[:, :N].double().numpy()
        want = oracle.epilogue(acc, alpha=0.5, beta=1.0, cin=c64)
        tol = 0.5 * 1e-3 * bound + 2.0 ** -20 * (np.abs(0.5 * acc) + np.abs(c64)) + oracle.ulp(want, gen.F32)
        err = np.abs(out[:M, :N].double().numpy() - want)
        assert (err <= tol).all(), "%s: max excess %g" % (name, float((err - tol).max()))


def test_tf32_strided_batched_shared_a():
    nb, M, N, K = 3, 200, 300, 100
    lda = ldb = round_up(K, 4)
    a = gen.make_operands(M, N, K, gen.F32, gen.B_NK, gen.ints(-4, 4), None, seed=26, lda=lda, ldb=ldb)[0]
    Bs = [gen.make_operands(M, N, K, gen.F32, gen.B_NK, gen.ints(-4, 4), None, seed=27 + i, lda=lda, ldb=ldb)[1]
          for i in range(nb)]
    A = a.to(DEV)
    B = torch.stack(Bs).to(DEV)
    ldc = round_up(N, 4)
    Cd = torch.full((nb, M, ldc), float("nan"), dtype=torch.float32, device=DEV)
    rc = tgemm.tgemm_run_strided_batched(nb, M, N, K, A.data_ptr(), lda, 0, B.data_ptr(), ldb, N * ldb, gen.B_NK,
                                         Cd.data_ptr(), ldc, M * ldc, gen.F32, gen.F32, None, None, None)
    assert rc == tgemm.OK, tgemm.status_string(rc)
    assert tgemm.tgemm_check() == tgemm.OK
    out = Cd.cpu()
    for i in range(nb):
        ref, _ = oracle.gemm(a, Bs[i], M, N, K, lda, ldb, gen.B_NK, TF32)
        assert np.array_equal(bits(out[i, :, :N], gen.F32), oracle.round_bits(ref, gen.F32)), "batch %d" % i


def test_tf32_rejections():
    M, N, K = 64, 64, 64
    A = torch.zeros((M, K + 4), dtype=torch.float32, device=DEV)
    B = torch.zeros((N, K), dtype=torch.float32, device=DEV)
    Cd = torch.zeros((M, N), dtype=torch.float32, device=DEV)

    def call(layout=gen.B_NK, lda=K, cfg=None):
        args = (M, N, K, A.data_ptr(), lda, B.data_ptr(), K, layout, Cd.data_ptr(), N, gen.F32, gen.F32, None)
        return tgemm.tgemm_run(*args) if cfg is None else tgemm.tgemm_run_config(*args, cfg)

    assert call(layout=gen.B_KN) == tgemm.ERR_UNSUPPORTED
    assert call(lda=K + 2) == tgemm.ERR_MISALIGNED                    # 264-byte rows
    assert call(cfg=C(bn=16, stages=4, group_m=1, split_k=2, swap_ab=1)) == tgemm.ERR_UNSUPPORTED
    assert call() == tgemm.OK and tgemm.tgemm_check() == tgemm.OK


def test_tf32_matmul_helper():
    a, b = f32_operands(130, 72, 40, gen.ints(-2, 2), seed=28)
    out = tgemm.matmul(a.to(DEV), b.to(DEV), gen.B_NK)
    assert out.dtype == torch.float32
    ref, _ = oracle.gemm(a, b, 130, 72, 40, a.shape[1], b.shape[1], gen.B_NK, TF32)
    assert np.array_equal(bits(out.cpu(), gen.F32), oracle.round_bits(ref, gen.F32))
