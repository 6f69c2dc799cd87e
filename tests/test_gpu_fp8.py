"""GPU parity of FP8 operands (E4M3 "fn" and E5M2, B stored N x K) against the
FP64 oracle: the same defining sum C_ij = sum_k A_ik B_kj over the decoded
FP8 values, FP32 accumulation, FP16/BF16/FP32 output.

Every FP8 value is exact in FP32 and so is every product of two of them
(at most 4 + 4 significand bits), so the only error is the FP32 accumulation
and the output rounding: the bound of the 16-bit cases,
    |C_gpu - C_ref| <= 1e-3 * sum_k |A_ik||B_kj| + ulp_out(C_ref),
holds unchanged.  Integer-valued inputs give exact sums and are compared bit
for bit with the oracle's round-to-nearest-even of the exact result.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from dense_tiled_gemm_persistent_gb300 import inputs as gen
from dense_tiled_gemm_persistent_gb300 import tgemm

from gpu_util import assert_close, bits, ensure_built, round_up, sampled_points

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
FP8 = {"e4m3": gen.E4M3, "e5m2": gen.E5M2}


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


def fp8_operands(M, N, K, dt, dist, seed, dist_b=None):
    """Seeded FP8 operands, rows padded to 16 bytes (16 elements) with NaN."""
    return gen.make_operands(M, N, K, dt, gen.B_NK, dist, dist_b, seed, lda=round_up(max(K, 1), 16),
                             ldb=round_up(max(K, 1), 16), pad_value=float("nan"))


def run(a, b, M, N, K, dt, out_dtype, cfg=None, ep=None, c_fill=float("nan")):
    A, B = a.to(DEV), b.to(DEV)
    ldc = round_up(max(N, 1), 16 // gen.DTYPE_SIZE[out_dtype])
    Cd = torch.full((max(M, 1), ldc), c_fill, dtype=gen.TORCH_DTYPE[out_dtype], device=DEV)
    args = (M, N, K, A.data_ptr(), a.shape[1], B.data_ptr(), b.shape[1], gen.B_NK, Cd.data_ptr(), ldc, dt,
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
@pytest.mark.parametrize("fp8", sorted(FP8))
@pytest.mark.parametrize("out_dtype", [gen.F32, gen.BF16], ids=["f32", "bf16"])
def test_fp8_integers_bit_exact(name, fp8, out_dtype):
    # 300 x 520: ragged in both tile directions; K = 200: one full and one
    # ragged 128-element k-block, the rest read as zeros.
    dt = FP8[fp8]
    M, N, K = 300, 520, 200
    a, b = fp8_operands(M, N, K, dt, gen.ints(-3, 3), seed=11)
    out = run(a, b, M, N, K, dt, out_dtype, CONFIGS[name])
    ref, _ = oracle.gemm(a, b, M, N, K, a.shape[1], b.shape[1], gen.B_NK, dt)
    got = bits(out[:M, :N], out_dtype)
    want = oracle.round_bits(ref, out_dtype)
    assert np.array_equal(got, want), "%d bit mismatches" % (got != want).sum()


@pytest.mark.parametrize("name", sorted(CONFIGS))
@pytest.mark.parametrize("fp8", sorted(FP8))
@pytest.mark.parametrize("out_dtype", [gen.F32, gen.F16, gen.BF16], ids=["f32", "f16", "bf16"])
def test_fp8_random_matches_oracle(name, fp8, out_dtype):
    dt = FP8[fp8]
    M, N, K = 520, 777, 1040
    a, b = fp8_operands(M, N, K, dt, gen.normal(0, 1), seed=12, dist_b=gen.uniform(-2, 2))
    out = run(a, b, M, N, K, dt, out_dtype, CONFIGS[name])
    ref, bound = oracle.gemm(a, b, M, N, K, a.shape[1], b.shape[1], gen.B_NK, dt)
    assert_close(out[:M, :N].double().numpy(), ref, bound, out_dtype, "%s %s" % (name, fp8))


@pytest.mark.parametrize("name", ["pair_streamk", "quad_streamk"])
@pytest.mark.parametrize("fp8", sorted(FP8))
def test_fp8_stream_k_integers_bit_exact(name, fp8):
    # 1100 x 1300 with K = 3000 (24 k-blocks of 128 FP8 elements): enough
    # k-blocks that the tail is shared out by k-range on both kernels.
    dt = FP8[fp8]
    M, N, K = 1100, 1300, 3000
    a, b = fp8_operands(M, N, K, dt, gen.ints(-3, 3), seed=15)
    out = run(a, b, M, N, K, dt, gen.F32, CONFIGS[name])
    ref, _ = oracle.gemm(a, b, M, N, K, a.shape[1], b.shape[1], gen.B_NK, dt)
    got = bits(out[:M, :N], gen.F32)
    want = oracle.round_bits(ref, gen.F32)
    assert np.array_equal(got, want), "%d bit mismatches" % (got != want).sum()


@pytest.mark.parametrize("fp8", sorted(FP8))
@pytest.mark.parametrize("M,N,K", [(1, 1, 16), (16, 4096, 4096), (64, 300, 2000), (129, 257, 4112),
                                   (1024, 1024, 16384)])
def test_fp8_shapes(fp8, M, N, K):
    # M <= 128 goes to the in-cluster swap-AB kernel; the deep-K case is the
    # stream-K pick's home ground.
    dt = FP8[fp8]
    a, b = fp8_operands(M, N, K, dt, gen.uniform(-1, 1), seed=13)
    out = run(a, b, M, N, K, dt, gen.F32)
    if M * N * K <= 600 * 1000 * 1000:
        ref, bound = oracle.gemm(a, b, M, N, K, a.shape[1], b.shape[1], gen.B_NK, dt)
        assert_close(out[:M, :N].double().numpy(), ref, bound, gen.F32)
    else:
        ii, jj = sampled_points(M, N, seed=5, n_random=2048)
        ref, bound = oracle.gemm_elements(a, b, M, N, K, a.shape[1], b.shape[1], gen.B_NK, dt, ii, jj)
        assert_close(out[:M, :N].double().numpy()[ii, jj], ref, bound, gen.F32)


def test_fp8_scaled_epilogue_bias_gelu():
    # The usual FP8 recipe: per-tensor scales folded into alpha, then bias
    # and GELU, all fused into the store.
    dt = gen.E4M3
    M, N, K = 300, 520, 1000
    a, b = fp8_operands(M, N, K, dt, gen.normal(0, 2), seed=14)
    g = torch.Generator().manual_seed(3)
    bias = torch.randn(N, generator=g, dtype=torch.float32)
    bias_d = bias.to(DEV)
    alpha = 0.0625
    ep = tgemm.Epilogue(alpha=alpha, beta=0.0, c_in=None, ldc_in=0, bias=bias_d.data_ptr(), bias_dtype=gen.F32,
                        act=tgemm.ACT_GELU_TANH)
    for name in ("cta256", "pair", "pair_streamk", "quad_streamk"):
        out = run(a, b, M, N, K, dt, gen.BF16, CONFIGS[name], ep=ep)
        ref, bound = oracle.gemm(a, b, M, N, K, a.shape[1], b.shape[1], gen.B_NK, dt)
        want = oracle.epilogue(ref, alpha=alpha, bias=bias.double().numpy(), act=oracle.ACT_GELU_TANH)
        tol_src = 1.13 * (abs(alpha) * 1e-3 * bound + 2.0 ** -20 * (np.abs(alpha * ref) + np.abs(bias.numpy())))
        err = np.abs(out[:M, :N].double().numpy() - want)
        lim = tol_src + oracle.ulp(want, gen.BF16)
        assert (err <= lim).all(), "%s: max excess %g" % (name, float((err - lim).max()))


@pytest.mark.parametrize("fp8", sorted(FP8))
def test_fp8_strided_batched_shared_b(fp8):
    dt = FP8[fp8]
    nb, M, N, K = 3, 200, 300, 272
    lda = ldb = round_up(K, 16)
    As = [gen.make_operands(M, N, K, dt, gen.B_NK, gen.ints(-4, 4), None, seed=20 + i, lda=lda, ldb=ldb)[0]
          for i in range(nb)]
    b = gen.make_operands(M, N, K, dt, gen.B_NK, gen.ints(-4, 4), None, seed=30, lda=lda, ldb=ldb)[1]
    A = torch.stack(As).to(DEV)
    B = b.to(DEV)
    ldc = round_up(N, 4)
    Cd = torch.full((nb, M, ldc), float("nan"), dtype=torch.float32, device=DEV)
    rc = tgemm.tgemm_run_strided_batched(nb, M, N, K, A.data_ptr(), lda, M * lda, B.data_ptr(), ldb, 0, gen.B_NK,
                                         Cd.data_ptr(), ldc, M * ldc, dt, gen.F32, None, None, None)
    assert rc == tgemm.OK, tgemm.status_string(rc)
    assert tgemm.tgemm_check() == tgemm.OK
    out = Cd.cpu()
    for i in range(nb):
        ref, _ = oracle.gemm(As[i], b, M, N, K, lda, ldb, gen.B_NK, dt)
        assert np.array_equal(bits(out[i, :, :N], gen.F32), oracle.round_bits(ref, gen.F32)), "batch %d" % i


def test_fp8_rejections():
    dt = gen.E4M3
    M, N, K = 64, 64, 64
    A = torch.zeros((M, K + 16), dtype=torch.float8_e4m3fn, device=DEV)
    B = torch.zeros((N, K), dtype=torch.float8_e4m3fn, device=DEV)
    Cd = torch.zeros((M, N), dtype=torch.float32, device=DEV)

    def call(layout=gen.B_NK, lda=K, cfg=None, out=gen.F32):
        args = (M, N, K, A.data_ptr(), lda, B.data_ptr(), K, layout, Cd.data_ptr(), N, dt, out, None)
        return tgemm.tgemm_run(*args) if cfg is None else tgemm.tgemm_run_config(*args, cfg)

    assert call(layout=gen.B_KN) == tgemm.ERR_UNSUPPORTED            # FP8 B must be K-major
    assert call(lda=K + 8) == tgemm.ERR_MISALIGNED                    # 72-byte rows
    skinny = C(bn=16, stages=4, group_m=1, split_k=2, swap_ab=1)
    assert call(cfg=skinny) == tgemm.ERR_UNSUPPORTED                  # the workspace reduction is 16-bit only
    assert call(cfg=C(bn=128, stages=4)) == tgemm.ERR_UNSUPPORTED     # no such FP8 instantiation
    cfg = tgemm.Config()
    assert tgemm.load().tgemm_query_config(16, 4096, 4096, gen.B_NK, dt, gen.BF16, ctypes.byref(cfg)) == 0
    assert cfg.swap_ab == 2 and cfg.bn == 16                          # the in-cluster swap-AB kernel
    assert tgemm.load().tgemm_query_config(16, 4096, 4096, gen.B_KN, dt, gen.BF16, ctypes.byref(cfg)) == \
        tgemm.ERR_UNSUPPORTED
    # noalloc entry: 16-bit operands only
    rc = tgemm.tgemm_run_noalloc(M, N, K, A.data_ptr(), K, B.data_ptr(), K, gen.B_NK, Cd.data_ptr(), N, dt,
                                 gen.F32, None)
    assert rc == tgemm.ERR_UNSUPPORTED
    assert tgemm.tgemm_check() == tgemm.OK


def test_fp8_matmul_helper_defaults_to_bf16():
    a, b = fp8_operands(130, 72, 48, gen.E5M2, gen.ints(-2, 2), seed=40)
    out = tgemm.matmul(a.to(DEV), b.to(DEV), gen.B_NK)
    assert out.dtype == torch.bfloat16
    ref, _ = oracle.gemm(a, b, 130, 72, 48, a.shape[1], b.shape[1], gen.B_NK, gen.E5M2)
    assert np.array_equal(bits(out.cpu(), gen.BF16), oracle.round_bits(ref, gen.BF16))


# ---- few rows of A: the in-cluster swap-AB split-K kernel (kind::f8f6f4) ----

CLUSTER_STAGES = {16: 12, 32: 10, 64: 9, 128: 6}
CLUSTER_MAX_SPLITS = {16: 8, 32: 8, 64: 7, 128: 4}
HALF_STAGES = {16: 6, 32: 5, 64: 4}
HALF_MAX_SPLITS = {16: 8, 32: 7, 64: 4}


def cluster_cfg(npad, splits, half=False):
    return C(bm=128, bn=npad, stages=(HALF_STAGES if half else CLUSTER_STAGES)[npad], cluster_m=splits, group_m=1,
             split_k=splits, swap_ab=2)


@pytest.mark.parametrize("npad,half", [(16, False), (16, True), (32, False), (32, True), (64, False), (64, True),
                                       (128, False)], ids=lambda v: str(v))
@pytest.mark.parametrize("fp8", sorted(FP8))
def test_fp8_cluster_split_k_integers_exact(npad, half, fp8):
    """Every legal cluster size (first, second, middle, last), 8 ragged
    128-element k-blocks, ragged N: bit-exact against the oracle."""
    dt = FP8[fp8]
    M, N, K = (100 if npad == 128 else min(npad, 40)), 700, 1000
    a, b = fp8_operands(M, N, K, dt, gen.ints(-3, 3), seed=61 + npad)
    ref, _ = oracle.gemm(a, b, M, N, K, a.shape[1], b.shape[1], gen.B_NK, dt)
    top = (HALF_MAX_SPLITS if half else CLUSTER_MAX_SPLITS)[npad]
    for splits in sorted({1, 2, (top + 1) // 2, top}):
        for out_dtype in (gen.F32, gen.BF16):
            out = run(a, b, M, N, K, dt, out_dtype, cluster_cfg(npad, splits, half))
            got = bits(out[:M, :N], out_dtype)
            want = oracle.round_bits(ref, out_dtype)
            assert np.array_equal(got, want), "splits=%d out=%d: %d bit mismatches" % (
                splits, out_dtype, (got != want).sum())


@pytest.mark.parametrize("splits", [2, 4])
def test_fp8_cluster_split_k_one_k_block_per_cta(splits):
    dt = gen.E4M3
    M, N = 16, 384
    for K in (128 * splits, 128 * splits + 48):
        a, b = fp8_operands(M, N, K, dt, gen.ints(-3, 3), seed=67 + K)
        out = run(a, b, M, N, K, dt, gen.F32, cluster_cfg(16, splits, True))
        ref, _ = oracle.gemm(a, b, M, N, K, a.shape[1], b.shape[1], gen.B_NK, dt)
        assert np.array_equal(bits(out[:M, :N], gen.F32), oracle.round_bits(ref, gen.F32)), "K=%d" % K


@pytest.mark.parametrize("fp8", sorted(FP8))
@pytest.mark.parametrize("M", [1, 7, 16, 33, 64, 100, 128])
def test_fp8_skinny_default_pick_matches_oracle(fp8, M):
    dt = FP8[fp8]
    N, K = 4096, 4096
    cfg = tgemm.Config()
    assert tgemm.load().tgemm_query_config(M, N, K, gen.B_NK, dt, gen.BF16, ctypes.byref(cfg)) == 0
    assert cfg.swap_ab == 2
    a, b = fp8_operands(M, N, K, dt, gen.normal(0, 1), seed=70 + M, dist_b=gen.uniform(-1, 1))
    for out_dtype in (gen.BF16, gen.F32):
        out = run(a, b, M, N, K, dt, out_dtype)
        ref, bound = oracle.gemm(a, b, M, N, K, a.shape[1], b.shape[1], gen.B_NK, dt)
        assert_close(out[:M, :N].double().numpy(), ref, bound, out_dtype, "M=%d %s" % (M, fp8))


def test_fp8_cluster_split_k_with_fused_epilogue():
    """alpha, beta * C_in, bias and GELU applied by the owning ranks."""
    dt = gen.E4M3
    M, N, K = 24, 1000, 2048
    a, b = fp8_operands(M, N, K, dt, gen.normal(0, 1), seed=73, dist_b=gen.uniform(-1, 1))
    g = torch.Generator().manual_seed(74)
    bias = torch.randn(N, generator=g).to(torch.bfloat16)
    ldc = round_up(N, 8)
    cin = torch.randn(M, ldc, generator=g).to(torch.bfloat16)
    cin_d, bias_d = cin.to(DEV), bias.to(DEV)
    alpha, beta, act = 0.5, -1.0, tgemm.ACT_GELU_TANH
    ep = tgemm.Epilogue(alpha=alpha, beta=beta, c_in=cin_d.data_ptr(), ldc_in=ldc, bias=bias_d.data_ptr(),
                        bias_dtype=gen.BF16, act=act)
    out = run(a, b, M, N, K, dt, gen.BF16, cluster_cfg(32, 4), ep=ep)
    acc, bound = oracle.gemm(a, b, M, N, K, a.shape[1], b.shape[1], gen.B_NK, dt)
    cin64, bias64 = cin[:, :N].double().numpy(), bias.double().numpy()
    want = oracle.epilogue(acc, alpha, beta, cin64, bias64, act)
    mag = np.abs(alpha * acc) + np.abs(beta * cin64) + np.abs(bias64)[None, :]
    tol = 1.13 * (abs(alpha) * 1e-3 * bound + 2.0 ** -20 * mag) + oracle.ulp(want, gen.BF16)
    err = np.abs(out[:M, :N].double().numpy() - want)
    assert (err <= tol).all(), "max excess %g" % float((err - tol).max())
