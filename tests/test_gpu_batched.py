"""GPU parity of the strided-batched GEMM: every batch against the oracle's
defining sum on that batch's slices (the batched form of section 2.4.9.1 of
the CUDA Programming Guide 13.4.2, unofficial Chinese translation)."""
import numpy as np
import pytest
import torch

import oracle
from dense_tiled_gemm_persistent_gb300 import inputs as gen
from dense_tiled_gemm_persistent_gb300 import tgemm

from gpu_util import assert_close, bits, ensure_built, round_up

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


CONFIGS = {
    "auto": None,
    "cta256": C(),
    "cta128": C(bn=128, stages=6),
    "cta128_2stage": C(bn=128, stages=2),
    "pair": C(bm=256, stages=6, cluster_m=2),
    "pair_streamk": C(bm=256, stages=6, cluster_m=2, split_k=0),
    "quad": C(bm=256, stages=6, cluster_m=4),
    "quad_streamk": C(bm=256, stages=6, cluster_m=4, split_k=0),
}


def batched_case(nb, M, N, K, layout, cfg, share_a=False, share_b=False, dist=None, out_dtype=gen.F32, ep=None,
                 exact=False):
    dist = dist or gen.normal(0, 1)
    lda = round_up(K, 8)
    b_rows, b_cols = (K, N) if layout == gen.B_KN else (N, K)
    ldb = round_up(b_cols, 8)
    ldc = round_up(N, 16 // gen.DTYPE_SIZE[out_dtype])
    As, Bs = [], []
    for b in range(nb):
        a, bb = gen.make_operands(M, N, K, gen.BF16, layout, dist, None, seed=100 + b, lda=lda, ldb=ldb)
        As.append(a)
        Bs.append(bb)
    if share_a:
        As = [As[0]] * nb
    if share_b:
        Bs = [Bs[0]] * nb
    A = torch.stack(As[:1] if share_a else As).to(DEV)
    B = torch.stack(Bs[:1] if share_b else Bs).to(DEV)
    Cd = torch.full((nb, M, ldc), float("nan"), dtype=gen.TORCH_DTYPE[out_dtype], device=DEV)
    rc = tgemm.tgemm_run_strided_batched(nb, M, N, K, A.data_ptr(), lda, 0 if share_a else M * lda, B.data_ptr(), ldb,
                                         0 if share_b else b_rows * ldb, layout, Cd.data_ptr(), ldc, M * ldc,
                                         gen.BF16, out_dtype, None, ep, cfg)
    assert rc == 0, tgemm.status_string(rc)
    assert tgemm.tgemm_check() == 0
    out = Cd.cpu()
    for b in range(nb):
        ref, bound = oracle.gemm(As[b], Bs[b], M, N, K, lda, ldb, layout, gen.BF16)
        if exact:
            assert np.array_equal(bits(out[b, :, :N], out_dtype), oracle.round_bits(ref, out_dtype)), "batch %d" % b
        else:
            assert_close(out[b, :, :N].double().numpy(), ref, bound, out_dtype, "batch %d" % b)
    return out, As, Bs


@pytest.mark.parametrize("name", sorted(CONFIGS))
@pytest.mark.parametrize("layout", [gen.B_NK, gen.B_KN], ids=["nk", "kn"])
def test_batched_integers_exact(name, layout):
    batched_case(3, 300, 520, 200, layout, CONFIGS[name], dist=gen.ints(-2, 2), exact=True)


@pytest.mark.parametrize("share", ["a", "b"])
def test_batched_shared_operand(share):
    """A zero stride shares one operand across all batches."""
    batched_case(4, 256, 384, 320, gen.B_NK, None, share_a=share == "a", share_b=share == "b")


def test_batched_many_small_problems_one_launch():
    batched_case(17, 64, 96, 80, gen.B_NK, None, out_dtype=gen.BF16)


def test_batched_skinny_rows_use_the_tile_kernels():
    batched_case(5, 16, 700, 512, gen.B_NK, None)


def test_batch_of_one_equals_tgemm_run():
    M, N, K = 300, 520, 200
    a, b = gen.make_operands(M, N, K, gen.BF16, gen.B_NK, gen.normal(0, 1), None, seed=9, lda=200, ldb=200)
    A, B = a.to(DEV), b.to(DEV)
    C1 = torch.empty(M, N, device=DEV)
    C2 = torch.empty(M, N, device=DEV)
    assert tgemm.tgemm_run(M, N, K, A.data_ptr(), 200, B.data_ptr(), 200, gen.B_NK, C1.data_ptr(), N, gen.BF16,
                           gen.F32, None) == 0
    assert tgemm.tgemm_run_strided_batched(1, M, N, K, A.data_ptr(), 200, 0, B.data_ptr(), 200, 0, gen.B_NK,
                                           C2.data_ptr(), N, 0, gen.BF16, gen.F32, None, None, None) == 0
    assert tgemm.tgemm_check() == 0
    assert torch.equal(C1, C2)


def test_batched_with_epilogue_steps_c_in_like_c():
    nb, M, N, K = 3, 200, 264, 128
    ldc = 264
    cin = torch.randn(nb, M, ldc).to(DEV)
    bias = torch.randn(N).to(DEV)
    ep = tgemm.Epilogue(alpha=0.5, beta=2.0, c_in=cin.data_ptr(), ldc_in=ldc, bias=bias.data_ptr(),
                        bias_dtype=gen.F32, act=tgemm.ACT_RELU)
    out, As, Bs = None, [], []
    lda, ldb = 128, 128
    for b in range(nb):
        a, bb = gen.make_operands(M, N, K, gen.BF16, gen.B_NK, gen.normal(0, 1), None, seed=200 + b)
        As.append(a)
        Bs.append(bb)
    A, B = torch.stack(As).to(DEV), torch.stack(Bs).to(DEV)
    Cd = torch.empty(nb, M, ldc, device=DEV)
    rc = tgemm.tgemm_run_strided_batched(nb, M, N, K, A.data_ptr(), lda, M * lda, B.data_ptr(), ldb, N * ldb, gen.B_NK,
                                         Cd.data_ptr(), ldc, M * ldc, gen.BF16, gen.F32, None, ep, None)
    assert rc == 0 and tgemm.tgemm_check() == 0
    for b in range(nb):
        acc, bound = oracle.gemm(As[b], Bs[b], M, N, K, lda, ldb, gen.B_NK, gen.BF16)
        ref = oracle.epilogue(acc, 0.5, 2.0, cin[b, :, :N].double().cpu().numpy(), bias.double().cpu().numpy(),
                              oracle.ACT_RELU)
        got = Cd[b, :, :N].double().cpu().numpy()
        tol = 0.5e-3 * bound + 2.0 ** -20 * (np.abs(0.5 * acc) + np.abs(2 * cin[b, :, :N].double().cpu().numpy())
                                              + np.abs(bias.double().cpu().numpy())) + oracle.ulp(ref, gen.F32)
        assert np.all(np.abs(got - ref) <= tol), "batch %d" % b


def test_batched_empty_k_and_zero_batches():
    nb, M, N = 3, 40, 64
    Cd = torch.full((nb, M, N), 5.0, device=DEV)
    x = torch.empty(64, dtype=torch.bfloat16, device=DEV)
    assert tgemm.tgemm_run_strided_batched(nb, M, N, 0, x.data_ptr(), 8, 0, x.data_ptr(), 8, 0, gen.B_NK,
                                           Cd.data_ptr(), N, M * N, gen.BF16, gen.F32, None, None, None) == 0
    assert tgemm.tgemm_check() == 0 and torch.count_nonzero(Cd).item() == 0
    Cd.fill_(5.0)
    assert tgemm.tgemm_run_strided_batched(0, M, N, 16, x.data_ptr(), 16, 0, x.data_ptr(), 16, 0, gen.B_NK,
                                           Cd.data_ptr(), N, M * N, gen.BF16, gen.F32, None, None, None) == 0
    assert tgemm.tgemm_check() == 0 and torch.all(Cd == 5.0)


def test_batched_rejects_overlapping_strides():
    x = torch.empty(1 << 16, dtype=torch.bfloat16, device=DEV)
    p = x.data_ptr()
    args = lambda sa, sb, sc: (3, 64, 64, 64, p, 64, sa, p, 64, sb, gen.B_NK, p, 64, sc, gen.BF16, gen.BF16, None,
                               None, None)
    assert tgemm.tgemm_run_strided_batched(*args(100, 0, 4096)) == tgemm.ERR_INVALID_ARG   # A batches overlap
    assert tgemm.tgemm_run_strided_batched(*args(4096, 4096, 64)) == tgemm.ERR_INVALID_ARG  # C batches overlap
    assert tgemm.tgemm_run_strided_batched(*args(4100, 0, 4096)) == tgemm.ERR_MISALIGNED
