"""GPU parity of the fused epilogue D = act(alpha*(A*B) + beta*C_in + bias)
against the FP64 oracle, on every kernel family.

Tolerance: the GEMM's bound scaled by |alpha|, plus FP32 rounding of the
epilogue's terms (2^-20 of each magnitude), times the activation's Lipschitz
constant (1 for none and ReLU, 1.13 for the tanh-form GELU), plus one unit in
the last place of the output type at the oracle's value.
"""
import numpy as np
import pytest
import torch

import oracle
from dense_tiled_gemm_persistent_gb300 import inputs as gen
from dense_tiled_gemm_persistent_gb300 import tgemm

from gpu_util import ensure_built, operands, round_up

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
    "cta256": C(),
    "cta128": C(bn=128, stages=6),
    "cta128_2stage": C(bn=128, stages=2),
    "pair": C(bm=256, stages=6, cluster_m=2),
    "pair_streamk": C(bm=256, stages=6, cluster_m=2, split_k=0),
    "quad": C(bm=256, stages=6, cluster_m=4),
    "quad_streamk": C(bm=256, stages=6, cluster_m=4, split_k=0),
    "skinny_cluster": C(bn=16, stages=12, cluster_m=3, group_m=1, split_k=3, swap_ab=2),
    "skinny_workspace": C(bn=16, stages=4, group_m=1, split_k=5, swap_ab=1),
}

EPILOGUES = {
    "alpha": dict(alpha=0.5),
    "beta": dict(beta=1.5),
    "bias": dict(bias=True),
    "relu": dict(act=tgemm.ACT_RELU),
    "gelu": dict(act=tgemm.ACT_GELU_TANH),
    "all": dict(alpha=-0.75, beta=0.5, bias=True, act=tgemm.ACT_GELU_TANH),
}


def run_case(cfg_name, epi_name, out_dtype=gen.BF16, bias_dtype=gen.F32, layout=gen.B_NK, inplace=False, K=None):
    skinny = cfg_name.startswith("skinny")
    M, N = (16, 600) if skinny else (300, 520)
    K = 1000 if K is None else K
    a, b = operands(M, N, K, gen.BF16, layout, gen.normal(0, 1), seed=61, dist_b=gen.normal(0, 0.05))
    e = EPILOGUES[epi_name]
    alpha, beta, act = e.get("alpha", 1.0), e.get("beta", 0.0), e.get("act", tgemm.ACT_NONE)
    tdt = gen.TORCH_DTYPE[out_dtype]
    ldc = round_up(N, 16 // gen.DTYPE_SIZE[out_dtype])
    g = torch.Generator().manual_seed(7)
    cin = torch.randn(M, ldc, generator=g).to(tdt)
    bias = torch.randn(N, generator=g).to(gen.TORCH_DTYPE[bias_dtype]) if e.get("bias") else None
    A, B = a.to(DEV), b.to(DEV)
    Cd = cin.to(DEV) if inplace else torch.full((M, ldc), float("nan"), dtype=tdt, device=DEV)
    cin_d = Cd if inplace else cin.to(DEV)
    bias_d = bias.to(DEV) if bias is not None else None
    ep = tgemm.Epilogue(alpha=alpha, beta=beta, c_in=cin_d.data_ptr() if beta else None, ldc_in=ldc,
                        bias=bias_d.data_ptr() if bias_d is not None else None, bias_dtype=bias_dtype, act=act)
    rc = tgemm.tgemm_run_ex(M, N, K, A.data_ptr(), A.shape[1], B.data_ptr(), B.shape[1], layout, Cd.data_ptr(), ldc,
                            gen.BF16, out_dtype, None, ep, CONFIGS[cfg_name])
    assert rc == 0, tgemm.status_string(rc)
    assert tgemm.tgemm_check() == 0
    got = Cd[:, :N].double().cpu().numpy()
    acc, bound = oracle.gemm(a, b, M, N, K, a.shape[1], b.shape[1], layout, gen.BF16)
    cin64 = cin[:, :N].double().numpy() if beta else None
    bias64 = bias.double().numpy() if bias is not None else None
    ref = oracle.epilogue(acc, alpha, beta, cin64, bias64, act)
    lip = 1.13 if act == tgemm.ACT_GELU_TANH else 1.0
    mag = np.abs(alpha * acc) + (np.abs(beta * cin64) if beta else 0) + (np.abs(bias64)[None, :] if bias is not None else 0)
    tol = lip * (abs(alpha) * 1e-3 * bound + 2.0 ** -20 * mag) + oracle.ulp(ref, out_dtype)
    bad = ~(np.abs(got - ref) <= tol)
    assert not bad.any(), "%s/%s: %d bad, first %s got %r want %r" % (
        cfg_name, epi_name, bad.sum(), tuple(np.argwhere(bad)[0]), got[tuple(np.argwhere(bad)[0])],
        ref[tuple(np.argwhere(bad)[0])])


@pytest.mark.parametrize("cfg_name", sorted(CONFIGS))
@pytest.mark.parametrize("epi_name", sorted(EPILOGUES))
def test_epilogue_every_kernel(cfg_name, epi_name):
    run_case(cfg_name, epi_name)


@pytest.mark.parametrize("cfg_name", ["cta256", "pair", "skinny_cluster"])
@pytest.mark.parametrize("out_dtype", [gen.F32, gen.F16], ids=["o32", "o16"])
@pytest.mark.parametrize("bias_dtype", [gen.F16, gen.BF16], ids=["b16", "bbf16"])
def test_epilogue_output_and_bias_types(cfg_name, out_dtype, bias_dtype):
    run_case(cfg_name, "all", out_dtype=out_dtype, bias_dtype=bias_dtype, layout=gen.B_KN)


@pytest.mark.parametrize("cfg_name", ["cta128", "pair_streamk", "quad_streamk", "skinny_workspace"])
def test_epilogue_in_place_accumulate(cfg_name):
    """C_in may be C itself: D = alpha*A*B + beta*C_old."""
    run_case(cfg_name, "beta", inplace=True)


def test_epilogue_with_empty_k():
    M, N = 70, 96
    cin = torch.randn(M, N).to(torch.bfloat16).to(DEV)
    bias = torch.randn(N).to(DEV)
    Cd = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    ep = tgemm.Epilogue(alpha=3.0, beta=2.0, c_in=cin.data_ptr(), ldc_in=N, bias=bias.data_ptr(),
                        bias_dtype=gen.F32, act=tgemm.ACT_RELU)
    x = torch.empty(16, dtype=torch.bfloat16, device=DEV)
    rc = tgemm.tgemm_run_ex(M, N, 0, x.data_ptr(), 8, x.data_ptr(), 8, gen.B_NK, Cd.data_ptr(), N, gen.BF16,
                            gen.BF16, None, ep, None)
    assert rc == 0 and tgemm.tgemm_check() == 0
    ref = oracle.epilogue(np.zeros((M, N)), 3.0, 2.0, cin.double().cpu().numpy(), bias.double().cpu().numpy(),
                          oracle.ACT_RELU)
    got = Cd.double().cpu().numpy()
    assert np.all(np.abs(got - ref) <= 2.0 ** -20 * (np.abs(ref) + 1) + oracle.ulp(ref, gen.BF16))


def test_epilogue_rejects_bad_arguments():
    x = torch.empty(1 << 12, dtype=torch.bfloat16, device=DEV)
    p = x.data_ptr()
    args = (128, 128, 64, p, 64, p, 64, gen.B_NK, p, 128, gen.BF16, gen.BF16, None)
    assert tgemm.tgemm_run_ex(*args, tgemm.Epilogue(alpha=1, act=9), None) == tgemm.ERR_INVALID_ARG
    assert tgemm.tgemm_run_ex(*args, tgemm.Epilogue(alpha=1, beta=1.0, c_in=None, ldc_in=128), None) \
        == tgemm.ERR_INVALID_ARG
    assert tgemm.tgemm_run_ex(*args, tgemm.Epilogue(alpha=1, beta=1.0, c_in=p + 2, ldc_in=128), None) \
        == tgemm.ERR_MISALIGNED
    assert tgemm.tgemm_run_ex(*args, tgemm.Epilogue(alpha=1, bias=p, bias_dtype=7), None) == tgemm.ERR_INVALID_ARG
