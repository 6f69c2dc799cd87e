"""Pins of the CPU oracle against things other than itself.

Each test ties one oracle routine to what the pages or the mathematics fix:
exact rational brute force (the defining sum of "Writing high-performance
matrix multiplication with NVIDIA CUDA Tile", "What is matrix
multiplication?"), identity and permutation matrices, integer inputs whose
result is exact, linearity in B, numpy's float64 matmul, and numpy/torch
conversions for the decoding, rounding and spacing routines.
"""
import math
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

from dense_tiled_gemm_persistent_gb300 import inputs as gen

F16, BF16, F32 = 0, 1, 2
KN, NK = 0, 1


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def exact_value(bits: int, dtype: int) -> Fraction:
    """Exact value of a 16-bit pattern via the standard library / torch."""
    if dtype == F16:
        return Fraction(struct.unpack("<e", struct.pack("<H", bits))[0])
    f = struct.unpack("<f", struct.pack("<I", bits << 16))[0]   # bf16 = top half of an f32
    return Fraction(f)


def fraction_gemm(A, B, M, N, K, lda, ldb, layout, dtype):
    """C and the bound as exact rationals, straight from the definition."""
    a = A.reshape(-1)
    b = B.reshape(-1)
    C = [[Fraction(0)] * N for _ in range(M)]
    R = [[Fraction(0)] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            s, r = Fraction(0), Fraction(0)
            for k in range(K):
                x = exact_value(int(a[i * lda + k]), dtype)
                y = exact_value(int(b[k * ldb + j] if layout == KN else b[j * ldb + k]), dtype)
                s += x * y
                r += abs(x) * abs(y)
            C[i][j], R[i][j] = s, r
    return C, R


# --- decoding ------------------------------------------------------------

def test_decode_f16_all_patterns_match_numpy(orc):
    bits = np.arange(65536, dtype=np.uint32)
    got = orc.decode(bits, F16)
    ref = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_decode_bf16_all_patterns_match_torch(orc):
    bits = np.arange(65536, dtype=np.uint32)
    got = orc.decode(bits, BF16)
    ref = torch.from_numpy(bits.astype(np.uint16).view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


# --- rounding to the output format (round-to-nearest-even) ----------------

def _probe_values(rng, lo_exp, hi_exp, n=20000):
    mant = rng.random(n) + 1.0
    expo = rng.integers(lo_exp, hi_exp, n)
    sign = rng.choice([-1.0, 1.0], n)
    return sign * np.ldexp(mant, expo)


def test_round_f16_matches_numpy(orc):
    rng = np.random.default_rng(11)
    x = np.concatenate([
        _probe_values(rng, -30, 18),
        # exact ties between neighbouring binary16 values, incl. subnormals and overflow edge
        (np.arange(-2048, 2048) + 0.5) * 2.0 ** -24,
        (np.arange(1024, 2048) + 0.5) * 2.0 ** 5,
        [0.0, -0.0, 65504.0, 65519.99, 65520.0, -65520.0, 1e6, np.inf, -np.inf, 2.0 ** -25, 2.0 ** -26],
    ])
    got = orc.round_bits(x, F16).astype(np.uint16)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def test_round_f32_matches_numpy(orc):
    rng = np.random.default_rng(12)
    x = np.concatenate([_probe_values(rng, -160, 130),
                        [0.0, -0.0, 3.4028235677973366e38, 3.5e38, 1e-46, 2.0 ** -150]])
    got = orc.round_bits(x, F32)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float32).view(np.uint32)
    assert np.array_equal(got, ref)


def test_round_bf16_matches_torch(orc):
    # float32-representable inputs, so torch's float32 -> bfloat16 rounding is a
    # single correct rounding of the same value
    rng = np.random.default_rng(13)
    x = _probe_values(rng, -140, 127).astype(np.float32)
    ties = ((np.arange(-256, 256, dtype=np.float64) + 0.5) * 2.0 ** -7).astype(np.float32)
    x = np.concatenate([x, ties, np.float32([0.0, 3.3895314e38, 3.39e38, 1e-40])])
    got = orc.round_bits(x.astype(np.float64), BF16).astype(np.uint16)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


# --- unit in the last place ------------------------------------------------

def test_ulp_f16_f32_match_numpy_spacing(orc):
    rng = np.random.default_rng(14)
    h = rng.integers(1, 0x7BFF, 5000).astype(np.uint16).view(np.float16)   # positive finite
    assert np.array_equal(orc.ulp(h.astype(np.float64), F16), np.spacing(h).astype(np.float64))
    f = np.abs(rng.standard_normal(5000).astype(np.float32)) * np.float32(2.0 ** 20)
    assert np.array_equal(orc.ulp(f.astype(np.float64), F32), np.spacing(f).astype(np.float64))
    assert orc.ulp(np.array([0.0]), F16)[0] == 2.0 ** -24
    assert orc.ulp(np.array([0.0]), F32)[0] == 2.0 ** -149


def test_ulp_bf16_is_the_gap_to_the_next_pattern(orc):
    bits = np.arange(1, 0x7F7F, 37, dtype=np.uint32)          # positive finite bf16 patterns
    v = orc.decode(bits, BF16)
    gap = orc.decode(bits + 1, BF16) - v
    assert np.array_equal(orc.ulp(v, BF16), gap)


# --- the defining sum, exactly ----------------------------------------------

@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("layout", [KN, NK])
def test_brute_force_rational_exact_inputs(orc, dtype, layout):
    """Inputs on a 2^-10 grid in [-1, 1): every double sum is exact, so the
    oracle must equal the rational result bit for bit."""
    rng = np.random.default_rng(100 + 2 * dtype + layout)
    for trial in range(6):
        M, N, K = (int(v) for v in rng.integers(1, 7, 3))
        lda, ldb = K + int(rng.integers(0, 3)), (N if layout == KN else K) + int(rng.integers(0, 3))
        t = gen.TORCH_DTYPE[dtype]
        a = torch.from_numpy(rng.integers(-1024, 1024, (M, lda)) / 1024.0).to(t)
        b = torch.from_numpy(rng.integers(-1024, 1024, ((K if layout == KN else N), ldb)) / 1024.0).to(t)
        A, B = bits16(a), bits16(b)
        C, R = orc.gemm(A, B, M, N, K, lda, ldb, layout, dtype)
        Cf, Rf = fraction_gemm(A, B, M, N, K, lda, ldb, layout, dtype)
        for i in range(M):
            for j in range(N):
                assert C[i, j] == float(Cf[i][j]) and Fraction(C[i, j]) == Cf[i][j]
                assert R[i, j] == float(Rf[i][j])


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("layout", [KN, NK])
def test_brute_force_rational_random_bits(orc, dtype, layout):
    """Arbitrary finite patterns (wide exponent range): the oracle is within
    its double-precision error bound K * 2^-53 * sum|a||b| of the exact sum."""
    rng = np.random.default_rng(200 + 2 * dtype + layout)
    for trial in range(6):
        M, N, K = (int(v) for v in rng.integers(1, 9, 3))
        def finite_bits(shape):
            v = rng.integers(0, 65536, shape).astype(np.uint16)
            expo_mask = 0x7C00 if dtype == F16 else 0x7F80
            v[(v & expo_mask) == expo_mask] &= np.uint16(0x83FF if dtype == F16 else 0x807F)
            return v
        A = finite_bits((M, K))
        B = finite_bits((K, N) if layout == KN else (N, K))
        ldb = N if layout == KN else K
        C, R = orc.gemm(A, B, M, N, K, K, ldb, layout, dtype)
        Cf, Rf = fraction_gemm(A, B, M, N, K, K, ldb, layout, dtype)
        for i in range(M):
            for j in range(N):
                err = abs(Fraction(C[i, j]) - Cf[i][j])
                assert err <= Fraction(K) * Fraction(2) ** -53 * Rf[i][j]


# --- special cases ----------------------------------------------------------

@pytest.mark.parametrize("layout", [KN, NK])
def test_identity_right_and_left(orc, layout):
    M, K = 37, 29
    a, _ = gen.make_operands(M, K, K, F16, layout, gen.uniform(-4, 4), None, seed=5)
    I = torch.eye(K, dtype=torch.float16)   # symmetric: same store in KN and NK
    C, _ = orc.gemm(bits16(a), bits16(I), M, K, K, K, K, layout, F16)
    assert np.array_equal(C, a.double().numpy())
    # I * B = B for a K x N right operand
    N = 23
    _, b = gen.make_operands(K, N, K, BF16, layout, gen.uniform(-4, 4), None, seed=6)
    Ik = torch.eye(K, dtype=torch.bfloat16)
    C2, _ = orc.gemm(bits16(Ik), bits16(b), K, N, K, K, b.shape[1], layout, BF16)
    assert np.array_equal(C2, gen.b_logical(b, N, K, layout).double().numpy())


@pytest.mark.parametrize("layout", [KN, NK])
def test_permutation_matrices_permute_exactly(orc, layout):
    rng = np.random.default_rng(7)
    M, N, K = 19, 31, 31
    a, _ = gen.make_operands(M, N, K, F16, layout, gen.normal(0, 3), None, seed=8)
    perm = rng.permutation(K)
    P = torch.zeros(K, K, dtype=torch.float16)
    P[np.arange(K), perm] = 1.0                # (A P)[:, perm[k]] = A[:, k]
    store = P if layout == KN else P.t().contiguous()
    C, _ = orc.gemm(bits16(a), bits16(store), M, K, K, K, K, layout, F16)
    ref = np.empty((M, K))
    ref[:, perm] = a.double().numpy()
    assert np.array_equal(C, ref)
    # P^T B permutes the rows of B: (P^T B)[perm[k], :] = B[k, :]
    _, b = gen.make_operands(K, N, K, F16, layout, gen.normal(0, 3), None, seed=9)
    Pt = P.t().contiguous()
    C2, _ = orc.gemm(bits16(Pt), bits16(b), K, N, K, K, b.shape[1], layout, F16)
    bl = gen.b_logical(b, N, K, layout).double().numpy()
    ref2 = np.empty((K, N))
    ref2[perm, :] = bl
    assert np.array_equal(C2, ref2)


@pytest.mark.parametrize("layout", [KN, NK])
def test_integer_inputs_exact_against_integer_arithmetic(orc, layout):
    M, N, K = 24, 20, 33
    a, b = gen.make_operands(M, N, K, BF16, layout, gen.ints(-2, 2), None, seed=0)
    C, R = orc.gemm(bits16(a), bits16(b), M, N, K, K, b.shape[1], layout, BF16)
    ai = a.to(torch.int64).tolist()
    bi = gen.b_logical(b, N, K, layout).to(torch.int64).tolist()
    for i in range(M):
        for j in range(N):
            assert C[i, j] == sum(ai[i][k] * bi[k][j] for k in range(K))
            assert R[i, j] == sum(abs(ai[i][k] * bi[k][j]) for k in range(K))


def test_linearity_in_b(orc):
    M, N, K = 40, 36, 50
    a, b1 = gen.make_operands(M, N, K, F16, NK, gen.ints(-2, 2), None, seed=21)
    _, b2 = gen.make_operands(M, N, K, F16, NK, gen.ints(-2, 2), None, seed=22)
    s = (b1.float() + b2.float()).to(torch.float16)          # exact: small integers
    C1, _ = orc.gemm(bits16(a), bits16(b1), M, N, K, K, K, NK, F16)
    C2, _ = orc.gemm(bits16(a), bits16(b2), M, N, K, K, K, NK, F16)
    C3, _ = orc.gemm(bits16(a), bits16(s), M, N, K, K, K, NK, F16)
    assert np.array_equal(C3, C1 + C2)


@pytest.mark.parametrize("layout", [KN, NK])
@pytest.mark.parametrize("dtype", [F16, BF16])
def test_numpy_float64_matmul_crosscheck(orc, layout, dtype):
    M, N, K = 128, 96, 256
    a, b = gen.make_operands(M, N, K, dtype, layout, gen.normal(0, 1), None, seed=31)
    C, R = orc.gemm(bits16(a), bits16(b), M, N, K, K, b.shape[1], layout, dtype)
    ref = a.double().numpy() @ gen.b_logical(b, N, K, layout).double().numpy()
    assert np.all(np.abs(C - ref) <= 1e-12 * R)
    assert np.all(R >= np.abs(C))


def test_transposed_operand_is_detected(orc):
    """Reading B with the wrong layout changes the result on a non-square case."""
    M, N, K = 8, 12, 12
    a, b = gen.make_operands(M, N, K, F16, NK, gen.ints(-2, 2), None, seed=41)
    C_nk, _ = orc.gemm(bits16(a), bits16(b), M, N, K, K, K, NK, F16)
    C_kn, _ = orc.gemm(bits16(a), bits16(b), M, N, K, K, K, KN, F16)
    assert not np.array_equal(C_nk, C_kn)
    ref = a.double().numpy() @ b.double().numpy().T
    assert np.array_equal(C_nk, ref)


def test_padding_is_never_read(orc):
    M, N, K = 17, 9, 21
    a, b = gen.make_operands(M, N, K, F16, KN, gen.uniform(-1, 1), None, seed=51,
                             lda=K + 11, ldb=N + 7, pad_value=float("nan"))
    C, R = orc.gemm(bits16(a), bits16(b), M, N, K, K + 11, N + 7, KN, F16)
    assert np.all(np.isfinite(C)) and np.all(np.isfinite(R))


def test_elements_and_row_ranges_agree_with_full(orc):
    M, N, K = 33, 45, 70
    a, b = gen.make_operands(M, N, K, BF16, NK, gen.normal(0, 1), None, seed=61)
    C, R = orc.gemm(bits16(a), bits16(b), M, N, K, K, K, NK, BF16, threads=3)
    rng = np.random.default_rng(0)
    ii, jj = rng.integers(0, M, 200), rng.integers(0, N, 200)
    e, eb = orc.gemm_elements(bits16(a), bits16(b), M, N, K, K, K, NK, BF16, ii, jj)
    assert np.array_equal(e, C[ii, jj]) and np.array_equal(eb, R[ii, jj])
    Cr, Rr = orc.gemm_rows(bits16(a), bits16(b), M, N, K, K, K, NK, BF16, 5, 19, threads=4)
    assert np.array_equal(Cr, C[5:19]) and np.array_equal(Rr, R[5:19])
    # thread count never changes a result
    C1, _ = orc.gemm(bits16(a), bits16(b), M, N, K, K, K, NK, BF16, threads=1)
    assert np.array_equal(C1, C)


def test_empty_sum_and_empty_shapes(orc):
    """K = 0 is the empty sum: C = 0.  M = 0 or N = 0 give empty results."""
    a = np.zeros((4, 1), np.uint16)
    b = np.zeros((1, 5), np.uint16)
    C, R = orc.gemm(a, b, 4, 5, 0, 1, 5, KN, F16)
    assert C.shape == (4, 5) and not C.any() and not R.any()
    C0, _ = orc.gemm(a, b, 0, 5, 1, 1, 5, KN, F16)
    assert C0.shape == (0, 5)


def test_bad_arguments_rejected(orc):
    a = np.zeros((4, 4), np.uint16)
    with pytest.raises(ValueError):
        orc.gemm(a, a, 4, 4, 4, 3, 4, KN, F16)      # lda < K
    with pytest.raises(ValueError):
        orc.gemm(a, a, 4, 4, 4, 4, 4, KN, F32)      # FP32 is not an input format


# --- fused epilogue ---------------------------------------------------------

def test_epilogue_identity_scaling_and_bias(orc):
    rng = np.random.default_rng(71)
    C = rng.standard_normal((9, 13))
    assert np.array_equal(orc.epilogue(C), C)                       # alpha 1, nothing else
    assert np.array_equal(orc.epilogue(C, alpha=2.0), 2.0 * C)      # exact doubling
    bias = rng.standard_normal(13)
    assert np.array_equal(orc.epilogue(C, bias=bias), C + bias[None, :])
    cin = rng.standard_normal((9, 13))
    assert np.array_equal(orc.epilogue(C, alpha=0.0, beta=1.0, cin=cin), cin)
    # beta * C_in with C_in = C gives (alpha + beta) C for exact small values
    Ci = rng.integers(-50, 50, (9, 13)).astype(np.float64)
    assert np.array_equal(orc.epilogue(Ci, alpha=3.0, beta=-2.0, cin=Ci), Ci)


def test_epilogue_relu_is_max_with_zero(orc):
    C = np.array([[-2.0, -0.0, 0.0, 1.5, -1e-300, 7.0]])
    assert np.array_equal(orc.epilogue(C, act=orc.ACT_RELU), np.maximum(C, 0.0))


def test_epilogue_gelu_tanh_odd_part_and_torch(orc):
    x = np.linspace(-8, 8, 4001)
    g = orc.epilogue(x[None, :], act=orc.ACT_GELU_TANH)[0]
    gm = orc.epilogue(-x[None, :], act=orc.ACT_GELU_TANH)[0]
    # tanh is odd, so gelu(x) - gelu(-x) = x exactly in the tanh form
    assert np.allclose(g - gm, x, rtol=0, atol=1e-15)
    assert g[2000] == 0.0                                           # gelu(0) = 0
    # the library's tanh-approximated GELU (float64) agrees
    ref = torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    assert np.allclose(g, ref, rtol=1e-14, atol=1e-14)
    # far from zero it is the identity or zero
    assert abs(g[-1] - 8.0) < 1e-12 and abs(g[0]) < 1e-12


# --- FP8 inputs ----------------------------------------------------------------

E4M3, E5M2 = 3, 4


@pytest.mark.parametrize("dtype,tdt", [(E4M3, torch.float8_e4m3fn), (E5M2, torch.float8_e5m2)])
def test_decode_fp8_all_patterns_match_torch(orc, dtype, tdt):
    bits = np.arange(256, dtype=np.uint32)
    got = orc.decode(bits, dtype)
    ref = torch.from_numpy(bits.astype(np.uint8)).view(tdt).double().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


@pytest.mark.parametrize("dtype,tdt", [(E4M3, torch.float8_e4m3fn), (E5M2, torch.float8_e5m2)])
@pytest.mark.parametrize("layout", [KN, NK])
def test_fp8_brute_force_rational(orc, dtype, tdt, layout):
    """FP8 products have at most 8 significant bits and a bounded exponent
    range, so small double sums are exact: equal to the rational result."""
    rng = np.random.default_rng(300 + dtype + layout)
    for _ in range(5):
        M, N, K = (int(v) for v in rng.integers(1, 7, 3))
        a = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(tdt)
        b = torch.from_numpy(rng.standard_normal((K, N) if layout == KN else (N, K)).astype(np.float32)).to(tdt)
        C, R = orc.gemm(a, b, M, N, K, K, b.shape[1], layout, dtype)
        av, bv = a.double().numpy(), b.double().numpy()
        for i in range(M):
            for j in range(N):
                s = sum(Fraction(float(av[i, k])) * Fraction(float(bv[k, j] if layout == KN else bv[j, k]))
                        for k in range(K))
                assert Fraction(C[i, j]) == s


def test_fp8_integers_exact(orc):
    M, N, K = 20, 24, 40
    g = torch.Generator().manual_seed(5)
    a = torch.randint(-2, 3, (M, K), generator=g).float().to(torch.float8_e4m3fn)
    b = torch.randint(-2, 3, (N, K), generator=g).float().to(torch.float8_e5m2)
    # same-type operands only on the GPU; the oracle itself decodes either
    C, _ = orc.gemm(a, b.float().to(torch.float8_e4m3fn), M, N, K, K, K, NK, E4M3)
    assert np.array_equal(C, a.double().numpy() @ b.double().numpy().T)


# --- FP32 operands read as TF32 --------------------------------------------------
#
# TF32 keeps the FP32 sign, the 8-bit exponent and the top 10 of the 23
# fraction bits.  The pins below restate that format with Python's struct
# module (an FP32 pattern with its low 13 bits cleared) and with closed-form
# values, never through the oracle's own decoder.

TF32 = 5


def tf32_exact(bits: int) -> Fraction:
    return Fraction(struct.unpack("<f", struct.pack("<I", bits & 0xFFFFE000))[0])


def f32_bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


def test_tf32_decode_closed_forms(orc):
    cases = {
        f32_bits(1.0 + 3 * 2.0 ** -12): 1.0,                    # 0.75 of a TF32 step: dropped, not rounded up
        f32_bits(-(1.0 + 3 * 2.0 ** -12)): -1.0,                # toward zero for negatives too
        f32_bits(1.0 + 2.0 ** -10): 1.0 + 2.0 ** -10,           # one TF32 step is kept
        f32_bits(1.0 + 2.0 ** -10 + 2.0 ** -11): 1.0 + 2.0 ** -10,
        f32_bits(3.0): 3.0,
        0x7F7FFFFF: (2.0 - 2.0 ** -10) * 2.0 ** 127,            # largest FP32 -> largest TF32
        0x00000001: 0.0,                                         # smallest subnormal drops out
        0x00002000: 2.0 ** -136,                                 # lowest kept subnormal bit
        0x80000000: -0.0,
        0x7F800000: math.inf,
    }
    bits = np.array(list(cases), dtype=np.uint32)
    got = orc.decode(bits, TF32)
    for b, g in zip(bits.tolist(), got.tolist()):
        assert g == cases[b] and math.copysign(1, g) == math.copysign(1, cases[b]), hex(b)


def test_tf32_decode_matches_struct_on_random_patterns(orc):
    rng = np.random.default_rng(17)
    bits = rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32)
    bits = bits[(bits & 0x7F800000) != 0x7F800000]            # finite patterns
    got = orc.decode(bits, TF32)
    ref = np.array([float(tf32_exact(int(b))) for b in bits.tolist()])
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("layout", [KN, NK])
def test_tf32_brute_force_rational(orc, layout):
    """Random FP32 patterns in a bounded exponent range: every product of
    two TF32 values has at most 22 significant bits, so the oracle is within
    K * 2^-53 * bound of the exact rational sum of truncated values."""
    rng = np.random.default_rng(400 + layout)
    for _ in range(6):
        M, N, K = (int(v) for v in rng.integers(1, 8, 3))
        def pats(shape):
            x = rng.standard_normal(shape).astype(np.float32) * np.float32(3.0)
            return x.view(np.uint32)
        A = pats((M, K))
        B = pats((K, N) if layout == KN else (N, K))
        ldb = N if layout == KN else K
        C, R = orc.gemm(A, B, M, N, K, K, ldb, layout, TF32)
        for i in range(M):
            for j in range(N):
                s, r = Fraction(0), Fraction(0)
                for k in range(K):
                    x = tf32_exact(int(A[i, k]))
                    y = tf32_exact(int(B[k, j] if layout == KN else B[j, k]))
                    s += x * y
                    r += abs(x) * abs(y)
                assert abs(Fraction(C[i, j]) - s) <= Fraction(K) * Fraction(2) ** -53 * r
                assert R[i, j] == float(r)


def test_tf32_equals_f16_on_values_both_hold_exactly(orc):
    """FP16 values have 10 fraction bits, so in FP32 storage they are TF32
    values already: the TF32 product equals the FP16 one exactly."""
    M, N, K = 33, 21, 70
    g = torch.Generator().manual_seed(8)
    a16 = (torch.rand(M, K, generator=g) * 4 - 2).half()
    b16 = (torch.rand(N, K, generator=g) * 4 - 2).half()
    C16, R16 = orc.gemm(a16, b16, M, N, K, K, K, NK, F16)
    C32, R32 = orc.gemm(a16.float(), b16.float(), M, N, K, K, K, NK, TF32)
    assert np.array_equal(C16, C32) and np.array_equal(R16, R32)


def test_tf32_integers_exact_and_low_bits_ignored(orc):
    M, N, K = 16, 12, 50
    g = torch.Generator().manual_seed(9)
    a = torch.randint(-3, 4, (M, K), generator=g).float()
    b = torch.randint(-3, 4, (K, N), generator=g).float()
    want = a.double().numpy() @ b.double().numpy()
    C, _ = orc.gemm(a, b, M, N, K, K, N, KN, TF32)
    assert np.array_equal(C, want)
    # setting any of the 13 dropped bits of every element leaves C unchanged
    noise = torch.randint(0, 1 << 13, (M, K), generator=g, dtype=torch.int32)
    a_noisy = (a.view(torch.int32) | torch.where(a != 0, noise, torch.zeros_like(noise))).view(torch.float32)
    C2, _ = orc.gemm(a_noisy, b, M, N, K, K, N, KN, TF32)
    assert np.array_equal(C2, want)
