"""Seeded synthetic operands for C = A*B.

This module only draws random numbers and lays them out; it holds none of the
product's arithmetic.  The CUDA path (through the C ABI) and the CPU oracle
both consume exactly the tensors made here.

Recipe (the pages give seeds and distributions but no generator):
  * ``g = torch.Generator("cpu").manual_seed(seed)``;
  * A's M x K values are drawn first, then B's values in its storage
    orientation (K x N for layout KN, N x K for layout NK), both in float32;
  * uniform(a, b) is ``a + (b - a) * torch.rand``; normal(mu, sigma) is
    ``mu + sigma * torch.randn``; ints(lo, hi) is ``torch.randint(lo, hi + 1)``;
  * the float32 draws are rounded to FP16/BF16/FP8 with ``Tensor.to`` (RNE;
    FP8 draws are kept inside the FP8 type's finite range by the caller);
  * a leading dimension larger than the row length pads each row; the pad
    holds ``pad_value`` (NaN by default for the poison tests), never data.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Tuple

import torch

F16, BF16, F32, E4M3, E5M2 = 0, 1, 2, 3, 4
B_KN, B_NK = 0, 1

TORCH_DTYPE = {F16: torch.float16, BF16: torch.bfloat16, F32: torch.float32,
               E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}
DTYPE_NAME = {F16: "f16", BF16: "bf16", F32: "f32", E4M3: "e4m3", E5M2: "e5m2"}
DTYPE_SIZE = {F16: 2, BF16: 2, F32: 4, E4M3: 1, E5M2: 1}


@dataclass(frozen=True)
class Dist:
    """A value distribution: kind in {"uniform", "normal", "ints"}."""
    kind: str
    a: float
    b: float

    def describe(self) -> str:
        if self.kind == "uniform":
            return "uniform[%g,%g)" % (self.a, self.b)
        if self.kind == "normal":
            return "normal(%g,%g)" % (self.a, self.b)
        return "ints{%d..%d}" % (int(self.a), int(self.b))

    def draw(self, shape, g: torch.Generator) -> torch.Tensor:
        if self.kind == "uniform":
            return self.a + (self.b - self.a) * torch.rand(shape, generator=g, dtype=torch.float32)
        if self.kind == "normal":
            return self.a + self.b * torch.randn(shape, generator=g, dtype=torch.float32)
        if self.kind == "ints":
            return torch.randint(int(self.a), int(self.b) + 1, shape, generator=g).to(torch.float32)
        raise ValueError("unknown distribution %r" % (self.kind,))


def uniform(a: float, b: float) -> Dist:
    return Dist("uniform", a, b)


def normal(mu: float, sigma: float) -> Dist:
    return Dist("normal", mu, sigma)


def ints(lo: int, hi: int) -> Dist:
    return Dist("ints", lo, hi)


def _pad(values: torch.Tensor, ld: int, pad_value: float) -> torch.Tensor:
    rows, cols = values.shape
    if ld == cols:
        return values.contiguous()
    out = torch.full((rows, ld), pad_value, dtype=values.dtype)
    out[:, :cols] = values
    return out


def make_operands(M: int, N: int, K: int, in_dtype: int, b_layout: int,
                  dist_a: Dist, dist_b: Optional[Dist], seed: int,
                  lda: Optional[int] = None, ldb: Optional[int] = None,
                  pad_value: float = float("nan")) -> Tuple[torch.Tensor, torch.Tensor]:
    """Seeded CPU operands: A stored M x lda, B stored K x ldb (KN) or N x ldb (NK)."""
    dist_b = dist_b or dist_a
    lda = K if lda is None else lda
    b_rows, b_cols = (K, N) if b_layout == B_KN else (N, K)
    ldb = b_cols if ldb is None else ldb
    if lda < K or ldb < b_cols:
        raise ValueError("leading dimension shorter than the row")
    g = torch.Generator("cpu").manual_seed(seed)
    a = dist_a.draw((M, K), g)
    b = dist_b.draw((b_rows, b_cols), g)
    t = TORCH_DTYPE[in_dtype]
    return _pad(a.to(t), lda, pad_value), _pad(b.to(t), ldb, pad_value)


def b_logical(B: torch.Tensor, N: int, K: int, b_layout: int) -> torch.Tensor:
    """The K x N logical view of a stored B (a view, no arithmetic)."""
    return B[:K, :N] if b_layout == B_KN else B[:N, :K].t()


@dataclass(frozen=True)
class Workload:
    """One named synthetic GEMM problem."""
    name: str
    M: int
    N: int
    K: int
    in_dtype: int
    out_dtype: int
    b_layout: int
    dist_a: Dist
    dist_b: Dist
    seed: int

    def operands(self, **kw):
        return make_operands(self.M, self.N, self.K, self.in_dtype, self.b_layout,
                             self.dist_a, self.dist_b, self.seed, **kw)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def algorithmic_bytes(self) -> int:
        """A and B read once, C written once: the method's minimum traffic."""
        e_in, e_out = DTYPE_SIZE[self.in_dtype], DTYPE_SIZE[self.out_dtype]
        return self.M * self.K * e_in + self.K * self.N * e_in + self.M * self.N * e_out


# The five problem families the benchmark configuration lists, by shape, the
# FP8 and FP32 (multiplied as TF32) forms of the square one, and two more
# shapes (below).
WORKLOADS = {
    w.name: w for w in [
        Workload("gemm_256x256x256_f16_kn_f32", 256, 256, 256, F16, F32, B_KN,
                 uniform(-1, 1), uniform(-1, 1), 0),
        Workload("gemm_256x256x256_f16_kn_f32_ints", 256, 256, 256, F16, F32, B_KN,
                 ints(-2, 2), ints(-2, 2), 0),
        Workload("gemm_4000x3000x5000_bf16_nk_bf16", 4000, 3000, 5000, BF16, BF16, B_NK,
                 normal(0, 1), normal(0, 1), 1),
        Workload("gemm_4096x4096x4096_f16_kn_f16", 4096, 4096, 4096, F16, F16, B_KN,
                 uniform(-1, 1), uniform(-1, 1), 2),
        Workload("gemm_8192x8192x8192_f16_nk_f16", 8192, 8192, 8192, F16, F16, B_NK,
                 uniform(-0.5, 0.5), uniform(-0.5, 0.5), 3),
        Workload("proj_16384x14336x4096_bf16_nk_bf16", 16384, 14336, 4096, BF16, BF16, B_NK,
                 normal(0, 1), normal(0, 0.02), 4),
        Workload("proj_16x4096x4096_bf16_nk_bf16", 16, 4096, 4096, BF16, BF16, B_NK,
                 normal(0, 1), normal(0, 0.02), 4),
        Workload("gemm_8192x8192x8192_e4m3_nk_bf16", 8192, 8192, 8192, E4M3, BF16, B_NK,
                 normal(0, 1), normal(0, 1), 5),
        Workload("gemm_8192x8192x8192_tf32_nk_f32", 8192, 8192, 8192, F32, F32, B_NK,
                 uniform(-0.5, 0.5), uniform(-0.5, 0.5), 6),
        # a 128-token projection (the 65-128-row swap-AB kernel), a short-K
        # product (16 k-blocks per tile) and an FP8 projection: shapes outside
        # the benchmark configuration, named so that the benchmark can time and
        # profile them
        Workload("proj_128x4096x4096_bf16_nk_bf16", 128, 4096, 4096, BF16, BF16, B_NK,
                 normal(0, 1), normal(0, 0.02), 7),
        Workload("gemm_8192x4864x1024_f16_nk_f16", 8192, 4864, 1024, F16, F16, B_NK,
                 uniform(-0.5, 0.5), uniform(-0.5, 0.5), 8),
        # an FP8 weight (E4M3) read by 16 tokens: the in-cluster swap-AB
        # kernel on kind::f8f6f4, HBM-bound
        Workload("proj_16x4096x4096_e4m3_nk_bf16", 16, 4096, 4096, E4M3, BF16, B_NK,
                 normal(0, 1), normal(0, 0.5), 9),
    ]
}


# ---- operands on the output cast's edge cases ------------------------------

CAST_EDGE_KINDS = ("f16_overflow", "f16_subnormal", "bf16_overflow")


def cast_edge_operands(kind: str, M: int, N: int, K: int, b_layout: int, seed: int, scale: int = 1,
                       lda: Optional[int] = None, ldb: Optional[int] = None,
                       pad_value: float = float("nan")) -> Tuple[torch.Tensor, torch.Tensor]:
    """Seeded operands (K > 64) whose exact products sit on the edges of the
    FP32 -> FP16/BF16 cast, with every partial sum exact in FP32 whatever the
    summation order (all values are integer multiples of one power of two,
    far below 2^24 units, and the terms of one output never change sign).

    f16_overflow (FP16): A[i, k] = 1 and B[k, j] = +-1023 * scale for k < 64,
        then 20 fixed k positions spread over the rest of K with A in {0, 1}
        and B in {0, +-4 * scale}: scale * C[i, j] = +-(65472 + 4c) * scale,
        c in 0..20 -- around FP16's largest finite value 65504, through the
        tie at 65520 that rounds to infinity, and past it.  The sign
        alternates by column.
    f16_subnormal (FP16): A = 2^-12 * a, B = 2^-13 * b with a, b uniform
        integers in -2..2: C = 2^-25 * n, mostly below FP16's smallest normal
        2^-14, odd n falling half-way between two subnormals.
    bf16_overflow (BF16): A[i, k] = 2^56 and B[k, j] = +-2^55 * 32640 for
        k < 4 (the sum is BF16's largest finite value, 255 * 2^120), then 15
        fixed k positions with A in {0, 2^58} and B in {0, +-2^58}:
        C = +-(130560 + 32c) * 2^111, c in 0..15 -- the tie at
        130816 * 2^111 rounds to infinity, and the largest sum stays below
        FP32's largest finite value.
    """
    if K <= 64:
        raise ValueError("cast-edge operands need K > 64")
    g = torch.Generator("cpu").manual_seed(seed)
    a = torch.zeros((M, K), dtype=torch.float64)
    bl = torch.zeros((K, N), dtype=torch.float64)        # logical K x N
    sign = torch.where(torch.arange(N) % 2 == 0, 1.0, -1.0).to(torch.float64)
    if kind == "f16_overflow":
        dt = torch.float16
        a[:, :64] = 1.0
        bl[:64, :] = 1023.0 * scale * sign
        pos = 64 + (torch.arange(20) * (K - 64)) // 20
        a[:, pos] = (torch.rand((M, 20), generator=g) < 0.75).to(torch.float64)
        bl[pos, :] = (torch.rand((20, N), generator=g) < 0.75).to(torch.float64) * 4.0 * scale * sign
    elif kind == "f16_subnormal":
        dt = torch.float16
        a = torch.randint(-2, 3, (M, K), generator=g).to(torch.float64) * 2.0 ** -12
        bl = torch.randint(-2, 3, (K, N), generator=g).to(torch.float64) * 2.0 ** -13
    elif kind == "bf16_overflow":
        dt = torch.bfloat16
        a[:, :4] = 2.0 ** 56
        bl[:4, :] = 32640.0 * 2.0 ** 55 * sign
        pos = 64 + (torch.arange(15) * (K - 64)) // 15
        a[:, pos] = (torch.rand((M, 15), generator=g) < 0.75).to(torch.float64) * 2.0 ** 58
        bl[pos, :] = (torch.rand((15, N), generator=g) < 0.75).to(torch.float64) * 2.0 ** 58 * sign
    else:
        raise ValueError("unknown cast-edge kind %r" % (kind,))
    b = bl if b_layout == B_KN else bl.t().contiguous()
    lda = K if lda is None else lda
    ldb = b.shape[1] if ldb is None else ldb
    ta, tb = a.to(dt), b.to(dt)
    if not (torch.equal(ta.double(), a) and torch.equal(tb.double(), b)):
        raise AssertionError("cast-edge values are not exact in the input type")
    return _pad(ta, lda, pad_value), _pad(tb, ldb, pad_value)


def cast_edge_in_dtype(kind: str) -> int:
    return BF16 if kind == "bf16_overflow" else F16


def cast_edge_out_dtype(kind: str) -> int:
    return BF16 if kind == "bf16_overflow" else F16
