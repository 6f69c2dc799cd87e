"""CPU oracle for C = A*B (test infrastructure only).

Only the tests, the package smoke entry and the benchmark's CPU-baseline leg
may import this package.  The product path never does.
"""
from .oracle import (  # noqa: F401
    build,
    gemm,
    gemm_rows,
    gemm_elements,
    round_bits,
    ulp,
    decode,
    epilogue,
    ACT_NONE,
    ACT_RELU,
    ACT_GELU_TANH,
    F16,
    BF16,
    F32,
    E4M3,
    E5M2,
    TF32,
    B_KN,
    B_NK,
)
