"""Planted mistakes in the oracle must be caught by its pins.

Each case compiles a copy of the oracle source with one plausible slip (a
dropped term, a wrong sign, a transposed or mis-strided operand, an exponent
bias off by one, ties rounded away from zero, a spacing off by a factor of
two) and runs the pin suite against it in a child process.  The suite has to
fail for every mutant.  Everything runs on the CPU.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "tgemm_oracle.c")

MUTANTS = {
    "dropped_last_term_nk": ("for (int64_t k = 0; k < p->K; ++k) {\n            double a = elem(p, p->A, arow + k), b = elem(p, p->B, bcol + k);",
                             "for (int64_t k = 0; k < p->K - 1; ++k) {\n            double a = elem(p, p->A, arow + k), b = elem(p, p->B, bcol + k);"),
    "dropped_last_term_kn": ("for (int64_t k = 0; k < p->K; ++k) {\n            double a = elem(p, p->A, arow + k), b = elem(p, p->B, k * p->ldb + j);",
                             "for (int64_t k = 0; k < p->K - 1; ++k) {\n            double a = elem(p, p->A, arow + k), b = elem(p, p->B, k * p->ldb + j);"),
    "wrong_sign": ("            s += a * b;\n            r += fabs(a) * fabs(b);\n        }\n    } else {",
                   "            s -= a * b;\n            r += fabs(a) * fabs(b);\n        }\n    } else {"),
    "transposed_b_kn": ("elem(p, p->B, k * p->ldb + j)", "elem(p, p->B, j * p->ldb + k)"),
    "wrong_row_nk": ("const int64_t bcol = j * p->ldb;", "const int64_t bcol = i * p->ldb;"),
    "ignores_lda": ("const int64_t arow = i * p->lda;", "const int64_t arow = i * p->K;"),
    "f16_bias_off_by_one": ("expo - 25); /* 1.frac", "expo - 24); /* 1.frac"),
    "bf16_fraction_width": ("(frac | 0x80), expo - 134)", "(frac | 0x80), expo - 133)"),
    "ties_away_from_zero": ("double r = nearbyint(a / q) * q;", "double r = round(a / q) * q;"),
    "ulp_factor_two": ("return ldexp(1.0, e - p + 1);", "return ldexp(1.0, e - p);"),
    "bound_signed": ("r += fabs(a) * fabs(b);\n        }\n    } else {", "r += a * fabs(b);\n        }\n    } else {"),
    "gelu_constant": ("0.044715 * x * x * x", "0.047715 * x * x * x"),
    "bias_row_index": ("x += bias[j];", "x += bias[i % cols];"),
    "beta_dropped": ("if (cin) x += beta * cin[i * ldcin + j];", "if (cin) x += cin[i * ldcin + j];"),
    "e4m3_bias": ("(double)(frac | 8), expo - 10)", "(double)(frac | 8), expo - 9)"),
    "e5m2_subnormal": ("ldexp((double)frac, -16);", "ldexp((double)frac, -15);"),
    "fp8_read_as_16bit": ("p->tab[p->esz == 1 ?", "p->tab[p->esz == 3 ?"),
    "tf32_keeps_low_bits": ("uint32_t t = u & 0xffffe000u;", "uint32_t t = u;"),
    "tf32_nine_fraction_bits": ("uint32_t t = u & 0xffffe000u;", "uint32_t t = u & 0xffffc000u;"),
    "tf32_read_as_16bit": ("if (p->esz == 4) return", "if (p->esz == 5) return"),
    "alpha_dropped": ("double x = alpha * D[i * ldd + j];", "double x = D[i * ldd + j];"),
    "relu_passes_magnitude": ("if (act == 1) return x > 0.0 ? x : 0.0;", "if (act == 1) return fabs(x);"),
    "gelu_sqrt_pi_over_2": ("const double c = 0.7978845608028654;", "const double c = 1.2533141373155003;"),
    "overflow_saturates": ("    if (r >= limit)\n        return sign_bit | (exp_all_ones << fbits);",
                           "    if (r >= limit)\n        return sign_bit | (((exp_all_ones - 1u) << fbits) | ((1u << fbits) - 1u));"),
    "fp32_accumulator": ("double s = 0.0, r = 0.0;", "float s = 0.0f; double r = 0.0;"),
    "thread_shares_drop_a_row": ("w[t].last = first + total * (t + 1) / nt;",
                                 "w[t].last = first + total * (t + 1) / nt - (t + 1 < nt);"),
    "element_indices_swapped": ("dot(w->p, w->ii[t], w->jj[t], &w->out[t], &w->out_bound[t]);",
                                "dot(w->p, w->jj[t], w->ii[t], &w->out[t], &w->out_bound[t]);"),
    "row_range_offset_ignored": ("w->C[(i - w->row0) * w->ldc + j] = c;", "w->C[i * w->ldc + j] = c;"),
    "subnormals_flushed": ("        uint32_t frac = (uint32_t)(r / ldexp(1.0, emin - fbits));\n        return sign_bit | frac;",
                           "        uint32_t frac = 0u * (uint32_t)(r / ldexp(1.0, emin - fbits));\n        return sign_bit | frac;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation anchor missing: %s" % name
    mutated = src.replace(old, new, 1)
    c_path = tmp_path / "mutant.c"
    so_path = tmp_path / "libmutant.so"
    c_path.write_text(mutated)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(so_path), str(c_path),
                    "-lpthread", "-lm"], check=True)
    env = dict(os.environ, TGEMM_ORACLE_LIB=str(so_path))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "pins did not catch mutant %s:\n%s" % (name, r.stdout[-2000:])
