/*
 * CPU oracle for the tiled dense matrix multiply C = A * B.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this file; only the tests, the package's smoke entry and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or
 * helper with the CUDA library: it decodes its own input formats, rounds with
 * its own routine and never touches a GPU.
 *
 * What it computes (the defining sum, written out):
 *   "Writing high-performance matrix multiplication with NVIDIA CUDA Tile"
 *   (juejin.cn, section "What is matrix multiplication?"):
 *       C[i][j] = sum over k of A[i][k] * B[k][j]
 *   The CUDA Programming Guide 13.4.2, section 2.4.9.1 "Matrix multiplication"
 *   (unofficial Chinese translation) fixes the precision contract used here:
 *   FP16/BF16 operands, a wider accumulator, one cast when the result is
 *   stored.  The oracle accumulates in IEEE double.  FP16 and BF16 values are
 *   exact in double and so is every product of two of them (at most 22
 *   significant bits), so the only rounding is in the additions: at most
 *   K * 2^-53 * sum_k |A_ik||B_kj|, far below any tolerance applied to the GPU
 *   result.
 *
 * Layouts: A is row-major M x K with leading dimension lda (A[i*lda + k]).
 *   B is either K x N row-major (layout KN: B[k*ldb + j]) or stored N x K
 *   row-major (layout NK: B[j*ldb + k]).  Elements are 16-bit patterns
 *   (FP16, BF16), 8-bit patterns (FP8 E4M3, E5M2) or 32-bit FP32 patterns
 *   taken as TF32.
 *
 * FP32 operands (the pages pick a separate, smaller tile for them in
 * "Writing high-performance matrix multiplication with NVIDIA CUDA Tile",
 * section "Launching the kernel from the host", and say no more about how
 * they are multiplied) are read as TF32: sign, 8-bit exponent and the top 10
 * fraction bits, the low 13 fraction bits dropped (truncation toward zero),
 * which is how the tensor core reads 32-bit containers.  Every product of
 * two TF32 values is exact in double (at most 22 significant bits).
 *
 * Pins (tests/test_oracle_pins.py): exact rational brute force on tiny
 * shapes, identity and permutation matrices, integer inputs with an exact
 * result, linearity in B, numpy float64 matmul, and numpy/torch casts for the
 * rounding routine.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <pthread.h>

enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_F32 = 2, ORC_E4M3 = 3, ORC_E5M2 = 4, ORC_TF32 = 5 };
enum { ORC_B_KN = 0, ORC_B_NK = 1 };

/* ---- input decoding (IEEE binary16 and bfloat16 bit patterns) ---------- */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double decode_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24);                 /* subnormal: frac * 2^-24 */
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(frac | 0x400), expo - 25); /* 1.frac * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
static double decode_bf16(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int expo = (b >> 7) & 0xff;
    int frac = b & 0x7f;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -133);                /* subnormal: frac * 2^-133 */
    else if (expo == 255)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(frac | 0x80), expo - 134); /* 1.frac * 2^(e-127) */
    return sign ? -v : v;
}

/* FP8 E4M3 (the "fn" variant: no infinities): 1 sign, 4 exponent bits (bias
 * 7), 3 fraction bits; S.1111.111 is NaN, the largest finite value 448. */
static double decode_e4m3(uint8_t b)
{
    int sign = (b >> 7) & 1, expo = (b >> 3) & 0xf, frac = b & 7;
    double v;
    if (expo == 15 && frac == 7)
        v = NAN;
    else if (expo == 0)
        v = ldexp((double)frac, -9);                  /* subnormal: frac/8 * 2^-6 */
    else
        v = ldexp((double)(frac | 8), expo - 10);     /* 1.frac * 2^(e-7) */
    return sign ? -v : v;
}

/* FP8 E5M2: 1 sign, 5 exponent bits (bias 15), 2 fraction bits, IEEE-style
 * infinities and NaNs. */
static double decode_e5m2(uint8_t b)
{
    int sign = (b >> 7) & 1, expo = (b >> 2) & 0x1f, frac = b & 3;
    double v;
    if (expo == 31)
        v = frac ? NAN : INFINITY;
    else if (expo == 0)
        v = ldexp((double)frac, -16);                 /* subnormal: frac/4 * 2^-14 */
    else
        v = ldexp((double)(frac | 4), expo - 17);     /* 1.frac * 2^(e-15) */
    return sign ? -v : v;
}

/* TF32 from an FP32 pattern: keep sign, exponent and the top 10 fraction
 * bits.  Clearing bits only ever moves a finite value toward zero; zeros,
 * subnormals and infinities keep their class (a NaN whose payload sits only
 * in the dropped bits would read as an infinity). */
static double decode_tf32(uint32_t u)
{
    uint32_t t = u & 0xffffe000u;
    float f;
    memcpy(&f, &t, sizeof f);
    return (double)f;
}

static double g_table[5][65536];
static int g_table_ready[5];
static pthread_mutex_t g_table_lock = PTHREAD_MUTEX_INITIALIZER;

static const double *decode_table(int dtype)
{
    pthread_mutex_lock(&g_table_lock);
    if (!g_table_ready[dtype]) {
        for (uint32_t u = 0; u < 65536; ++u)
            g_table[dtype][u] = dtype == ORC_F16    ? decode_f16((uint16_t)u)
                                : dtype == ORC_BF16 ? decode_bf16((uint16_t)u)
                                : dtype == ORC_E4M3 ? decode_e4m3((uint8_t)u)
                                                    : decode_e5m2((uint8_t)u);
        g_table_ready[dtype] = 1;
    }
    pthread_mutex_unlock(&g_table_lock);
    return g_table[dtype];
}

double oracle_decode(uint32_t bits, int dtype)
{
    if (dtype == ORC_F16) return decode_f16((uint16_t)bits);
    if (dtype == ORC_BF16) return decode_bf16((uint16_t)bits);
    if (dtype == ORC_E4M3) return decode_e4m3((uint8_t)bits);
    if (dtype == ORC_E5M2) return decode_e5m2((uint8_t)bits);
    if (dtype == ORC_F32) {
        float f;
        uint32_t u = bits;
        memcpy(&f, &u, sizeof f);
        return (double)f;
    }
    if (dtype == ORC_TF32) return decode_tf32(bits);
    return NAN;
}

/* ---- one output element: the defining dot product ---------------------- */

typedef struct {
    int64_t M, N, K;
    const void *A; int64_t lda;
    const void *B; int64_t ldb; int b_layout;
    const double *tab;                              /* decode table of 8/16-bit patterns (NULL for TF32) */
    int esz;                                        /* bytes per input element: 2, 1 for FP8, 4 for TF32 */
} problem_t;

/* Value of element `idx` of an input array. */
static double elem(const problem_t *p, const void *base, int64_t idx)
{
    if (p->esz == 4) return decode_tf32(((const uint32_t *)base)[idx]);
    return p->tab[p->esz == 1 ? ((const uint8_t *)base)[idx] : ((const uint16_t *)base)[idx]];
}

static void dot(const problem_t *p, int64_t i, int64_t j, double *c, double *bound)
{
    double s = 0.0, r = 0.0;
    const int64_t arow = i * p->lda;
    if (p->b_layout == ORC_B_NK) {
        const int64_t bcol = j * p->ldb;            /* column j of B is row j of the N x K store */
        for (int64_t k = 0; k < p->K; ++k) {
            double a = elem(p, p->A, arow + k), b = elem(p, p->B, bcol + k);
            s += a * b;
            r += fabs(a) * fabs(b);
        }
    } else {
        for (int64_t k = 0; k < p->K; ++k) {
            double a = elem(p, p->A, arow + k), b = elem(p, p->B, k * p->ldb + j);
            s += a * b;
            r += fabs(a) * fabs(b);
        }
    }
    *c = s;
    *bound = r;
}

/* ---- full or partial products, optionally threaded --------------------- */

typedef struct {
    const problem_t *p;
    int64_t first, last;          /* work items [first, last) */
    /* rows mode: C and Bound hold rows [row0, ...) */
    int64_t row0;
    double *C; int64_t ldc; double *Bound; int64_t ldbound;
    /* element mode */
    const int64_t *ii, *jj; double *out, *out_bound;
} work_t;

static void *rows_worker(void *arg)
{
    work_t *w = (work_t *)arg;
    for (int64_t i = w->first; i < w->last; ++i)
        for (int64_t j = 0; j < w->p->N; ++j) {
            double c, b;
            dot(w->p, i, j, &c, &b);
            w->C[(i - w->row0) * w->ldc + j] = c;
            if (w->Bound) w->Bound[(i - w->row0) * w->ldbound + j] = b;
        }
    return NULL;
}

static void *elems_worker(void *arg)
{
    work_t *w = (work_t *)arg;
    for (int64_t t = w->first; t < w->last; ++t)
        dot(w->p, w->ii[t], w->jj[t], &w->out[t], &w->out_bound[t]);
    return NULL;
}

static int run_split(void *(*fn)(void *), work_t proto, int64_t first, int64_t last, int threads)
{
    int64_t total = last - first;
    if (total <= 0) return 0;
    int nt = threads < 1 ? 1 : (threads > 256 ? 256 : threads);
    if ((int64_t)nt > total) nt = (int)total;
    pthread_t tid[256];
    work_t w[256];
    int inline_run[256];
    for (int t = 0; t < nt; ++t) {
        w[t] = proto;
        w[t].first = first + total * t / nt;
        w[t].last = first + total * (t + 1) / nt;
        inline_run[t] = (nt == 1) || pthread_create(&tid[t], NULL, fn, &w[t]) != 0;
        if (inline_run[t]) fn(&w[t]);
    }
    for (int t = 0; t < nt; ++t)
        if (!inline_run[t]) pthread_join(tid[t], NULL);
    return 0;
}

static int in_esz(int in_dtype)
{
    return in_dtype == ORC_TF32 ? 4 : (in_dtype == ORC_E4M3 || in_dtype == ORC_E5M2) ? 1 : 2;
}

static int check_problem(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int b_layout, int in_dtype)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (in_dtype != ORC_F16 && in_dtype != ORC_BF16 && in_dtype != ORC_E4M3 && in_dtype != ORC_E5M2 &&
        in_dtype != ORC_TF32)
        return -1;
    if (b_layout != ORC_B_KN && b_layout != ORC_B_NK) return -1;
    if (lda < K) return -1;
    if (b_layout == ORC_B_KN ? ldb < N : ldb < K) return -1;
    return 0;
}

/*
 * Rows [row_begin, row_end) of C (all N columns) and of the bound
 * sum_k |A_ik||B_kj|.  Row i of C lands at C[(i - row_begin) * ldc], the
 * same for Bound, which may be NULL.  Returns 0 on success, -1 on a bad argument.
 */
int oracle_gemm_rows(int64_t M, int64_t N, int64_t K,
                     const void *A, int64_t lda,
                     const void *B, int64_t ldb, int b_layout, int in_dtype,
                     int64_t row_begin, int64_t row_end,
                     double *C, int64_t ldc, double *Bound, int64_t ldbound, int threads)
{
    if (check_problem(M, N, K, lda, ldb, b_layout, in_dtype)) return -1;
    if (row_begin < 0 || row_end > M || row_begin > row_end) return -1;
    problem_t p = {M, N, K, A, lda, B, ldb, b_layout, in_dtype == ORC_TF32 ? NULL : decode_table(in_dtype),
                   in_esz(in_dtype)};
    work_t proto;
    memset(&proto, 0, sizeof proto);
    proto.p = &p; proto.row0 = row_begin; proto.C = C; proto.ldc = ldc; proto.Bound = Bound; proto.ldbound = ldbound;
    return run_split(rows_worker, proto, row_begin, row_end, threads);
}

/* The full product: rows [0, M). */
int oracle_gemm(int64_t M, int64_t N, int64_t K,
                const void *A, int64_t lda,
                const void *B, int64_t ldb, int b_layout, int in_dtype,
                double *C, int64_t ldc, double *Bound, int64_t ldbound, int threads)
{
    return oracle_gemm_rows(M, N, K, A, lda, B, ldb, b_layout, in_dtype, 0, M,
                            C, ldc, Bound, ldbound, threads);
}

/*
 * Selected elements (ii[t], jj[t]) for t < count: out[t] = C[ii][jj],
 * out_bound[t] = sum_k |A_ik||B_kj|.  Used for sampled checks at sizes where
 * the full product would take too long.
 */
int oracle_gemm_elements(int64_t M, int64_t N, int64_t K,
                         const void *A, int64_t lda,
                         const void *B, int64_t ldb, int b_layout, int in_dtype,
                         int64_t count, const int64_t *ii, const int64_t *jj,
                         double *out, double *out_bound, int threads)
{
    if (check_problem(M, N, K, lda, ldb, b_layout, in_dtype)) return -1;
    for (int64_t t = 0; t < count; ++t)
        if (ii[t] < 0 || ii[t] >= M || jj[t] < 0 || jj[t] >= N) return -1;
    problem_t p = {M, N, K, A, lda, B, ldb, b_layout, in_dtype == ORC_TF32 ? NULL : decode_table(in_dtype),
                   in_esz(in_dtype)};
    work_t proto;
    memset(&proto, 0, sizeof proto);
    proto.p = &p; proto.ii = ii; proto.jj = jj; proto.out = out; proto.out_bound = out_bound;
    return run_split(elems_worker, proto, 0, count, threads);
}

/* ---- output rounding and the unit in the last place -------------------- */

/* Precision p (significant bits incl. the implicit one), minimum normal
 * exponent and maximum exponent of each output format. */
static void format_of(int dtype, int *p, int *emin, int *emax)
{
    switch (dtype) {
    case ORC_F16:  *p = 11; *emin = -14;  *emax = 15;  break;
    case ORC_BF16: *p = 8;  *emin = -126; *emax = 127; break;
    default:       *p = 24; *emin = -126; *emax = 127; break;
    }
}

/*
 * Spacing of the output format at |x|: 2^(max(floor(log2|x|), emin) - p + 1).
 * For |x| below the smallest normal (and for 0) this is the subnormal spacing.
 * This is the "one unit in the last place of the output dtype" term of the
 * acceptance bound.
 */
double oracle_ulp(double x, int dtype)
{
    int p, emin, emax;
    format_of(dtype, &p, &emin, &emax);
    double a = fabs(x);
    int e = emin;
    if (a != 0.0 && isfinite(a)) {
        int ex;
        frexp(a, &ex);             /* a = f * 2^ex, f in [0.5, 1): floor(log2 a) = ex - 1 */
        if (ex - 1 > e) e = ex - 1;
        if (e > emax) e = emax;
    }
    return ldexp(1.0, e - p + 1);
}

/*
 * Round a double to the output format, round-to-nearest-even, overflow to
 * +-infinity, and return its bit pattern (16 bits for F16/BF16, 32 for F32).
 * The value is first rounded to a multiple of the format's spacing at |x|
 * (exact power-of-two scaling, then nearbyint, which rounds ties to even in
 * the default rounding mode); the result is then encoded field by field.
 */
uint32_t oracle_round_bits(double x, int dtype)
{
    int p, emin, emax;
    format_of(dtype, &p, &emin, &emax);
    int ebits = dtype == ORC_F16 ? 5 : 8;
    int fbits = p - 1;
    int bias = (1 << (ebits - 1)) - 1;
    uint32_t sign = signbit(x) ? 1u : 0u;
    uint32_t exp_all_ones = (1u << ebits) - 1u;
    uint32_t sign_bit = sign << (ebits + fbits);
    if (isnan(x))
        return (exp_all_ones << fbits) | (1u << (fbits - 1));      /* quiet NaN */
    double a = fabs(x);
    if (isinf(a))
        return sign_bit | (exp_all_ones << fbits);
    if (a == 0.0)
        return sign_bit;
    int ex;
    frexp(a, &ex);
    int e = ex - 1;
    if (e < emin) e = emin;
    double q = ldexp(1.0, e - fbits);          /* spacing in the binade of a */
    double r = nearbyint(a / q) * q;           /* a / q is exact: q is a power of two */
    double limit = ldexp(1.0, emax + 1);       /* first value past the largest finite */
    if (r >= limit)
        return sign_bit | (exp_all_ones << fbits);
    double min_normal = ldexp(1.0, emin);
    if (r < min_normal) {
        uint32_t frac = (uint32_t)(r / ldexp(1.0, emin - fbits));
        return sign_bit | frac;
    }
    int er;
    frexp(r, &er);
    er -= 1;                                    /* rounding may have moved r up one binade */
    uint32_t frac = (uint32_t)(r / ldexp(1.0, er - fbits)) - (1u << fbits);
    return sign_bit | ((uint32_t)(er + bias) << fbits) | frac;
}

/* ---- fused epilogue ----------------------------------------------------
 *
 * D[i][j] = act(alpha * C[i][j] + beta * Cin[i][j] + bias[j]), with C the
 * exact product from above, all in double.  act: 0 none, 1 ReLU max(x, 0),
 * 2 GELU in its tanh form, 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
 * The pages name epilogue fusion (the Croqtile tutorial's comparison with
 * cuBLAS) without defining one; this is the usual affine-plus-activation
 * form.  cin or bias may be NULL (treated as zero).  In place on D.
 */
static double act_apply(double x, int act)
{
    if (act == 1) return x > 0.0 ? x : 0.0;
    if (act == 2) {
        const double c = 0.7978845608028654;     /* sqrt(2 / pi) */
        return 0.5 * x * (1.0 + tanh(c * (x + 0.044715 * x * x * x)));
    }
    return x;
}

void oracle_epilogue(int64_t rows, int64_t cols, double *D, int64_t ldd, double alpha, double beta,
                     const double *cin, int64_t ldcin, const double *bias, int act)
{
    for (int64_t i = 0; i < rows; ++i)
        for (int64_t j = 0; j < cols; ++j) {
            double x = alpha * D[i * ldd + j];
            if (cin) x += beta * cin[i * ldcin + j];
            if (bias) x += bias[j];
            D[i * ldd + j] = act_apply(x, act);
        }
}

/* Vector forms for the test harness. */
void oracle_round_bits_n(const double *x, int64_t n, int dtype, uint32_t *out)
{
    for (int64_t t = 0; t < n; ++t) out[t] = oracle_round_bits(x[t], dtype);
}

void oracle_ulp_n(const double *x, int64_t n, int dtype, double *out)
{
    for (int64_t t = 0; t < n; ++t) out[t] = oracle_ulp(x[t], dtype);
}

void oracle_decode_n(const uint32_t *bits, int64_t n, int dtype, double *out)
{
    for (int64_t t = 0; t < n; ++t) out[t] = oracle_decode(bits[t], dtype);
}
