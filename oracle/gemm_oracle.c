/*
 * Oracle for the dense fp16 matrix product C = A * B — TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow and meant to be obviously correct: a stride-aware triple loop that
 * decodes each fp16 operand to double, accumulates the K products in double and
 * rounds the sum once to fp16 (round to nearest, ties to even).  It shares no
 * code with the GPU library and is only loaded by the tests, the smoke check and
 * the bench's CPU-baseline leg.
 *
 * What it follows:
 *  - the definition C[m,n] = sum_k A[m,k] * B[k,n]: TileLang tutorial ch. 14
 *    "GEMM operators", section 2.1 (rung 1, the naive blocked version) and the
 *    AI-infra knowledge base page "Matrix multiplication and memory-access
 *    optimisation", section 02 (the direct triple loop);
 *  - element offsets from strides, in elements, A at m*s_am + k*s_ak and B at
 *    k*s_bk + n*s_bn, with 64-bit index arithmetic done before the multiply:
 *    "Triton GEMM: from one output tile to addresses, boundaries and data reuse",
 *    sections "Shape states the meaning, stride decides the address" and
 *    "Putting addresses and boundaries into a short kernel";
 *  - the precision points fp16 inputs, wide accumulation, one final rounding to
 *    fp16 (which may round or overflow): same Triton page, the paragraph on the
 *    three precision positions after the wrapper.  The oracle accumulates in
 *    double, wider than the kernel's fp32, so it is the higher-precision
 *    reference on the same fp16 inputs that the page's testing section asks for.
 *
 * fp16 <-> double conversions are written here from the IEEE 754 binary16
 * format (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits;
 * subnormals; exponent 31 for inf/NaN).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* binary16 bits -> double (exact: every binary16 value is a double). */
double oracle_half_to_double(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1f;
    const int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);               /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);   /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* Round a non-negative double to an integer, ties to even. */
static double round_half_even(double v)
{
    double fl = floor(v);
    double d = v - fl;                            /* exact for v < 2^52 */
    if (d > 0.5) return fl + 1.0;
    if (d < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* double -> binary16 bits, round to nearest even; overflow to +-inf; NaN kept. */
uint16_t oracle_double_to_half(double x)
{
    const uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return (uint16_t)(sign | 0x7e00);
    double a = fabs(x);
    /* The largest finite half is 65504 = 2047 * 2^5; the midpoint to the next
       step (2^16) is 65520 and ties to the even significand 2048, i.e. inf. */
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: the value is q * 2^-24 with q an integer 0..1024
           (q == 1024 is the smallest normal, which the same bits encode). */
        double q = round_half_even(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)q);
    }
    int e2;
    frexp(a, &e2);                    /* a = r * 2^e2, r in [0.5, 1) */
    int E = e2 - 1;                   /* a in [2^E, 2^(E+1)), E in [-14, 15] */
    double q = round_half_even(ldexp(a, 10 - E));   /* in [1024, 2048] */
    if (q == 2048.0) { q = 1024.0; E += 1; }
    if (E > 15) return (uint16_t)(sign | 0x7c00);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)((int)q - 1024));
}

/* Decode table, filled once from oracle_half_to_double. */
static double g_dec[65536];
static int g_dec_ready = 0;

static void ensure_table(void)
{
    if (g_dec_ready) return;
    for (int i = 0; i < 65536; ++i) g_dec[i] = oracle_half_to_double((uint16_t)i);
    g_dec_ready = 1;
}

void oracle_init(void) { ensure_table(); }

/*
 * C[m*ldc + n] = fp16( sum_{k<K} A[m*s_am + k*s_ak] * B[k*s_bk + n*s_bn] )
 * for 0 <= m < M, 0 <= n < N.  Accumulation in double in order k = 0..K-1.
 * Elements of C outside the M x N view are not touched.  `threads` > 1 splits
 * the output rows over OpenMP threads (each element's sum is unchanged).
 */
void oracle_gemm_f16(const uint16_t *A, int64_t s_am, int64_t s_ak,
                     const uint16_t *B, int64_t s_bk, int64_t s_bn,
                     uint16_t *C, int64_t ldc,
                     int64_t M, int64_t N, int64_t K, int threads)
{
    ensure_table();
    if (threads < 1) threads = 1;
#pragma omp parallel for num_threads(threads) schedule(dynamic, 1)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += g_dec[A[m * s_am + k * s_ak]] * g_dec[B[k * s_bk + n * s_bn]];
            C[m * ldc + n] = oracle_double_to_half(acc);
        }
    }
}

/*
 * The same sums left unrounded: S[m*lds + n] = sum_{k<K} A[..] * B[..] in
 * double, k = 0..K-1.  The fused-epilogue oracle applies its bias, activation
 * and gate product to these before its single rounding to fp16.
 */
void oracle_gemm_f64(const uint16_t *A, int64_t s_am, int64_t s_ak,
                     const uint16_t *B, int64_t s_bk, int64_t s_bn,
                     double *S, int64_t lds,
                     int64_t M, int64_t N, int64_t K, int threads)
{
    ensure_table();
    if (threads < 1) threads = 1;
#pragma omp parallel for num_threads(threads) schedule(dynamic, 1)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += g_dec[A[m * s_am + k * s_ak]] * g_dec[B[k * s_bk + n * s_bn]];
            S[m * lds + n] = acc;
        }
    }
}

/*
 * Sampled form of the same definition, for outputs too many to compute whole:
 * out[i] = fp16( sum_k A[a_off[i] + k*s_ak] * B[b_off[i] + k*s_bk] ), where
 * a_off[i] = m_i*s_am (start of row m_i of A) and b_off[i] = n_i*s_bn (start of
 * column n_i of B) are supplied by the caller, who may also pass compacted
 * copies of just the needed rows/columns.  exact[i] receives the double sum
 * before rounding (may be NULL).
 */
void oracle_dot_f16(const uint16_t *A, const int64_t *a_off, int64_t s_ak,
                    const uint16_t *B, const int64_t *b_off, int64_t s_bk,
                    int64_t K, int64_t count, uint16_t *out, double *exact,
                    int threads)
{
    ensure_table();
    if (threads < 1) threads = 1;
#pragma omp parallel for num_threads(threads) schedule(static)
    for (int64_t i = 0; i < count; ++i) {
        double acc = 0.0;
        const uint16_t *a = A + a_off[i];
        const uint16_t *b = B + b_off[i];
        for (int64_t k = 0; k < K; ++k)
            acc += g_dec[a[k * s_ak]] * g_dec[b[k * s_bk]];
        out[i] = oracle_double_to_half(acc);
        if (exact) exact[i] = acc;
    }
}

/* Bulk conversions, used by the oracle's own pins. */
void oracle_half_to_double_n(const uint16_t *h, double *d, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) d[i] = oracle_half_to_double(h[i]);
}

void oracle_double_to_half_n(const double *d, uint16_t *h, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) h[i] = oracle_double_to_half(d[i]);
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
