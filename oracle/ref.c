/*
 * CPU oracle for the skinny BF16 decode projection.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes (the plain definition of the operation):
 *
 *   ref[m][n] = sum_{k<K} x[m][k] * W[n][k]          (the projection)
 *   s[m][n]   = sqrt( sum_{k<K} (x[m][k] * W[n][k])^2 )
 *
 * Sources: page "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.gemm.
 * warp_splitk", class PreparedWarpSplitK docstring (out[M, N] = x[M, K] @
 * weight[N, K]^T, x and out packed row-major); page "vllm.models.glm5next.
 * nvidia.specialized_decode.gemm", class Projection (x @ weight.T).  The
 * second quantity s is the scale in the acceptance bound
 * |y - ref| <= 8e-3 |ref| + 2e-3 s that the tests apply.
 *
 * Arithmetic: the bf16 inputs are widened exactly to double (a bf16 value is
 * the top 16 bits of an IEEE binary32), each product is exact in double
 * (8 + 8 significand bits < 53), and the sum runs sequentially over k in
 * double.  Built with -O2 -fno-fast-math -ffp-contract=off so that no FMA
 * contraction or reassociation changes that order.  The optional OpenMP
 * loop only splits independent (m, n) outputs between threads.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 bit pattern -> exact double: the pattern is the high half of a binary32. */
static double bf16_bits_to_double(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

void oracle_bf16_to_f64(const uint16_t* bits, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_bits_to_double(bits[i]);
}

/*
 * Round a double to the nearest bf16 value, ties to even, by definition:
 * scale |v| so that its 8 significant bits sit left of the binary point,
 * round that to an integer (rint under the default round-to-nearest-even
 * mode), scale back.  bf16 shares binary32's exponent range: normals down
 * to 2^-126, subnormal spacing 2^-133, overflow to infinity past
 * (2 - 2^-8) * 2^127.
 */
static uint16_t double_to_bf16_bits(double v) {
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0x0000;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80);
    int e;
    (void)frexp(a, &e);           /* a = f * 2^e, 0.5 <= f < 1 */
    int shift = 8 - e;            /* a * 2^shift lies in [128, 256) */
    if (shift > 133) shift = 133; /* below 2^-126: fixed subnormal spacing 2^-133 */
    double q = rint(ldexp(a, shift));
    double r = ldexp(q, -shift);  /* exact: q has at most 9 significant bits */
    float f = (float)r;           /* exact for finite r; 2^128 becomes +inf */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

void oracle_round_bf16(const double* v, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = double_to_bf16_bits(v[i]);
}

/* IEEE binary16 bit pattern -> exact double: sign, 5-bit exponent (bias 15),
 * 10-bit fraction; exponent 0 holds zero and subnormals (fraction * 2^-24),
 * exponent 31 holds infinities and NaNs. */
static double fp16_bits_to_double(uint16_t bits) {
    const int sign = bits >> 15;
    const int e = (bits >> 10) & 0x1F;
    const int f = bits & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

void oracle_fp16_to_f64(const uint16_t* bits, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = fp16_bits_to_double(bits[i]);
}

/*
 * out[M, N] = x[M, K] @ W[N, K]^T in double, for 16-bit inputs of the given
 * type (0 = bf16, 1 = fp16; both operands the same type).  x has row pitch
 * ldx elements, W row pitch ldw elements; ref and s are dense [M, N].  s may
 * be NULL.  nthreads <= 0 means "OpenMP default"; without OpenMP the loop is
 * serial.
 */
void oracle_projection_typed(const uint16_t* x, int64_t ldx, const uint16_t* w, int64_t ldw,
                             int64_t M, int64_t N, int64_t K, double* ref, double* s,
                             int nthreads, int dtype) {
    double (*widen)(uint16_t) = dtype == 1 ? fp16_bits_to_double : bf16_bits_to_double;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
    for (int64_t n = 0; n < N; ++n) {
        const uint16_t* wn = w + n * ldw;
        for (int64_t m = 0; m < M; ++m) {
            const uint16_t* xm = x + m * ldx;
            double acc = 0.0, sq = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = widen(xm[k]) * widen(wn[k]);
                acc += p;
                sq += p * p;
            }
            ref[m * N + n] = acc;
            if (s) s[m * N + n] = sqrt(sq);
        }
    }
}

/* The bf16 projection (the operation's own input type). */
void oracle_projection(const uint16_t* x, int64_t ldx, const uint16_t* w, int64_t ldw,
                       int64_t M, int64_t N, int64_t K, double* ref, double* s,
                       int nthreads) {
    oracle_projection_typed(x, ldx, w, ldw, M, N, K, ref, s, nthreads, 0);
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
