/*
 * Oracle for the fused tensor-parallel matmul + collective operators.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link
 * or call this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header or table with the CUDA
 * path.
 *
 * What it computes (plain definitions, fp64 arithmetic):
 *
 *   The MindSpeed developer guide page on compute-communication parallelism
 *   (CoC), section "problem analysis" (问题分析), states the problem: in a
 *   tensor-parallel ColumnParallelLinear / RowParallelLinear the matmul is
 *   followed by AllReduce (no sequence parallelism) or by AllGather /
 *   ReduceScatter (sequence parallelism).  Section "fused-operator
 *   implementation" (融合算子实现) lists the fused operators.  With R ranks and
 *   rank r holding X_r and W_r, the per-rank partial product is
 *
 *       P_r[i, j] = sum_{t < k_r} X_r[i, t] * W_r[t, j]
 *
 *   and every operator is a composition of these partials (AllReduce sums
 *   them, ReduceScatter sums and hands rank r its row block, AllGather
 *   concatenates the X_r along rows first).  This file holds the pieces that
 *   need speed: exact decoding of the 16-bit input formats, IEEE binary16
 *   round-to-nearest-even encoding (for the w8A16 dequantisation, same page,
 *   "fused-operator implementation", last bullet) and the fp64 partial-product
 *   accumulation over a subset of output rows.  The Python side (oracle.py)
 *   composes them into the five operators.
 *
 * Built with -ffp-contract=off so that "acc += x * w" is a rounded multiply
 * followed by a rounded add on every host (no fused multiply-add on one host
 * and not on another).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- 16-bit formats ----------------------------------------------------
 * IEEE 754-2008 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits.  Exponent field 0 encodes zero / subnormals (value = f * 2^-24),
 * field 31 encodes inf / NaN.  Otherwise value = (1024 + f) * 2^(e - 25).
 */
double oracle_f16_to_f64(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1f;
    const int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + f), e - 25);
    }
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32; widening is exact. */
double oracle_bf16_to_f64(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round an exact double to the nearest binary16, ties to even (IEEE 754
 * roundTiesToEven), overflowing to +-inf.  Written from the definition: find
 * the binary16 quantum of |x|'s binade (2^(e-10) for normals, 2^-24 in the
 * subnormal range), express |x| in quanta (an exact power-of-two scaling),
 * round that to the nearest integer with ties to even, and re-encode. */
uint16_t oracle_f64_to_f16_rne(double x)
{
    const uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return (uint16_t)(sign | 0x7e00);
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7c00);
    if (a == 0.0) return sign;

    int E;
    (void)frexp(a, &E);     /* a = f * 2^E, f in [0.5, 1)  =>  a in [2^(E-1), 2^E) */
    int e = E - 1;          /* a in [2^e, 2^(e+1)) */
    if (e < -14) e = -14;   /* subnormal range shares the quantum 2^-24 */
    const double q = ldexp(1.0, e - 10);
    const double nq = a / q;            /* exact: division by a power of two */
    double fl = floor(nq);
    const double frac = nq - fl;        /* exact */
    if (frac > 0.5 || (frac == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
    /* fl is now an integer in [0, 2048] */
    uint32_t n = (uint32_t)fl;
    if (e == -14 && n < 1024) {
        return (uint16_t)(sign | n);    /* subnormal (or zero) */
    }
    if (n == 2048) { n = 1024; e += 1; }
    if (e + 15 >= 31) return (uint16_t)(sign | 0x7c00);
    return (uint16_t)(sign | ((uint32_t)(e + 15) << 10) | (n - 1024));
}

/* Round an exact double to the nearest bfloat16, ties to even, overflowing to
 * +-inf.  bfloat16 is binary32's sign, 8 exponent bits (bias 127) and the top
 * 7 fraction bits: in the binade [2^e, 2^(e+1)) the quantum is 2^(e-7), and
 * below 2^-126 the subnormal quantum 2^-133.  Same method as the binary16
 * encoder above: count quanta exactly, round ties to even, re-encode. */
uint16_t oracle_f64_to_bf16_rne(double x)
{
    const uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return (uint16_t)(sign | 0x7fc0);
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7f80);
    if (a == 0.0) return sign;

    int E;
    (void)frexp(a, &E);
    int e = E - 1;            /* a in [2^e, 2^(e+1)) */
    if (e < -126) e = -126;   /* subnormal range shares the quantum 2^-133 */
    const double q = ldexp(1.0, e - 7);
    const double nq = a / q;
    double fl = floor(nq);
    const double frac = nq - fl;
    if (frac > 0.5 || (frac == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
    /* fl is now an integer in [0, 256] */
    uint32_t n = (uint32_t)fl;
    if (e == -126 && n < 128) {
        return (uint16_t)(sign | n);    /* subnormal (or zero) */
    }
    if (n == 256) { n = 128; e += 1; }
    if (e + 127 >= 255) return (uint16_t)(sign | 0x7f80);
    return (uint16_t)(sign | ((uint32_t)(e + 127) << 7) | (n - 128));
}

static inline double decode16(int dtype, uint16_t v)
{
    return dtype == 1 ? oracle_bf16_to_f64(v) : oracle_f16_to_f64(v);
}

/* Bulk helpers so that the Python side never decodes element by element. */
void oracle_decode16(int dtype, const uint16_t* in, double* out, int64_t count)
{
    for (int64_t i = 0; i < count; ++i) out[i] = decode16(dtype, in[i]);
}

void oracle_encode_f16(const double* in, uint16_t* out, int64_t count)
{
    for (int64_t i = 0; i < count; ++i) out[i] = oracle_f64_to_f16_rne(in[i]);
}

void oracle_encode_bf16(const double* in, uint16_t* out, int64_t count)
{
    for (int64_t i = 0; i < count; ++i) out[i] = oracle_f64_to_bf16_rne(in[i]);
}

/* ---- one rank's partial product -------------------------------------------
 * acc[i, j] += sum_{t=0}^{k-1} X[rows[i], t] * W[t, j]      (fp64)
 *
 * X is a row-major 16-bit matrix with leading dimension ldx (elements), W a
 * row-major k x n 16-bit matrix with leading dimension ldw; dtype 0 = binary16,
 * 1 = bfloat16.  acc is nrows x n, row-major, and is added to, so calling this
 * for r = 0, 1, ..., R-1 forms sum_r P_r with every output element summed in
 * the order (r ascending, t ascending).  Threads split the output columns; each
 * element is owned by one thread, so the summation order does not depend on
 * the thread count.
 */
void oracle_accumulate_partial(int dtype,
                               const uint16_t* x, int64_t ldx,
                               const uint16_t* w, int64_t ldw,
                               int64_t k, int64_t n,
                               const int64_t* rows, int64_t nrows,
                               double* acc, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
    {
        int tid = 0, nth = 1;
#ifdef _OPENMP
        tid = omp_get_thread_num();
        nth = omp_get_num_threads();
#endif
        const int64_t j0 = n * tid / nth;
        const int64_t j1 = n * (tid + 1) / nth;
        const int64_t width = j1 - j0;
        double* wrow = (double*)malloc((size_t)(width > 0 ? width : 1) * sizeof(double));
        if (wrow != NULL && width > 0) {
            for (int64_t t = 0; t < k; ++t) {
                const uint16_t* wt = w + t * ldw + j0;
                for (int64_t j = 0; j < width; ++j) wrow[j] = decode16(dtype, wt[j]);
                for (int64_t i = 0; i < nrows; ++i) {
                    const double xv = decode16(dtype, x[rows[i] * ldx + t]);
                    double* a = acc + i * n + j0;
                    for (int64_t j = 0; j < width; ++j) a[j] += xv * wrow[j];
                }
            }
        }
        free(wrow);
    }
}

/* ---- w8A16 pseudo-quantised weight ------------------------------------------
 * Same page, "fused-operator implementation", last bullet: MATMUL_ALL_REDUCE
 * supports w8A16 pseudo-quantisation in fp16 at per-tensor, per-channel and
 * per-group granularity.  Reading (the page gives no formula): symmetric,
 * no zero point, one binary16 scale per granule, and
 *
 *     Wd[t, j] = binary16_RNE( q[t, j] * s(t, j) )
 *
 * with the product taken exactly in fp64 (an 8-bit integer times a binary16
 * scale has at most 19 significant bits).  q is this rank's k x n slab, whose
 * first row is row k_offset of the full K x n weight.  s(t, j) is
 *     gran 0 (per tensor):  scale[0]
 *     gran 1 (per channel): scale[j]                      (one per output column)
 *     gran 2 (per group):   scale[((k_offset + t) / group) * n + j]
 *                           (groups of `group` consecutive rows of the full K)
 */
void oracle_dequant_w8(const int8_t* q, int64_t k, int64_t n,
                       const uint16_t* scale, int gran, int64_t group,
                       int64_t k_offset, uint16_t* out)
{
    for (int64_t t = 0; t < k; ++t) {
        for (int64_t j = 0; j < n; ++j) {
            int64_t si = 0;
            if (gran == 1) si = j;
            else if (gran == 2) si = ((k_offset + t) / group) * n + j;
            const double s = oracle_f16_to_f64(scale[si]);
            out[t * n + j] = oracle_f64_to_f16_rne((double)q[t * n + j] * s);
        }
    }
}

/* ---- w8A16 extensions: zero point and bfloat16 activations -------------------
 * The page names the fp16 form only; these are the asymmetric and bfloat16
 * readings.  With an int8 zero point z(t, j) laid out like the scale (NULL:
 * symmetric, z = 0) and the activation type `dtype` (0 binary16, 1 bfloat16,
 * which is also the type of the scale and of the result):
 *
 *     Wd[t, j] = RNE_dtype( (q[t, j] - z(t, j)) * s(t, j) )
 *
 * (q - z) is an integer in [-255, 255] and the product is exact in fp64, so
 * the result is rounded once.  z(t, j) is indexed exactly like s(t, j).
 */
void oracle_dequant_w8_ex(const int8_t* q, int64_t k, int64_t n,
                          const uint16_t* scale, const int8_t* zero, int gran, int64_t group,
                          int64_t k_offset, int dtype, uint16_t* out)
{
    for (int64_t t = 0; t < k; ++t) {
        for (int64_t j = 0; j < n; ++j) {
            int64_t si = 0;
            if (gran == 1) si = j;
            else if (gran == 2) si = ((k_offset + t) / group) * n + j;
            const double s = decode16(dtype, scale[si]);
            const double z = zero ? (double)zero[si] : 0.0;
            const double v = ((double)q[t * n + j] - z) * s;
            out[t * n + j] = dtype == 1 ? oracle_f64_to_bf16_rne(v) : oracle_f64_to_f16_rne(v);
        }
    }
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
