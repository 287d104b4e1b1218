/*
 * sfar_oracle.c -- CPU oracle for the small-message AllReduce.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file.  It shares no code, header,
 * table or helper with the GPU library, and the GPU library never calls it.
 *
 * What it computes (the plain definition of an AllReduce, with the order and
 * rounding fixed):
 *   "Every Microsecond Counts" (page 1), section "Unified primitives and API
 *   design": recvReduce receives every peer's value and sums it in registers;
 *   the one-shot kernel reads its local value, broadcasts it, reduces what it
 *   receives and writes the result, so every rank ends with the same sum.
 *   Section "Tensor parallelism and AllReduce": the partial results of all
 *   GPUs are added and the total is handed back to every GPU.
 * The pages do not fix an order or a precision.  This oracle takes the
 * reading the hot path is held to: for each element i,
 *     acc = widen(in[0][i]);  acc = acc (+) widen(in[q][i]) for q = 1..R-1
 * with (+) an IEEE binary32 add rounded to nearest-even, then ONE rounding of
 * acc to the output type (nearest-even), stored to out[r][i] for every r.
 *
 * dtype 0 = bf16 (stored as the upper 16 bits of a binary32), dtype 1 = fp32.
 * Widening bf16 -> fp32 is exact (the bits shifted left by 16).  Narrowing
 * fp32 -> bf16 is written out from the IEEE definition of round to nearest,
 * ties to even, on the 16 dropped bits; a NaN stays a NaN of the same sign.
 * Subnormals are kept (no flush to zero).
 *
 * Build with -O2 -ffp-contract=off -fno-fast-math (the only arithmetic is
 * additions; the flags rule out contraction and value-changing rewrites).
 *
 * ORACLE_MUTANT (compile-time, tests only): 0 = the oracle.  Other values
 * plant one plausible mistake each, so the tests can show that the pins on
 * this oracle catch it.  The shipped object is always built with 0.
 */
#include <float.h>
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#if FLT_EVAL_METHOD != 0
#error "the oracle needs binary32 arithmetic evaluated in binary32"
#endif

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

#define ORACLE_BF16 0
#define ORACLE_FP32 1

static float widen_bf16(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
#if ORACLE_MUTANT == 10
    /* mutant: flush subnormal inputs to zero */
    if ((u & 0x7f800000u) == 0) { u &= 0x80000000u; memcpy(&f, &u, sizeof f); }
#endif
    return f;
}

/* binary32 -> bf16, round to nearest, ties to even (IEEE 754 roundTiesToEven
 * applied to the 16 low-order significand bits that are dropped). */
static uint16_t narrow_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)           /* NaN: keep sign, make quiet */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t kept = u >> 16;                         /* sign, exponent, 7 fraction bits */
    uint32_t dropped = u & 0xffffu;
#if ORACLE_MUTANT == 5
    (void)dropped;                                   /* mutant: truncate */
#elif ORACLE_MUTANT == 11
    if (dropped >= 0x8000u) kept += 1;               /* mutant: ties away from zero */
#else
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1;                                   /* a carry into the exponent is
                                                        the correct result, up to inf */
#endif
    return (uint16_t)kept;
}

static float load_elem(const void *p, int dtype, size_t i)
{
    if (dtype == ORACLE_BF16)
        return widen_bf16(((const uint16_t *)p)[i]);
    float f;
    memcpy(&f, (const unsigned char *)p + 4 * i, sizeof f);
    return f;
}

static void store_elem(void *p, int dtype, size_t i, float v)
{
    if (dtype == ORACLE_BF16)
        ((uint16_t *)p)[i] = narrow_bf16(v);
    else
        memcpy((unsigned char *)p + 4 * i, &v, sizeof v);
}

/* The reduction of element i over the R ranks, in the fixed order 0..R-1. */
static float fold(int R, int dtype, const void *const *in, size_t n, size_t i)
{
    (void)n;
#if ORACLE_MUTANT == 1
    float acc = load_elem(in[R - 1], dtype, i);      /* mutant: reversed order */
    for (int q = R - 2; q >= 0; --q)
        acc = acc + load_elem(in[q], dtype, i);
#elif ORACLE_MUTANT == 2
    float acc = load_elem(in[0], dtype, i);          /* mutant: bf16 accumulator */
    for (int q = 1; q < R; ++q) {
        acc = acc + load_elem(in[q], dtype, i);
        if (dtype == ORACLE_BF16) acc = widen_bf16(narrow_bf16(acc));
    }
#elif ORACLE_MUTANT == 3
    float acc = 0.0f;                                /* mutant: start from +0 */
    for (int q = 0; q < R; ++q)
        acc = acc + load_elem(in[q], dtype, i);
#elif ORACLE_MUTANT == 4
    float acc = load_elem(in[0], dtype, i);          /* mutant: drops the last rank */
    for (int q = 1; q < R - 1; ++q)
        acc = acc + load_elem(in[q], dtype, i);
#elif ORACLE_MUTANT == 7
    /* mutant: pairwise tree instead of a left fold */
    float v[64];
    int m = R;
    for (int q = 0; q < R; ++q) v[q] = load_elem(in[q], dtype, i);
    while (m > 1) {
        int h = 0;
        for (int q = 0; q + 1 < m; q += 2) v[h++] = v[q] + v[q + 1];
        if (m & 1) v[h++] = v[m - 1];
        m = h;
    }
    float acc = v[0];
#elif ORACLE_MUTANT == 8
    float acc = load_elem(in[0], dtype, i);          /* mutant: reads a neighbour */
    for (int q = 1; q < R; ++q)
        acc = acc + load_elem(in[q], dtype, (i + 1 < n) ? i + 1 : i);
#elif ORACLE_MUTANT == 9
    float acc = load_elem(in[0], dtype, i);          /* mutant: subtracts the last rank */
    for (int q = 1; q < R; ++q) {
        float x = load_elem(in[q], dtype, i);
        acc = (q == R - 1) ? acc - x : acc + x;
    }
#else
    float acc = load_elem(in[0], dtype, i);
    for (int q = 1; q < R; ++q)
        acc = acc + load_elem(in[q], dtype, i);
#endif
    return acc;
}

static void allreduce_range(int R, int dtype, const void *const *in, void *const *out,
                            size_t n, size_t lo, size_t hi)
{
    for (size_t i = lo; i < hi; ++i) {
        float acc = fold(R, dtype, in, n, i);
#if ORACLE_MUTANT == 6
        store_elem(out[0], dtype, i, acc);           /* mutant: only rank 0 gets it */
#else
        for (int r = 0; r < R; ++r)
            store_elem(out[r], dtype, i, acc);
#endif
    }
}

/*
 * sfar_oracle_allreduce: R host arrays in[0..R-1] of n elements each (dtype
 * as above) are reduced element by element; the result is written to every
 * out[0..R-1].  Inputs and outputs are host memory owned by the caller and
 * must not overlap.  Returns 0, or -1 for a bad argument (R < 1, R > 64,
 * unknown dtype, a NULL pointer with n > 0).
 */
int sfar_oracle_allreduce(int R, size_t n, int dtype, const void *const *in, void *const *out)
{
    if (R < 1 || R > 64 || (dtype != ORACLE_BF16 && dtype != ORACLE_FP32))
        return -1;
    if (n == 0)
        return 0;
    if (!in || !out)
        return -1;
    for (int r = 0; r < R; ++r)
        if (!in[r] || !out[r])
            return -1;
    allreduce_range(R, dtype, in, out, n, 0, n);
    return 0;
}

struct oracle_job {
    int R, dtype;
    const void *const *in;
    void *const *out;
    size_t n, lo, hi;
};

static void *oracle_worker(void *arg)
{
    struct oracle_job *j = (struct oracle_job *)arg;
    allreduce_range(j->R, j->dtype, j->in, j->out, j->n, j->lo, j->hi);
    return NULL;
}

/*
 * sfar_oracle_allreduce_mt: the same result as sfar_oracle_allreduce, with the
 * element range split over `threads` POSIX threads (each element is still
 * folded by one thread in the same order, so the bits are identical).  Used to
 * time the oracle on several host cores.
 */
int sfar_oracle_allreduce_mt(int R, size_t n, int dtype, const void *const *in,
                             void *const *out, int threads)
{
    if (threads <= 1 || n < 4096)
        return sfar_oracle_allreduce(R, n, dtype, in, out);
    if (R < 1 || R > 64 || (dtype != ORACLE_BF16 && dtype != ORACLE_FP32) || !in || !out)
        return -1;
    for (int r = 0; r < R; ++r)
        if (!in[r] || !out[r])
            return -1;
    if (threads > 256)
        threads = 256;
    pthread_t tid[256];
    struct oracle_job job[256];
    size_t per = (n + (size_t)threads - 1) / (size_t)threads;
    int started = 0;
    for (int t = 0; t < threads; ++t) {
        size_t lo = (size_t)t * per, hi = lo + per;
        if (lo >= n) break;
        if (hi > n) hi = n;
        job[t] = (struct oracle_job){R, dtype, in, out, n, lo, hi};
        if (pthread_create(&tid[t], NULL, oracle_worker, &job[t]) != 0) {
            oracle_worker(&job[t]);
            tid[t] = 0;
        }
        started = t + 1;
    }
    for (int t = 0; t < started; ++t)
        if (tid[t]) pthread_join(tid[t], NULL);
    return 0;
}

/* ------------------------------------------------------------------------
 * The step after the AllReduce: residual add and RMS normalisation.
 *
 * "vLLM distributed inference core" (page 2), section one: in a decode step
 * the compute stream runs the normalisation right after the AllReduce of the
 * attention output projection and of the MLP down projection; section two
 * puts it on the compute stream after the wait for the AllReduce.  The pages
 * give no formula and no precision.  Readings taken (root-mean-square
 * normalisation of the residual stream, the form used by current decoder
 * models; every rounding spelled out so the result is unique):
 *
 *   a[j]   = the AllReduce result of element j of the row, in the element
 *            type (exactly what sfar_oracle_allreduce stores);
 *   z[j]   = T(a[j] (+) res[j])      binary32 add, one rounding to type T;
 *   ms     = ldexp(float(S) (/) h, 2E - F)
 *                                    S = sum_j z[j]^2 with every term
 *            truncated to a multiple of 2^(2E - F), where 2^E is the
 *            smallest power of two above every |z[j]| of the row and
 *            F = 53 - c, c = ceil(log2 h): the sum is then exact in 64-bit
 *            integers (< 2^53) and independent of the order (S counts
 *            units of 2^(2E - F)); float(S) rounds once to binary32, the
 *            division by h is a binary32 division, and the scaling by
 *            2^(2E - F) rounds only in the subnormal range; against the
 *            largest square of the row (>= 2^(2E - 2)) it is short of the
 *            exact sum of squares by less than h 2^(2 - F) <= 2^(2c - 51)
 *            (2^-25 for h = 8192); a NaN in the row makes ms NaN, otherwise
 *            an infinity makes it +inf, and an all-zero row gives 0;
 *   rstd   = 1 (/) sqrt(ms (+) eps)  binary32, each operation rounded;
 *   y[j]   = T((z[j] (*) rstd) (*) w[j])   binary32 products, one rounding
 *            to T.
 * Outputs per rank r: out[r] = y, res_out[r] = z.
 * ------------------------------------------------------------------------ */

/* smallest c >= 0 with 2^c >= h */
static int ceil_log2(size_t h)
{
    int c = 0;
    while (((size_t)1 << c) < h)
        ++c;
    return c;
}

/* ms of one row of z (h binary32 values, already rounded to the type). */
static float row_mean_square(const float *z, size_t h)
{
    int any_nan = 0, any_inf = 0;
    double maxabs = 0.0;
    for (size_t j = 0; j < h; ++j) {
        if (isnan(z[j])) any_nan = 1;
        else if (isinf(z[j])) any_inf = 1;
        else if (fabs((double)z[j]) > maxabs) maxabs = fabs((double)z[j]);
    }
    if (any_nan) return NAN;
    if (any_inf) return INFINITY;
    if (maxabs == 0.0) return 0.0f;
    int E;
    (void)frexp(maxabs, &E);                    /* maxabs = m 2^E, 1/2 <= m < 1 */
#if ORACLE_MUTANT == 17
    E += 8;                                      /* mutant: coarser fixed point */
#endif
    const int F = 53 - ceil_log2(h);
    uint64_t S = 0;
    for (size_t j = 0; j < h; ++j) {
        const double u = ldexp((double)z[j], -E);   /* |u| < 1, exact */
        S += (uint64_t)floor(ldexp(u * u, F));      /* u*u exact: <= 48 bits */
    }
#if ORACLE_MUTANT == 13
    const float q = (float)S / (float)(h > 1 ? h - 1 : 1);                     /* mutant: h - 1 */
#else
    const float q = (float)S / (float)h;
#endif
    return ldexpf(q, 2 * E - F);
}

static float round_to(int dtype, float v)
{
    return dtype == ORACLE_BF16 ? widen_bf16(narrow_bf16(v)) : v;
}

/*
 * sfar_oracle_add_rmsnorm: for every rank r and row i (rows x h elements per
 * rank, row-major), the definitions above.  do_allreduce = 1: a = the
 * AllReduce of in[0..R-1]; do_allreduce = 0: a = in[r] itself (the
 * normalisation step alone).  weight holds h elements (shared by all ranks);
 * res[r] / res_out[r] / out[r] hold rows x h elements.  res_out[r] may be
 * res[r].  Host memory owned by the caller.  Returns 0, or -1 for a bad
 * argument.
 */
int sfar_oracle_add_rmsnorm(int R, size_t rows, size_t h, int dtype, const void *const *in,
                            const void *const *res, const void *weight, float eps, void *const *out,
                            void *const *res_out, int do_allreduce)
{
    if (R < 1 || R > 64 || h == 0 || (dtype != ORACLE_BF16 && dtype != ORACLE_FP32))
        return -1;
    if (rows == 0)
        return 0;
    if (!in || !res || !weight || !out || !res_out)
        return -1;
    float *z = (float *)malloc(h * sizeof(float));
    if (!z)
        return -1;
    for (int r = 0; r < R; ++r) {
        for (size_t i = 0; i < rows; ++i) {
            for (size_t j = 0; j < h; ++j) {
                const size_t e = i * h + j;
                const float a = do_allreduce ? round_to(dtype, fold(R, dtype, in, rows * h, e))
                                             : load_elem(in[r], dtype, e);
#if ORACLE_MUTANT == 12
                z[j] = a;                                        /* mutant: residual dropped */
#elif ORACLE_MUTANT == 16
                z[j] = a + load_elem(res[r], dtype, e);          /* mutant: z not rounded */
#else
                z[j] = round_to(dtype, a + load_elem(res[r], dtype, e));
#endif
            }
            const float ms = row_mean_square(z, h);
#if ORACLE_MUTANT == 14
            const float rstd = 1.0f / sqrtf(ms) + eps;          /* mutant: eps outside */
#else
            const float rstd = 1.0f / sqrtf(ms + eps);
#endif
            for (size_t j = 0; j < h; ++j) {
                const size_t e = i * h + j;
                const float t = z[j] * rstd;
#if ORACLE_MUTANT == 15
                const float y = t;                               /* mutant: weight dropped */
#else
                const float y = t * load_elem(weight, dtype, j);
#endif
                store_elem(out[r], dtype, e, y);
                store_elem(res_out[r], dtype, e, z[j]);
            }
        }
    }
    free(z);
    return 0;
}

/* ------------------------------------------------------------------------
 * The producer of the AllReduce in a tensor-parallel decode layer: the
 * row-parallel projection (GEMV) of every rank.
 *
 * "vLLM distributed inference core" (page 2), section one: with tensor
 * parallelism each layer's attention output projection and MLP down
 * projection end in an AllReduce; section three: the compute stream runs
 * the matrix product, records an event, and the communication stream runs
 * the AllReduce after it.  Rank r holds the rows of the weight matrix that
 * match its slice of the input: y_r = x_r W_r, x_r of k elements, W_r of
 * k x h (row-major), y_r of h elements -- the partial sums the AllReduce
 * adds.  The pages fix no summation order; the reading taken is the plain
 * definition of a matrix-vector product written as one sum per output
 * (bf16 inputs and output): y[j] = x[0] W[0][j] + x[1] W[1][j] + ... +
 * x[k-1] W[k-1][j], evaluated from the left -- every product rounded to
 * binary32 (exact unless it under- or overflows: the significands have 8
 * bits), added in row order (row 0 first) to a binary32 accumulator that
 * starts at +0, each addition rounded to nearest even -- then one rounding
 * to bf16.
 * ------------------------------------------------------------------------ */
static float gemv_column(const uint16_t *x, const uint16_t *W, size_t k, size_t h, size_t j)
{
#if ORACLE_MUTANT == 21
    /* mutant: 8 segments of ceil(k / 8) consecutive rows, each summed from +0,
       the segment sums then folded in segment order */
    const size_t c = (k + 7) / 8;
    float total = 0.0f;
    for (size_t s0 = 0; s0 < k; s0 += c) {
        float part = 0.0f;
        for (size_t i = s0; i < s0 + c && i < k; ++i)
            part = part + widen_bf16(x[i]) * widen_bf16(W[i * h + j]);
        total = s0 == 0 ? part : total + part;
    }
    return total;
#endif
    float acc = 0.0f;
    for (size_t n = 0; n < k; ++n) {
#if ORACLE_MUTANT == 18
        const size_t i = k - 1 - n;                                           /* mutant: rows folded from the last */
#else
        const size_t i = n;
#endif
#if ORACLE_MUTANT == 20
        const float p = widen_bf16(x[i]) * widen_bf16(W[j * k + i]);         /* mutant: W transposed */
#else
        const float p = widen_bf16(x[i]) * widen_bf16(W[i * h + j]);
#endif
#if ORACLE_MUTANT == 19
        if (i + 1 == k) continue;                                            /* mutant: last row dropped */
#endif
        acc = acc + p;
    }
    return acc;
}

/*
 * sfar_oracle_gemv: for every rank r, y[r][j] = the definition above for
 * x[r] (k bf16), W[r] (k x h bf16, row-major), j < h.  Host memory owned by
 * the caller.  Returns 0, or -1 for a bad argument.
 */
int sfar_oracle_gemv(int R, size_t k, size_t h, const void *const *x, const void *const *W, void *const *y)
{
    if (R < 1 || R > 64 || k == 0 || h == 0 || !x || !W || !y)
        return -1;
    for (int r = 0; r < R; ++r) {
        if (!x[r] || !W[r] || !y[r])
            return -1;
        for (size_t j = 0; j < h; ++j)
            ((uint16_t *)y[r])[j] =
                narrow_bf16(gemv_column((const uint16_t *)x[r], (const uint16_t *)W[r], k, h, j));
    }
    return 0;
}

/* The two conversions on their own, so that tests can pin them directly. */
uint16_t sfar_oracle_narrow_bf16(float f) { return narrow_bf16(f); }

/* The same conversion over an array: out[i] = bf16 bits of in[i], i < n. */
void sfar_oracle_narrow_bf16_n(const float *in, uint16_t *out, size_t n)
{
    for (size_t i = 0; i < n; ++i)
        out[i] = narrow_bf16(in[i]);
}
float sfar_oracle_widen_bf16(uint16_t b) { return widen_bf16(b); }
int sfar_oracle_mutant(void) { return ORACLE_MUTANT; }
