/*
 * gsi_oracle.c -- fp64 CPU oracle for the Gated Subspace Inference (GSI)
 * linear map.  TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
 * load this library.  The product path (the CUDA library and its Python
 * binding) never loads, links or calls it, and this file shares no code,
 * header, table or constant with the CUDA path.
 *
 * Citations "[GSI ...]" refer to the page "Technical summary: Gated Subspace
 * Inference for transformer acceleration" (Korean and Japanese editions of
 * the same summary carry the same sections and numbers).
 *
 * What the map computes, per token x in R^d, given W (d_out x d), an
 * orthonormal rank-k basis V_k (d x k), the cached image M = W V_k and a
 * threshold eps:
 *   g   = V_k^T x                      [GSI 2.1, definition under eq. 2]
 *   r   = x - V_k g                    [GSI 2.1, eq. 1 solved for r]
 *   rho = ||r|| / ||x||                [GSI 2.2, fast-path bullet]
 *   y   = M g  if rho <  eps           [GSI 2.2, fast-path bullet]
 *   y   = W x  if rho >= eps           [GSI 2.2, slow-path bullet]
 *
 * Readings taken where the page is silent (each also listed in the design doc):
 *   - ||.|| is the Euclidean 2-norm of a vector.
 *   - ||x|| = 0 gives rho = 0 (fast path; y = M 0 = 0 = W 0 either way).
 *   - A non-finite ||x|| (NaN or Inf anywhere in x) gives rho = NaN, and
 *     "rho < eps" is then false, so the token takes the slow path.
 *   - A tie rho == eps takes the slow path (the page's ">=" bullet).
 *   - The caller passes eps as the fp64 value of the fp32 threshold that the
 *     GPU receives, so both sides compare against the same number.
 *
 * Everything is plain fp64 with loops in the page's order.  No blocking, no
 * fusion, no reordering: g is formed completely before r, r before rho, and
 * rho before y.  OpenMP only splits independent tokens / output rows.
 *
 * Build (done by __graft_entry__.build() and by the test fixtures):
 *   gcc -O2 -std=c11 -ffp-contract=off -fopenmp -shared -fPIC \
 *       oracle/gsi_oracle.c -o oracle/libgsi_oracle.so -lm
 * -ffp-contract=off keeps a*b+c as two rounded operations on every host, so
 * the oracle gives the same bits on x86-64 and on aarch64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------------- */
/* bf16 storage format (1 sign, 8 exponent, 7 fraction bits).             */
/* ---------------------------------------------------------------------- */

/* Exact decode: a bf16 value is the top half of an IEEE binary32. */
static double bf16_decode(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round an fp64 value to the nearest bf16, ties to even, in one rounding
 * (no detour through fp32, which could round twice).  A finite bf16 has at
 * most 8 significant bits; its quantum at binary exponent e (v = m 2^e,
 * 0.5 <= |m| < 1) is 2^(e-8), and never below the subnormal quantum 2^-133.
 * rint() rounds to nearest-even under the default rounding mode. */
static uint16_t bf16_encode(double v)
{
    if (isnan(v))
        return (uint16_t)(signbit(v) ? 0xFFC0u : 0x7FC0u);
    if (v == 0.0 || isinf(v)) {
        float f = (float)v;
        uint32_t u;
        memcpy(&u, &f, sizeof u);
        return (uint16_t)(u >> 16);
    }
    int e;
    (void)frexp(v, &e);
    int q = e - 8;
    if (q < -133)
        q = -133;
    double r = ldexp(rint(ldexp(v, -q)), q);
    const double bf16_max = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
    if (fabs(r) > bf16_max)
        r = copysign(INFINITY, v);
    float f = (float)r; /* exact: r has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

void gsi_oracle_bf16_decode(const uint16_t *in, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = bf16_decode(in[i]);
}

void gsi_oracle_bf16_encode(const double *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = bf16_encode(in[i]);
}

/* ---------------------------------------------------------------------- */
/* The cached low-rank weight image M = W V_k          [GSI 2.1, eq. 2]   */
/* ---------------------------------------------------------------------- */

/* M (d_out x k, row-major) = W (d_out x d) times V (d x k), exact fp64 sums. */
void gsi_oracle_precompute_M(const double *W, const double *V, int64_t d_out,
                             int64_t d, int64_t k, double *M)
{
#pragma omp parallel for schedule(static)
    for (int64_t o = 0; o < d_out; ++o) {
        for (int64_t j = 0; j < k; ++j) {
            double s = 0.0;
            for (int64_t i = 0; i < d; ++i)
                s += W[o * d + i] * V[i * k + j];
            M[o * k + j] = s;
        }
    }
}

/* ---------------------------------------------------------------------- */
/* The gated map, token by token                       [GSI 2.1 - 2.2]    */
/* ---------------------------------------------------------------------- */

/* Projection and residual ratio of one token.
 *   g = V^T x            (k values)            [GSI 2.1, under eq. 2]
 *   r = x - V g          (d values)            [GSI 2.1, eq. 1]
 *   rho = ||r|| / ||x||                        [GSI 2.2]
 * r_out may be NULL. */
static double token_projection(const double *V, int64_t d, int64_t k,
                               const double *x, double *g, double *r_out)
{
    for (int64_t j = 0; j < k; ++j) {
        double s = 0.0;
        for (int64_t i = 0; i < d; ++i)
            s += V[i * k + j] * x[i];
        g[j] = s;
    }
    double xx = 0.0, rr = 0.0;
    for (int64_t i = 0; i < d; ++i) {
        double vg = 0.0;
        for (int64_t j = 0; j < k; ++j)
            vg += V[i * k + j] * g[j];
        double ri = x[i] - vg;
        if (r_out)
            r_out[i] = ri;
        xx += x[i] * x[i];
        rr += ri * ri;
    }
    double nx = sqrt(xx);
    double nr = sqrt(rr);
    if (!isfinite(nx))
        return NAN;
    if (nx == 0.0)
        return 0.0;
    return nr / nx;
}

/* The gated linear map over T tokens (rows of X, T x d, row-major).
 *   rho[t]  = residual ratio of token t
 *   gate[t] = 1 if token t takes the slow path (rho >= eps or rho is NaN),
 *             0 if it takes the fast path (rho < eps)
 *   Y[t]    = M g_t on the fast path, W x_t on the slow path (d_out values)
 * G (T x k) and R (T x d) are optional outputs (NULL to skip) holding g_t and
 * r_t.  Returns 0, or -1 on a bad argument. */
int gsi_oracle_forward(const double *W, const double *V, const double *M,
                       int64_t d_out, int64_t d, int64_t k, double eps,
                       const double *X, int64_t T, double *Y, double *rho,
                       uint8_t *gate, double *G, double *R)
{
    if (d_out < 0 || d <= 0 || k <= 0 || T < 0 || !V || !Y || !rho || !gate)
        return -1;
    if (T == 0)
        return 0;
    double *gbuf = (double *)malloc((size_t)(T * k) * sizeof(double));
    if (!gbuf)
        return -1;

    /* Gate of every token first: it depends on x, V and eps only. */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
        double *g = gbuf + t * k;
        double *r = R ? R + t * d : NULL;
        double p = token_projection(V, d, k, X + t * d, g, r);
        rho[t] = p;
        gate[t] = (p < eps) ? 0 : 1;
    }

    /* Then the branch the gate picked [GSI 2.2]. */
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t o = 0; o < d_out; ++o) {
            double s = 0.0;
            if (gate[t]) {              /* slow path: y = W x */
                const double *x = X + t * d;
                for (int64_t i = 0; i < d; ++i)
                    s += W[o * d + i] * x[i];
            } else {                    /* fast path: y = M g */
                const double *g = gbuf + t * k;
                for (int64_t j = 0; j < k; ++j)
                    s += M[o * k + j] * g[j];
            }
            Y[t * d_out + o] = s;
        }
    }
    if (G)
        memcpy(G, gbuf, (size_t)(T * k) * sizeof(double));
    free(gbuf);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Spectral norm by power iteration                    [GSI 2.2, Thm 4]   */
/* ---------------------------------------------------------------------- */

/* Largest singular value of A (m x n, row-major) by power iteration on
 * A^T A, from a seeded start vector (splitmix64 -> uniform(-1, 1)).  Stops
 * when the estimate changes by less than tol (relative) or after max_iter
 * steps.  The estimate ||A v|| with ||v|| = 1 never exceeds the true value;
 * a caller that needs an upper bound adds a margin.  Returns -1 on error. */
double gsi_oracle_spectral_norm(const double *A, int64_t m, int64_t n,
                                uint64_t seed, int max_iter, double tol)
{
    if (m <= 0 || n <= 0 || !A)
        return -1.0;
    double *v = (double *)malloc((size_t)n * sizeof(double));
    double *w = (double *)malloc((size_t)m * sizeof(double));
    if (!v || !w) {
        free(v);
        free(w);
        return -1.0;
    }
    uint64_t s = seed;
    for (int64_t i = 0; i < n; ++i) {
        s += 0x9E3779B97F4A7C15ull;
        uint64_t z = s;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
        z ^= z >> 31;
        v[i] = 2.0 * ((double)(z >> 11) / 9007199254740992.0) - 1.0;
    }
    double sigma = 0.0;
    for (int it = 0; it < max_iter; ++it) {
        double vv = 0.0;
        for (int64_t i = 0; i < n; ++i)
            vv += v[i] * v[i];
        double nv = sqrt(vv);
        if (nv == 0.0)
            break;
        for (int64_t i = 0; i < n; ++i)
            v[i] /= nv;
#pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < m; ++r) {
            double a = 0.0;
            for (int64_t c = 0; c < n; ++c)
                a += A[r * n + c] * v[c];
            w[r] = a;
        }
        double ww = 0.0;
        for (int64_t r = 0; r < m; ++r)
            ww += w[r] * w[r];
        double est = sqrt(ww);
        /* v <- A^T w */
#pragma omp parallel for schedule(static)
        for (int64_t c = 0; c < n; ++c) {
            double a = 0.0;
            for (int64_t r = 0; r < m; ++r)
                a += A[r * n + c] * w[r];
            v[c] = a;
        }
        int done = (it > 0 && fabs(est - sigma) <= tol * est);
        sigma = est;
        if (done)
            break;
    }
    free(v);
    free(w);
    return sigma;
}

/* Number of OpenMP threads the oracle runs with (1 without OpenMP). */
int gsi_oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
