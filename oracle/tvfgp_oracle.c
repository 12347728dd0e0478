/*
 * CPU oracle for the FGP step on the 3D isotropic TV dual.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow reference that the
 * GPU path is checked against.  Only the tests, the smoke check and the
 * bench's CPU-baseline / reference arm may load it; the library in
 * fgp_dual_stencil_gb300/ never includes, links or calls it, and it includes
 * nothing from there.
 *
 * What it computes (page "TV solver: the FGP step on the GPU", section
 * "What one step does"): Beck and Teboulle's fast gradient projection on the
 * dual of  min_{x >= 0} |x - b|^2 + 2 lambda TV(x)  in 3D, one step at a
 * time, in the order the page states it.  The momentum weights come from
 * the FISTA schedule  t_{k+1} = (1 + sqrt(1 + 4 t_k^2)) / 2,
 * m_k = (t_k - 1) / t_{k+1}  (the page names only m; the schedule is the
 * standard one of the FGP/FISTA method).
 *
 * Precision: the product computes in fp32, so the _f32 functions are the
 * parity oracle: each operation rounded to nearest in the written order,
 * no FMA contraction, IEEE division and square root.  The step 1/(12 lambda)
 * is evaluated in double and rounded once to float; the momentum weight m is
 * computed in double and rounded once to float per step.  The _f64 twins do
 * the same in double and serve the pins that need the exact mathematics.
 *
 * Pins (tests/test_oracle_pins.py): constant b keeps p = r = 0; adjoint
 * identity; |p| <= 1 and z >= 0; the two-voxel closed form on each axis;
 * exact power-of-two scaling; x<->y transposition equivariance; hand-derived
 * steps (tests/golden/hand_steps.txt); a matrix-form step built from the
 * definition of the forward difference; and agreement with a brute-force,
 * duality-gap-certified TV prox on tiny volumes.
 *
 * Parallelism: an optional OpenMP loop over z-planes.  Every voxel is
 * computed independently with no reduction, so results do not depend on the
 * thread count.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static inline size_t vox(int x, int y, int z, int nx, int ny)
{
    return (size_t)x + (size_t)nx * ((size_t)y + (size_t)ny * (size_t)z);
}

/* FISTA momentum schedule, in double. m[k] is the weight of step k. */
void oracle_momentum(double t0, int nsteps, double *m, double *t_final)
{
    double t = t0;
    for (int k = 0; k < nsteps; ++k) {
        double tn = (1.0 + sqrt(1.0 + 4.0 * t * t)) / 2.0;
        m[k] = (t - 1.0) / tn;
        t = tn;
    }
    if (t_final) *t_final = t;
}

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_get_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* fp32 instantiation */
#define REAL float
#define SUFFIX _f32
#define MAXR fmaxf
#define SQRTR sqrtf
#define STEP_OF(lam) ((float)(1.0 / (12.0 * (double)(lam))))
#include "tvfgp_oracle_body.h"
#undef REAL
#undef SUFFIX
#undef MAXR
#undef SQRTR
#undef STEP_OF

/* fp64 instantiation */
#define REAL double
#define SUFFIX _f64
#define MAXR fmax
#define SQRTR sqrt
#define STEP_OF(lam) (1.0 / (12.0 * (lam)))
#include "tvfgp_oracle_body.h"
#undef REAL
#undef SUFFIX
#undef MAXR
#undef SQRTR
#undef STEP_OF

/* ------------------------------------------------------------------------
 * Half-precision storage of the dual (page "TV solver: the FGP step on the
 * GPU", "Profiler counters", names a half-precision dual among the ways to
 * move fewer bytes, at the price of a different result).  p and r are stored as IEEE 754
 * binary16; every step loads them exactly into float, computes in the fp32
 * canonical order above, and rounds each stored value once to binary16,
 * round-to-nearest-even.  The conversions are written here from the
 * binary16 definition: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits; subnormals below 2^-14.
 * ------------------------------------------------------------------------ */

float oracle_half_to_float(unsigned short h)
{
    const int sign = (h >> 15) & 1, e = (h >> 10) & 0x1f, f = h & 0x3ff;
    float v;
    if (e == 0) v = ldexpf((float)f, -24);                       /* zero, subnormal */
    else if (e == 31) v = f ? NAN : INFINITY;
    else v = ldexpf((float)(1024 + f), e - 25);                  /* (1 + f/1024) 2^(e-15) */
    return sign ? -v : v;
}

unsigned short oracle_float_to_half(float x)
{
    if (isnan(x)) return 0x7e00;
    const unsigned short sign = signbit(x) ? 0x8000 : 0;
    const double a = fabs((double)x);
    if (a >= 65520.0) return sign | 0x7c00;      /* rounds past the largest finite, 65504 */
    if (a < 0x1p-14) {                            /* subnormal range: quantum 2^-24 */
        const double m = nearbyint(a * 0x1p24);  /* ties to even in the default mode */
        return sign | (unsigned short)m;          /* m == 1024 is the smallest normal */
    }
    int e;
    frexp(a, &e);                                 /* a = fr 2^e, fr in [0.5, 1) */
    e -= 1;                                       /* a in [2^e, 2^(e+1)) */
    double m = nearbyint(ldexp(a, 10 - e));      /* 1024 .. 2048 */
    if (m >= 2048.0) {
        m = 1024.0;
        e += 1;
    }
    if (e + 15 >= 31) return sign | 0x7c00;
    return sign | (unsigned short)((e + 15) << 10) | (unsigned short)((int)m - 1024);
}

void oracle_half_to_float_array(const unsigned short *h, float *f, size_t n)
{
    long long i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < (long long)n; ++i) f[i] = oracle_half_to_float(h[i]);
}

void oracle_float_to_half_array(const float *f, unsigned short *h, size_t n)
{
    long long i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < (long long)n; ++i) h[i] = oracle_float_to_half(f[i]);
}

/* z = max(b - lambda L(dual), 0) for a binary16 dual field. */
void oracle_primal_h16(int nx, int ny, int nz, const float *b, const unsigned short *dual,
                       float lambda, float *zout)
{
    size_t N = (size_t)nx * ny * nz;
    float *d = (float *)malloc(sizeof(float) * 3 * N);
    if (!d) return;
    oracle_half_to_float_array(dual, d, 3 * N);
    oracle_primal_f32(nx, ny, nz, b, d, lambda, zout);
    free(d);
}

/* One step with binary16 storage: the fp32 step on the exactly widened p and
 * r_src, then p and r_dst rounded to binary16. */
int oracle_fgp_step_h16(int nx, int ny, int nz, const float *b, unsigned short *p,
                        const unsigned short *r_src, unsigned short *r_dst, float lambda, float m)
{
    size_t N = (size_t)nx * ny * nz;
    float *pf = (float *)malloc(sizeof(float) * 3 * N);
    float *rs = (float *)malloc(sizeof(float) * 3 * N);
    float *rd = (float *)malloc(sizeof(float) * 3 * N);
    float *zw = (float *)malloc(sizeof(float) * N);
    if (!pf || !rs || !rd || !zw) {
        free(pf); free(rs); free(rd); free(zw);
        return -1;
    }
    oracle_half_to_float_array(p, pf, 3 * N);
    oracle_half_to_float_array(r_src, rs, 3 * N);
    oracle_fgp_step_f32(nx, ny, nz, b, pf, rs, rd, zw, lambda, m);
    oracle_float_to_half_array(pf, p, 3 * N);
    oracle_float_to_half_array(rd, r_dst, 3 * N);
    free(pf); free(rs); free(rd); free(zw);
    return 0;
}

/* nsteps steps with binary16 storage of p and r (updated in place). */
int oracle_fgp_run_h16(int nx, int ny, int nz, const float *b, unsigned short *p,
                       unsigned short *r, float lambda, int nsteps, double t0, double *t_final)
{
    size_t N = (size_t)nx * ny * nz;
    if (nsteps <= 0) {
        if (t_final) *t_final = t0;
        return 0;
    }
    double *m = (double *)malloc(sizeof(double) * (size_t)nsteps);
    unsigned short *other = (unsigned short *)malloc(sizeof(unsigned short) * 3 * N);
    if (!m || !other) {
        free(m); free(other);
        return -1;
    }
    oracle_momentum(t0, nsteps, m, t_final);
    unsigned short *src = r, *dst = other;
    int rc = 0;
    for (int k = 0; k < nsteps && rc == 0; ++k) {
        rc = oracle_fgp_step_h16(nx, ny, nz, b, p, src, dst, lambda, (float)m[k]);
        unsigned short *t = src; src = dst; dst = t;
    }
    if (rc == 0 && src != r) memcpy(r, src, sizeof(unsigned short) * 3 * N);
    free(m); free(other);
    return rc;
}
