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
