/*
 * Body of the CPU oracle, written once and compiled twice by
 * tvfgp_oracle.c: once with REAL = float (suffix _f32) and once with
 * REAL = double (suffix _f64).  TEST INFRASTRUCTURE ONLY: see the header of
 * tvfgp_oracle.c.
 *
 * Everything here follows the page "TV solver: the FGP step on the GPU",
 * section "What one step does":
 *
 *   z(j)  = max(b(j) - lambda * L(r)(j), 0)
 *   L(r)(j) = sum_a r_a(j) - r_a(j - e_a)
 *   g_a   = z(i) - z(i + e_a)
 *   q     = r(i) + g / (12 lambda)
 *   p'    = q / max(1, |q|)
 *   r(i)  = p' + m (p' - p(i));   p(i) = p'
 *
 * with the two boundary rules of the problem statement: r_a(-1) = 0 below
 * the lower face of axis a, and g_a = 0 where i + e_a leaves the volume.
 *
 * Layout: x fastest, voxel (x, y, z) at i = x + nx*(y + ny*z).  A dual field
 * is planar: component a (0 = x, 1 = y, 2 = z) of voxel i at a*N + i.
 * Each operation is rounded on its own, in the order written (no FMA
 * contraction; the build passes -ffp-contract=off).
 */

#define CAT2_(a, b) a##b
#define CAT2(a, b) CAT2_(a, b)
#define FN(name) CAT2(name, SUFFIX)

/* L(r)(j) for one voxel; the lower-face terms r_a(j - e_a) are 0. */
static REAL FN(adjoint_at)(const REAL *r0, const REAL *r1, const REAL *r2,
                           int x, int y, int z, int nx, int ny)
{
    size_t j = vox(x, y, z, nx, ny);
    size_t sx = 1, sy = (size_t)nx, sz = (size_t)nx * (size_t)ny;
    REAL d0 = r0[j] - (x > 0 ? r0[j - sx] : (REAL)0);
    REAL d1 = r1[j] - (y > 0 ? r1[j - sy] : (REAL)0);
    REAL d2 = r2[j] - (z > 0 ? r2[j - sz] : (REAL)0);
    return (d0 + d1) + d2;
}

/* out(j) = L(dual)(j) over the whole volume (step a1, on its own). */
void FN(oracle_adjoint)(int nx, int ny, int nz, const REAL *dual, REAL *out)
{
    size_t N = (size_t)nx * ny * nz;
    const REAL *r0 = dual, *r1 = dual + N, *r2 = dual + 2 * N;
    int z;
#pragma omp parallel for schedule(static)
    for (z = 0; z < nz; ++z)
        for (int y = 0; y < ny; ++y)
            for (int x = 0; x < nx; ++x)
                out[vox(x, y, z, nx, ny)] = FN(adjoint_at)(r0, r1, r2, x, y, z, nx, ny);
}

/* g_a(i) = z(i) - z(i + e_a), and 0 where i + e_a leaves the volume
 * (step a3, on its own).  g is planar [3][N]. */
void FN(oracle_gradient)(int nx, int ny, int nz, const REAL *zv, REAL *g)
{
    size_t N = (size_t)nx * ny * nz;
    size_t sy = (size_t)nx, sz = (size_t)nx * (size_t)ny;
    int z;
#pragma omp parallel for schedule(static)
    for (z = 0; z < nz; ++z)
        for (int y = 0; y < ny; ++y)
            for (int x = 0; x < nx; ++x) {
                size_t i = vox(x, y, z, nx, ny);
                g[i] = (x < nx - 1) ? zv[i] - zv[i + 1] : (REAL)0;
                g[N + i] = (y < ny - 1) ? zv[i] - zv[i + sy] : (REAL)0;
                g[2 * N + i] = (z < nz - 1) ? zv[i] - zv[i + sz] : (REAL)0;
            }
}

/* z = max(b - lambda * L(dual), 0) over the volume (steps a1 + a2, and the
 * stand-alone primal output a8). */
void FN(oracle_primal)(int nx, int ny, int nz, const REAL *b, const REAL *dual,
                       REAL lambda, REAL *zout)
{
    size_t N = (size_t)nx * ny * nz;
    const REAL *r0 = dual, *r1 = dual + N, *r2 = dual + 2 * N;
    int z;
#pragma omp parallel for schedule(static)
    for (z = 0; z < nz; ++z)
        for (int y = 0; y < ny; ++y)
            for (int x = 0; x < nx; ++x) {
                size_t j = vox(x, y, z, nx, ny);
                REAL L = FN(adjoint_at)(r0, r1, r2, x, y, z, nx, ny);
                REAL w = b[j] - lambda * L;
                zout[j] = MAXR(w, (REAL)0);
            }
}

/* One FGP step.  Reads b, p, r_src; writes p (in place), r_dst and the work
 * volume zw (N values, the primal z of r_src).  m is the momentum weight of
 * this step.  Steps a1..a5 in the page's order: first z for every voxel,
 * then the gradient, the dual step with its projection onto the unit ball,
 * and the extrapolation. */
void FN(oracle_fgp_step)(int nx, int ny, int nz, const REAL *b, REAL *p,
                         const REAL *r_src, REAL *r_dst, REAL *zw,
                         REAL lambda, REAL m)
{
    size_t N = (size_t)nx * ny * nz;
    size_t sy = (size_t)nx, sz = (size_t)nx * (size_t)ny;
    REAL s = STEP_OF(lambda);
    int z;

    FN(oracle_primal)(nx, ny, nz, b, r_src, lambda, zw);

#pragma omp parallel for schedule(static)
    for (z = 0; z < nz; ++z)
        for (int y = 0; y < ny; ++y)
            for (int x = 0; x < nx; ++x) {
                size_t i = vox(x, y, z, nx, ny);
                REAL g0 = (x < nx - 1) ? zw[i] - zw[i + 1] : (REAL)0;
                REAL g1 = (y < ny - 1) ? zw[i] - zw[i + sy] : (REAL)0;
                REAL g2 = (z < nz - 1) ? zw[i] - zw[i + sz] : (REAL)0;
                REAL q0 = r_src[i] + g0 * s;
                REAL q1 = r_src[N + i] + g1 * s;
                REAL q2 = r_src[2 * N + i] + g2 * s;
                REAL nrm = SQRTR((q0 * q0 + q1 * q1) + q2 * q2);
                REAL d = MAXR((REAL)1, nrm);
                REAL pp0 = q0 / d, pp1 = q1 / d, pp2 = q2 / d;
                r_dst[i] = pp0 + m * (pp0 - p[i]);
                r_dst[N + i] = pp1 + m * (pp1 - p[N + i]);
                r_dst[2 * N + i] = pp2 + m * (pp2 - p[2 * N + i]);
                p[i] = pp0;
                p[N + i] = pp1;
                p[2 * N + i] = pp2;
            }
}

/* nsteps FGP steps from (p, r) with the momentum schedule started at t0.
 * p and r are updated in place; the final r ends in r.  *t_final (if not
 * NULL) receives t after the last step.  Returns 0, or -1 when the work
 * buffers cannot be allocated. */
int FN(oracle_fgp_run)(int nx, int ny, int nz, const REAL *b, REAL *p, REAL *r,
                       REAL lambda, int nsteps, double t0, double *t_final)
{
    size_t N = (size_t)nx * ny * nz;
    double *m = NULL;
    REAL *other = NULL, *zw = NULL;
    if (nsteps <= 0) {
        if (t_final) *t_final = t0;
        return 0;
    }
    m = (double *)malloc(sizeof(double) * (size_t)nsteps);
    other = (REAL *)malloc(sizeof(REAL) * 3 * N);
    zw = (REAL *)malloc(sizeof(REAL) * N);
    if (!m || !other || !zw) {
        free(m); free(other); free(zw);
        return -1;
    }
    oracle_momentum(t0, nsteps, m, t_final);
    REAL *src = r, *dst = other;
    for (int k = 0; k < nsteps; ++k) {
        FN(oracle_fgp_step)(nx, ny, nz, b, p, src, dst, zw, lambda, (REAL)m[k]);
        REAL *t = src; src = dst; dst = t;
    }
    if (src != r) memcpy(r, src, sizeof(REAL) * 3 * N);
    free(m); free(other); free(zw);
    return 0;
}

#undef FN
#undef CAT2
#undef CAT2_
