/*
 * A plain C consumer of the tvfgp C ABI: no C++, no Python, no framework;
 * only the CUDA runtime for device memory.  Reads b from a file, runs nsteps
 * FGP steps from p = r = 0 with t0 = 1, takes the primal of p, and writes
 * p, r and z (raw fp32) and t after the last step.  Used by
 * tests/test_gpu_c_consumer.py.
 *
 *   c_abi_consumer B_FILE OUT_FILE NX NY NZ LAMBDA NSTEPS VARIANT
 */
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "tvfgp.h"

static int fail(const char *what, int code)
{
    fprintf(stderr, "%s failed: %d\n", what, code);
    return 1;
}

int main(int argc, char **argv)
{
    if (argc != 9) {
        fprintf(stderr, "usage: %s B_FILE OUT_FILE NX NY NZ LAMBDA NSTEPS VARIANT\n", argv[0]);
        return 2;
    }
    const int nx = atoi(argv[3]), ny = atoi(argv[4]), nz = atoi(argv[5]);
    const float lambda = (float)atof(argv[6]);
    const int nsteps = atoi(argv[7]), variant = atoi(argv[8]);
    const size_t n = (size_t)nx * ny * nz;
    float *hb = malloc(sizeof(float) * n), *hout = malloc(sizeof(float) * 7 * n);
    if (!hb || !hout) return fail("malloc", 0);
    FILE *f = fopen(argv[1], "rb");
    if (!f || fread(hb, sizeof(float), n, f) != n) return fail("reading b", 0);
    fclose(f);

    float *b, *p, *r, *z;
    if (cudaMalloc((void **)&b, sizeof(float) * n) || cudaMalloc((void **)&p, sizeof(float) * 3 * n) ||
        cudaMalloc((void **)&r, sizeof(float) * 3 * n) || cudaMalloc((void **)&z, sizeof(float) * n))
        return fail("cudaMalloc", 0);
    if (cudaMemcpy(b, hb, sizeof(float) * n, cudaMemcpyHostToDevice) ||
        cudaMemset(p, 0, sizeof(float) * 3 * n) || cudaMemset(r, 0, sizeof(float) * 3 * n))
        return fail("cudaMemcpy/cudaMemset", 0);

    tvfgp_t h = NULL;
    int rc = tvfgp_create_ex(nx, ny, nz, variant, 0u, &h);
    if (rc != TVFGP_OK) return fail(tvfgp_strerror(rc), rc);
    double t_final = 0.0;
    rc = tvfgp_run(h, b, p, r, lambda, nsteps, 1.0, NULL, &t_final);
    if (rc == TVFGP_OK) rc = tvfgp_primal(h, b, p, lambda, z, NULL);
    if (rc == TVFGP_OK) rc = tvfgp_check(h, NULL);
    if (rc != TVFGP_OK) return fail(tvfgp_strerror(rc), rc);
    const int ran = tvfgp_last_variant(h);
    tvfgp_destroy(h);

    if (cudaMemcpy(hout, p, sizeof(float) * 3 * n, cudaMemcpyDeviceToHost) ||
        cudaMemcpy(hout + 3 * n, r, sizeof(float) * 3 * n, cudaMemcpyDeviceToHost) ||
        cudaMemcpy(hout + 6 * n, z, sizeof(float) * n, cudaMemcpyDeviceToHost))
        return fail("cudaMemcpy back", 0);
    f = fopen(argv[2], "wb");
    if (!f || fwrite(hout, sizeof(float), 7 * n, f) != 7 * n) return fail("writing the output", 0);
    fclose(f);
    printf("%.17g %d\n", t_final, ran);
    cudaFree(b);
    cudaFree(p);
    cudaFree(r);
    cudaFree(z);
    free(hb);
    free(hout);
    return 0;
}
