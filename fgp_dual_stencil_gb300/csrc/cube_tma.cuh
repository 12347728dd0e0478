// CUBE_TMA variant of the FGP step: the page's cube-tiled kernel ("TV
// solver: the FGP step on the GPU", section "Variants", the 16 x 8 x 4 tile
// row), rebuilt around the tensor memory accelerator.
//
// A CTA owns a 16 x 8 x 4 tile of voxels.  One thread issues three-
// dimensional TMA copies of b on the tile and its upper halo (z is needed at
// the tile and at x+1, y+1, z+1) and of the three components of r on the
// tile grown by one voxel below and one above (z at a voxel reads r there
// and at its lower neighbours); meanwhile every thread loads its own p.
// After one bounded wait on the copies the CTA computes z once for every
// voxel of the grown tile (17 x 9 x 5, in quads and one scalar column) into
// shared memory, then each thread updates the dual of its quad of four x
// voxels with the same arithmetic as every other kernel.  Coordinates
// outside the volume read as zero, which is the r_a(-1) = 0 boundary.
//
// Unlike the z-march there is no pipeline across planes: a CTA loads,
// waits, computes and exits, and the latency of its copies is hidden only by
// the other CTAs resident on the SM.  That is the design the page compared,
// kept here for the same comparison.
#pragma once

#include "zmarch_tma.cuh"

namespace tvfgp {

constexpr int CB_TX = 16, CB_TY = 8, CB_TZ = 4;             // tile
constexpr int CB_THREADS = (CB_TX / 4) * CB_TY * CB_TZ;     // one thread per quad
// b box: x0..x0+19 (x0..x0+16 needed), y0..y0+8, z0..z0+4
constexpr int CB_BX = CB_TX + 4, CB_BY = CB_TY + 1, CB_BZ = CB_TZ + 1;
// r boxes: x0-4..x0+19 (x0-1..x0+16 needed), y0-1..y0+8, z0-1..z0+4
constexpr int CB_RX = CB_TX + 8, CB_RY = CB_TY + 2, CB_RZ = CB_TZ + 2;
// z of the grown tile x0..x0+16, y0..y0+8, z0..z0+4, row pitch CB_BX
constexpr int CB_ZX = CB_TX + 1;
constexpr int CB_BYTES_B = CB_BX * CB_BY * CB_BZ * 4;
constexpr int CB_BYTES_R = CB_RX * CB_RY * CB_RZ * 4;
constexpr int CB_OFF_B = 0;
constexpr int CB_OFF_R0 = zm_round128(CB_OFF_B + CB_BYTES_B);
constexpr int CB_OFF_R1 = zm_round128(CB_OFF_R0 + CB_BYTES_R);
constexpr int CB_OFF_R2 = zm_round128(CB_OFF_R1 + CB_BYTES_R);
constexpr int CB_OFF_Z = zm_round128(CB_OFF_R2 + CB_BYTES_R);
constexpr int CB_OFF_BAR = zm_round128(CB_OFF_Z + CB_BYTES_B);
constexpr int CB_OFF_FLAG = CB_OFF_BAR + 8;
constexpr int CB_SMEM = CB_OFF_FLAG + 16 + 128;              // + base alignment
constexpr int CB_TX_BYTES = CB_BYTES_B + 3 * CB_BYTES_R;
constexpr int CB_ZROWS = CB_BY * CB_BZ;                      // rows of the grown tile
constexpr int CB_ZTASKS = CB_ZROWS * (CB_TX / 4 + 1);        // 4 quads and 1 scalar per row

static_assert(CB_TX % 4 == 0 && CB_RX <= 256 && CB_BX <= 256, "TMA box limits");
static_assert((CB_BX * 4) % 16 == 0 && (CB_RX * 4) % 16 == 0, "TMA box rows are whole 16-byte units");

struct CubeArgs {
    CUtensorMap tb, t0, t1, t2;   // b, and r0, r1, r2 of the r read by this step
    StepArgs a;
    int *err;
    int max_polls;                // bound of the wait for data (the drain keeps ZM_MAX_POLLS), ...
    int poll_from;                // ... if poll_from <= 0 (a CTA waits once, for its only tile)
};

__global__ void __launch_bounds__(CB_THREADS) fgp_step_cube_tma(const __grid_constant__ CubeArgs ca)
{
    extern __shared__ unsigned char cb_raw[];
    unsigned char *smem = cb_raw + ((128 - (smem_addr(cb_raw) & 127)) & 127);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + CB_OFF_BAR);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + CB_OFF_FLAG);
    const float *Bs = reinterpret_cast<const float *>(smem + CB_OFF_B);
    const float *R0s = reinterpret_cast<const float *>(smem + CB_OFF_R0);
    const float *R1s = reinterpret_cast<const float *>(smem + CB_OFF_R1);
    const float *R2s = reinterpret_cast<const float *>(smem + CB_OFF_R2);
    float *Zs = reinterpret_cast<float *>(smem + CB_OFF_Z);

    const StepArgs &a = ca.a;
    const int nx = a.nx, ny = a.ny, nz = a.nz;
    const int tid = threadIdx.x;
    const int x0 = blockIdx.x * CB_TX, y0 = blockIdx.y * CB_TY, z0 = blockIdx.z * CB_TZ;

    if (tid == 0) {
        mbar_init(bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_expect_tx(bar, CB_TX_BYTES);
        tma_load_3d(smem + CB_OFF_B, &ca.tb, x0, y0, z0, bar);
        tma_load_3d(smem + CB_OFF_R0, &ca.t0, x0 - 4, y0 - 1, z0 - 1, bar);
        tma_load_3d(smem + CB_OFF_R1, &ca.t1, x0 - 4, y0 - 1, z0 - 1, bar);
        tma_load_3d(smem + CB_OFF_R2, &ca.t2, x0 - 4, y0 - 1, z0 - 1, bar);
    }

    // this thread's quad, and its own p, loaded before any wait
    const int qx = tid % (CB_TX / 4), ly = (tid / (CB_TX / 4)) % CB_TY, lz = tid / (CB_TX / 4 * CB_TY);
    const int lx = 4 * qx;
    const int x = x0 + lx, y = y0 + ly, z = z0 + lz;
    const bool inside = x < nx && y < ny && z < nz;
    const long long i = x + (long long)nx * (y + (long long)ny * z);
    float4 P0 = f4zero(), P1 = f4zero(), P2 = f4zero();
    if (inside) {
        P0 = ld_once4(a.p + i);
        P1 = ld_once4(a.p + a.N + i);
        P2 = ld_once4(a.p + 2 * a.N + i);
    }
    __syncthreads();                                  // the barrier is initialised
    if (!mbar_wait_tma(bar, 0, ca.poll_from <= 0 ? ca.max_polls : ZM_MAX_POLLS)) *abort_flag = 1;
    __syncthreads();
    if (*abort_flag) {
        if (tid == 0) {
            atomicExch(ca.err, kErrTimeout);
            mbar_wait_tma(bar, 0);                    // drain the copies (bounded)
        }
        return;
    }

    // z once per voxel of the grown tile: per row (ly', lz') 4 quads and the
    // scalar column x0+16
    for (int t = tid; t < CB_ZTASKS; t += CB_THREADS) {
        const int row = t / (CB_TX / 4 + 1), k = t % (CB_TX / 4 + 1);
        const int zy = row % CB_BY, zz = row / CB_BY;
        const int bo = row * CB_BX;                           // b and z row
        const int ro = ((zz + 1) * CB_RY + (zy + 1)) * CB_RX + 4;   // r at x0
        if (k < CB_TX / 4) {
            const int c = 4 * k;
            const float4 Z = zquad(lds4(Bs + bo + c), lds4(R0s + ro + c), lds4(R1s + ro + c), lds4(R2s + ro + c),
                                   R0s[ro + c - 1], lds4(R1s + ro + c - CB_RX), lds4(R2s + ro + c - CB_RX * CB_RY),
                                   a.lam, neg_zero(a.lam));
            *reinterpret_cast<float4 *>(Zs + bo + c) = Z;
        } else {
            const int c = CB_TX;
            Zs[bo + c] = zval(Bs[bo + c], a.lam, __fsub_rn(R0s[ro + c], R0s[ro + c - 1]),
                              __fsub_rn(R1s[ro + c], R1s[ro + c - CB_RX]),
                              __fsub_rn(R2s[ro + c], R2s[ro + c - CB_RX * CB_RY]));
        }
    }
    __syncthreads();
    if (!inside) return;

    // dual update of this thread's quad
    const int zo = (lz * CB_BY + ly) * CB_BX + lx;
    const int ro = ((lz + 1) * CB_RY + (ly + 1)) * CB_RX + 4 + lx;
    const float4 zc = lds4(Zs + zo);
    const float zx = Zs[zo + 4];
    const float4 zy = lds4(Zs + zo + CB_BX);
    const float4 zz = lds4(Zs + zo + CB_BX * CB_BY);
    const bool gy = y < ny - 1, gz = z < nz - 1;
    float4 G0, G1 = f4zero(), G2 = f4zero();
    G0.x = __fsub_rn(zc.x, zc.y);
    G0.y = __fsub_rn(zc.y, zc.z);
    G0.z = __fsub_rn(zc.z, zc.w);
    G0.w = (x + 3 < nx - 1) ? __fsub_rn(zc.w, zx) : 0.0f;
    if (gy) {
        G1.x = __fsub_rn(zc.x, zy.x); G1.y = __fsub_rn(zc.y, zy.y);
        G1.z = __fsub_rn(zc.z, zy.z); G1.w = __fsub_rn(zc.w, zy.w);
    }
    if (gz) {
        G2.x = __fsub_rn(zc.x, zz.x); G2.y = __fsub_rn(zc.y, zz.y);
        G2.z = __fsub_rn(zc.z, zz.z); G2.w = __fsub_rn(zc.w, zz.w);
    }
    float4 R0 = lds4(R0s + ro), R1 = lds4(R1s + ro), R2 = lds4(R2s + ro);
    dual_update4(R0, R1, R2, G0, G1, G2, P0, P1, P2, a.s, a.m, neg_zero(a.lam));
    st4(a.p + i, P0);
    st4(a.p + a.N + i, P1);
    st4(a.p + 2 * a.N + i, P2);
    st4(a.rd + i, R0);
    st4(a.rd + a.N + i, R1);
    st4(a.rd + 2 * a.N + i, R2);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

inline bool cube_encode(CUtensorMap *map, const float *base, int nx, int ny, int nz, int bx, int by, int bz)
{
    const cuuint64_t dims[3] = {(cuuint64_t)nx, (cuuint64_t)ny, (cuuint64_t)nz};
    const cuuint64_t strides[2] = {(cuuint64_t)nx * 4, (cuuint64_t)nx * ny * 4};
    const cuuint32_t box[3] = {(cuuint32_t)bx, (cuuint32_t)by, (cuuint32_t)bz};
    const cuuint32_t estr[3] = {1, 1, 1};
    return zm_encoder()(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, TVFGP_ZM_L2PROMO,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline const void *cube_kernel() { return reinterpret_cast<const void *>(&fgp_step_cube_tma); }
inline int cube_threads() { return CB_THREADS; }
inline size_t cube_smem_bytes() { return CB_SMEM; }
inline dim3 cube_grid(int nx, int ny, int nz)
{
    return dim3((nx + CB_TX - 1) / CB_TX, (ny + CB_TY - 1) / CB_TY, (nz + CB_TZ - 1) / CB_TZ);
}

// Kernel arguments of one step (tensor maps of b and of r_src's components).
inline bool cube_fill(const StepArgs &a, int *err, CubeArgs &ca)
{
    ca.a = a;
    ca.err = err;
    ca.max_polls = ZM_MAX_POLLS;
    ca.poll_from = 0;
    const float *r = a.rs;
    return cube_encode(&ca.tb, a.b, a.nx, a.ny, a.nz, CB_BX, CB_BY, CB_BZ) &&
           cube_encode(&ca.t0, r, a.nx, a.ny, a.nz, CB_RX, CB_RY, CB_RZ) &&
           cube_encode(&ca.t1, r + a.N, a.nx, a.ny, a.nz, CB_RX, CB_RY, CB_RZ) &&
           cube_encode(&ca.t2, r + 2 * a.N, a.nx, a.ny, a.nz, CB_RX, CB_RY, CB_RZ);
}

}  // namespace tvfgp
