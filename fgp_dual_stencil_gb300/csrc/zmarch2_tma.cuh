// ZMARCH2_TMA: two FGP steps per pass over HBM (temporal blocking of the
// z-march).
//
// The page ("TV solver: the FGP step on the GPU", "Profiler counters") ends
// at the compulsory 13 volumes per step: the only way to a cheaper step is to
// move fewer bytes.  Without changing the result, that means computing two
// steps from one read of (b, p^k, r^k) and one write of (p^{k+2}, r^{k+2}):
// 13 volumes per two steps.  The intermediate p^{k+1}, r^{k+1} never leave
// shared memory.
//
// A CTA owns the output tile x0..x0+TX-1, y0..y0+TY-1 and walks planes of z.
// Step k+1 at a voxel needs r^{k+1} at the voxel, at x-1, y-1, z-1, and (for
// z^{k+1} of its upper neighbours) at x+1, y+1, z+1.  So step k is evaluated
// on the tile grown by one voxel on every side in x and y (the ring E), one
// plane ahead of step k+1:
//
//   at iteration q:
//     A  z^k     of plane q+1 on x0-1..x0+TX+1, y0-1..y0+TY+1   (staged b, r^k)
//     B  step k  of plane q   on x0-1..x0+TX,   y0-1..y0+TY     (-> r^{k+1}, p^{k+1} in shared memory)
//     C  z^{k+1} of plane q   on x0..x0+TX,     y0..y0+TY       (b, r^{k+1})
//     D  step k+1 of plane q-1 on the tile                      (-> p^{k+2}, r^{k+2} in HBM)
//
// with a barrier after A, B and C.  Voxels of the ring that lie outside the
// volume get r^{k+1} = 0: that is the r(-1) = 0 boundary step k+1 sees.
// Every value is computed by the same expressions, in the same order, as in
// the one-step kernels, so the result is bitwise that of two single steps.
//
// Because neighbouring CTAs read p^k in their ring, p cannot be updated in
// place: the kernel reads (p_src, r_src) and writes (p_dst, r_dst).
//
// Every operand of a plane (b, r^k with a two-voxel halo, p^k on the ring)
// arrives by TMA (non-multicast) into a ring of shared-memory stages, planes
// ahead of use, with bounded mbarrier waits (timeout: error word set, copies
// drained, return).
#pragma once

#include "zmarch_tma.cuh"

namespace tvfgp {

#ifndef TVFGP_Z2_TX
#define TVFGP_Z2_TX 32
#endif
#ifndef TVFGP_Z2_TY
#define TVFGP_Z2_TY 16
#endif
#ifndef TVFGP_Z2_THREADS
#define TVFGP_Z2_THREADS 256
#endif
#ifndef TVFGP_Z2_STAGES
#define TVFGP_Z2_STAGES 3
#endif
#ifndef TVFGP_Z2_MINB
#define TVFGP_Z2_MINB 2
#endif

constexpr int Z2_TX = TVFGP_Z2_TX;          // output tile width
constexpr int Z2_TY = TVFGP_Z2_TY;          // output tile height
constexpr int Z2_THREADS = TVFGP_Z2_THREADS;
constexpr int Z2_STAGES = TVFGP_Z2_STAGES;

// staged boxes: all start at x0-4 (a 16-byte aligned column) and are TX+8 wide
constexpr int Z2_BW = Z2_TX + 8;
constexpr int Z2_HB = Z2_TY + 3;            // b:   y0-1 .. y0+TY+1
constexpr int Z2_HR = Z2_TY + 4;            // r^k: y0-2 .. y0+TY+1
constexpr int Z2_HP = Z2_TY + 2;            // p^k: y0-1 .. y0+TY
constexpr int Z2_BYTES_B = Z2_BW * Z2_HB * 4;
constexpr int Z2_BYTES_R = Z2_BW * Z2_HR * 4;
constexpr int Z2_BYTES_P = Z2_BW * Z2_HP * 4;
constexpr int Z2_OFF_B = 0;
constexpr int Z2_OFF_R0 = zm_round128(Z2_OFF_B + Z2_BYTES_B);
constexpr int Z2_OFF_R1 = Z2_OFF_R0 + zm_round128(Z2_BYTES_R);
constexpr int Z2_OFF_R2 = Z2_OFF_R1 + zm_round128(Z2_BYTES_R);
constexpr int Z2_OFF_P0 = Z2_OFF_R2 + zm_round128(Z2_BYTES_R);
constexpr int Z2_OFF_P1 = Z2_OFF_P0 + zm_round128(Z2_BYTES_P);
constexpr int Z2_OFF_P2 = Z2_OFF_P1 + zm_round128(Z2_BYTES_P);
constexpr int Z2_STAGE_STRIDE = Z2_OFF_P2 + zm_round128(Z2_BYTES_P);
constexpr int Z2_TX_BR = Z2_BYTES_B + 3 * Z2_BYTES_R;
constexpr int Z2_TX_ALL = Z2_TX_BR + 3 * Z2_BYTES_P;

// regions (local coordinates lx = x - x0, ly = y - y0)
constexpr int Z2_ZKW = Z2_TX + 3, Z2_ZKH = Z2_TY + 3;     // z^k:     lx -1..TX+1, ly -1..TY+1
constexpr int Z2_UKW = Z2_TX + 2, Z2_UKH = Z2_TY + 2;     // step k:  lx -1..TX,   ly -1..TY
constexpr int Z2_Z1W = Z2_TX + 1, Z2_Z1H = Z2_TY + 1;     // z^{k+1}: lx  0..TX,   ly  0..TY
constexpr int Z2_PITCH = Z2_TX + 4;                       // row pitch of the shared rings

// shared rings, two slots each (a plane is written two iterations after the
// slot was last read, with a barrier in between)
constexpr int Z2_RING_ZK = Z2_ZKH * Z2_PITCH;             // floats per slot
constexpr int Z2_RING_MR = 3 * Z2_UKH * Z2_PITCH;
constexpr int Z2_RING_MP = 3 * Z2_TY * Z2_TX;
constexpr int Z2_RING_Z1 = Z2_Z1H * Z2_PITCH;
constexpr int Z2_OFF_PREV = Z2_STAGES * Z2_STAGE_STRIDE;  // r2^k of the plane below the first
constexpr int Z2_OFF_ZK = zm_round128(Z2_OFF_PREV + Z2_BYTES_R);
constexpr int Z2_OFF_MR = zm_round128(Z2_OFF_ZK + 2 * Z2_RING_ZK * 4);
constexpr int Z2_OFF_MP = zm_round128(Z2_OFF_MR + 2 * Z2_RING_MR * 4);
constexpr int Z2_OFF_Z1 = zm_round128(Z2_OFF_MP + 2 * Z2_RING_MP * 4);
constexpr int Z2_OFF_BAR = zm_round128(Z2_OFF_Z1 + 2 * Z2_RING_Z1 * 4);
constexpr int Z2_OFF_FLAG = Z2_OFF_BAR + 8 * (Z2_STAGES + 1);
constexpr int Z2_SMEM = Z2_OFF_FLAG + 16 + 128;

static_assert(Z2_TX % 4 == 0 && Z2_BW <= 256 && Z2_HR <= 256, "TMA box limits");
static_assert(Z2_STAGES >= 2, "two stages at least");
static_assert(Z2_SMEM * TVFGP_Z2_MINB <= 227 * 1024, "CTAs per SM must fit in shared memory");

struct Zmarch2Args {
    CUtensorMap tb, tr0, tr1, tr2, tp0, tp1, tp2;   // b, r_src (3), p_src (3)
    float *p_dst, *r_dst;
    float lam, s, m0, m1;                           // m0: step k, m1: step k+1
    int nx, ny, nz;
    long long N;
    int *err;
    int zc;                                         // output planes per CTA
};

__global__ void __launch_bounds__(Z2_THREADS, TVFGP_Z2_MINB)
fgp_step2_zmarch_tma(const __grid_constant__ Zmarch2Args za)
{
    extern __shared__ unsigned char z2_raw[];
    unsigned char *smem = z2_raw + ((128 - (smem_addr(z2_raw) & 127)) & 127);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Z2_OFF_BAR);   // [STAGES] + prev
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Z2_OFF_FLAG);
    float *ZK = reinterpret_cast<float *>(smem + Z2_OFF_ZK);
    float *MR = reinterpret_cast<float *>(smem + Z2_OFF_MR);
    float *MP = reinterpret_cast<float *>(smem + Z2_OFF_MP);
    float *Z1 = reinterpret_cast<float *>(smem + Z2_OFF_Z1);

    const int nx = za.nx, ny = za.ny, nz = za.nz;
    const int tid = threadIdx.x;
    const int x0 = blockIdx.x * Z2_TX, y0 = blockIdx.y * Z2_TY;
    const int z0 = blockIdx.z * za.zc;
    const int ze = min(z0 + za.zc, nz);        // output planes [z0, ze)
    const int f = max(z0 - 1, 0);              // first plane of step k
    const int uk_last = min(ze, nz - 1);       // last plane of step k (and of z^{k+1})
    const int last = min(ze + 1, nz - 1);      // last staged plane (z^k of plane ze+1)
    const float lam = za.lam, s = za.s, m0 = za.m0, m1 = za.m1;

    if (tid == 0) {
        for (int k = 0; k <= Z2_STAGES; ++k) mbar_init(&bars[k], 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();

    auto slot = [&](int q) { return (q - f) % Z2_STAGES; };
    auto stage = [&](int q) { return smem + slot(q) * Z2_STAGE_STRIDE; };
    auto parity = [&](int q) { return static_cast<uint32_t>(((q - f) / Z2_STAGES) & 1); };
    auto issue = [&](int q) {                   // thread 0 only
        unsigned char *st = stage(q);
        uint64_t *bar = &bars[slot(q)];
        const bool with_p = q <= uk_last;       // the plane past the last step-k plane feeds z^k only
        mbar_expect_tx(bar, with_p ? Z2_TX_ALL : Z2_TX_BR);
        tma_load_3d(st + Z2_OFF_B, &za.tb, x0 - 4, y0 - 1, q, bar);
        tma_load_3d(st + Z2_OFF_R0, &za.tr0, x0 - 4, y0 - 2, q, bar);
        tma_load_3d(st + Z2_OFF_R1, &za.tr1, x0 - 4, y0 - 2, q, bar);
        tma_load_3d(st + Z2_OFF_R2, &za.tr2, x0 - 4, y0 - 2, q, bar);
        if (with_p) {
            tma_load_3d(st + Z2_OFF_P0, &za.tp0, x0 - 4, y0 - 1, q, bar);
            tma_load_3d(st + Z2_OFF_P1, &za.tp1, x0 - 4, y0 - 1, q, bar);
            tma_load_3d(st + Z2_OFF_P2, &za.tp2, x0 - 4, y0 - 1, q, bar);
        }
    };

    // element accessors of a staged plane (local coordinates)
    auto sB = [](const unsigned char *st, int lx, int ly) {
        return reinterpret_cast<const float *>(st + Z2_OFF_B)[(ly + 1) * Z2_BW + lx + 4];
    };
    auto sR = [](const unsigned char *st, int off, int lx, int ly) {
        return reinterpret_cast<const float *>(st + off)[(ly + 2) * Z2_BW + lx + 4];
    };
    auto sP = [](const unsigned char *st, int off, int lx, int ly) {
        return reinterpret_cast<const float *>(st + off)[(ly + 1) * Z2_BW + lx + 4];
    };
    auto zk = [&](int q, int lx, int ly) -> float & {
        return ZK[(q & 1) * Z2_RING_ZK + (ly + 1) * Z2_PITCH + lx + 1];
    };
    auto mr = [&](int q, int a, int lx, int ly) -> float & {
        return MR[(q & 1) * Z2_RING_MR + (a * Z2_UKH + ly + 1) * Z2_PITCH + lx + 1];
    };
    auto mp = [&](int q, int a, int lx, int ly) -> float & {
        return MP[(q & 1) * Z2_RING_MP + (a * Z2_TY + ly) * Z2_TX + lx];
    };
    auto z1 = [&](int q, int lx, int ly) -> float & {
        return Z1[(q & 1) * Z2_RING_Z1 + ly * Z2_PITCH + lx];
    };

    // z^k of plane q on the grown region; r2lo_st: the staged plane q-1 (or
    // the r2 buffer of the plane below the first), nullptr at plane 0
    auto zk_plane = [&](int q, const unsigned char *st, const float *r2lo) {
        for (int idx = tid; idx < Z2_ZKW * Z2_ZKH; idx += Z2_THREADS) {
            const int lx = idx % Z2_ZKW - 1, ly = idx / Z2_ZKW - 1;
            const float d0 = __fsub_rn(sR(st, Z2_OFF_R0, lx, ly), sR(st, Z2_OFF_R0, lx - 1, ly));
            const float d1 = __fsub_rn(sR(st, Z2_OFF_R1, lx, ly), sR(st, Z2_OFF_R1, lx, ly - 1));
            const float lo = r2lo ? r2lo[(ly + 2) * Z2_BW + lx + 4] : 0.0f;
            const float d2 = __fsub_rn(sR(st, Z2_OFF_R2, lx, ly), lo);
            zk(q, lx, ly) = zval(sB(st, lx, ly), lam, d0, d1, d2);
        }
    };

    if (tid == 0) {
        if (f > 0) {
            mbar_expect_tx(&bars[Z2_STAGES], Z2_BYTES_R);
            tma_load_3d(smem + Z2_OFF_PREV, &za.tr2, x0 - 4, y0 - 2, f - 1, &bars[Z2_STAGES]);
        }
        for (int q = f; q <= last && q < f + Z2_STAGES; ++q) issue(q);
    }
    int next_issue = f + Z2_STAGES;

    // prologue: z^k of plane f
    {
        bool ok = true;
        if (f > 0) ok = mbar_wait_tma(&bars[Z2_STAGES], 0);
        ok = ok && mbar_wait_tma(&bars[slot(f)], parity(f));
        if (ok) {
            const float *lo = f > 0 ? reinterpret_cast<const float *>(smem + Z2_OFF_PREV) : nullptr;
            zk_plane(f, stage(f), lo);
        } else {
            *abort_flag = 1;
        }
    }
    __syncthreads();

    float *p0d = za.p_dst, *p1d = za.p_dst + za.N, *p2d = za.p_dst + 2 * za.N;
    float *r0d = za.r_dst, *r1d = za.r_dst + za.N, *r2d = za.r_dst + 2 * za.N;

    int qlast = f - 1;                          // planes <= qlast+1 were waited for
    for (int q = f; q <= ze && *abort_flag == 0; ++q) {
        qlast = q;
        // A: z^k of plane q+1
        if (q + 1 <= last) {
            if (mbar_wait_tma(&bars[slot(q + 1)], parity(q + 1))) {
                const float *lo = reinterpret_cast<const float *>(stage(q) + Z2_OFF_R2);
                zk_plane(q + 1, stage(q + 1), lo);
            } else {
                *abort_flag = 1;
            }
        }
        __syncthreads();
        if (*abort_flag) break;

        // B: step k on plane q over the grown tile -> r^{k+1}, p^{k+1}
        if (q <= uk_last) {
            const unsigned char *st = stage(q);
            const bool hasZ = q + 1 < nz;
            for (int idx = tid; idx < Z2_UKW * Z2_UKH; idx += Z2_THREADS) {
                const int lx = idx % Z2_UKW - 1, ly = idx / Z2_UKW - 1;
                const int x = x0 + lx, y = y0 + ly;
                float r0 = 0.0f, r1 = 0.0f, r2 = 0.0f;
                float p0 = 0.0f, p1 = 0.0f, p2 = 0.0f;
                if (x >= 0 && x < nx && y >= 0 && y < ny) {
                    const float zc = zk(q, lx, ly);
                    const float g0 = (x < nx - 1) ? __fsub_rn(zc, zk(q, lx + 1, ly)) : 0.0f;
                    const float g1 = (y < ny - 1) ? __fsub_rn(zc, zk(q, lx, ly + 1)) : 0.0f;
                    const float g2 = hasZ ? __fsub_rn(zc, zk(q + 1, lx, ly)) : 0.0f;
                    r0 = sR(st, Z2_OFF_R0, lx, ly);
                    r1 = sR(st, Z2_OFF_R1, lx, ly);
                    r2 = sR(st, Z2_OFF_R2, lx, ly);
                    p0 = sP(st, Z2_OFF_P0, lx, ly);
                    p1 = sP(st, Z2_OFF_P1, lx, ly);
                    p2 = sP(st, Z2_OFF_P2, lx, ly);
                    dual_update(r0, r1, r2, g0, g1, g2, p0, p1, p2, s, m0);
                }
                mr(q, 0, lx, ly) = r0;
                mr(q, 1, lx, ly) = r1;
                mr(q, 2, lx, ly) = r2;
                if (lx >= 0 && lx < Z2_TX && ly >= 0 && ly < Z2_TY) {
                    mp(q, 0, lx, ly) = p0;
                    mp(q, 1, lx, ly) = p1;
                    mp(q, 2, lx, ly) = p2;
                }
            }
        }
        __syncthreads();

        // C: z^{k+1} of plane q on the tile plus its x+1 column and y+1 row
        if (q >= z0 && q <= uk_last) {
            const unsigned char *st = stage(q);
            for (int idx = tid; idx < Z2_Z1W * Z2_Z1H; idx += Z2_THREADS) {
                const int lx = idx % Z2_Z1W, ly = idx / Z2_Z1W;
                const float d0 = __fsub_rn(mr(q, 0, lx, ly), mr(q, 0, lx - 1, ly));
                const float d1 = __fsub_rn(mr(q, 1, lx, ly), mr(q, 1, lx, ly - 1));
                const float d2 = __fsub_rn(mr(q, 2, lx, ly), q > 0 ? mr(q - 1, 2, lx, ly) : 0.0f);
                z1(q, lx, ly) = zval(sB(st, lx, ly), lam, d0, d1, d2);
            }
        }
        __syncthreads();
        // every read of plane q's stage is done: the slot takes the next plane
        if (tid == 0 && next_issue <= last && q <= uk_last) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(next_issue++);
        }

        // D: step k+1 on plane q-1 over the tile -> p^{k+2}, r^{k+2} in HBM
        const int qd = q - 1;
        if (qd >= z0 && qd < ze) {
            const bool hasZ = qd + 1 < nz;
            for (int idx = tid; idx < Z2_TX * Z2_TY; idx += Z2_THREADS) {
                const int lx = idx % Z2_TX, ly = idx / Z2_TX;
                const int x = x0 + lx, y = y0 + ly;
                if (x >= nx || y >= ny) continue;
                const float zc = z1(qd, lx, ly);
                const float g0 = (x < nx - 1) ? __fsub_rn(zc, z1(qd, lx + 1, ly)) : 0.0f;
                const float g1 = (y < ny - 1) ? __fsub_rn(zc, z1(qd, lx, ly + 1)) : 0.0f;
                const float g2 = hasZ ? __fsub_rn(zc, z1(qd + 1, lx, ly)) : 0.0f;
                float r0 = mr(qd, 0, lx, ly), r1 = mr(qd, 1, lx, ly), r2 = mr(qd, 2, lx, ly);
                float p0 = mp(qd, 0, lx, ly), p1 = mp(qd, 1, lx, ly), p2 = mp(qd, 2, lx, ly);
                dual_update(r0, r1, r2, g0, g1, g2, p0, p1, p2, s, m1);
                const long long i = x + (long long)nx * (y + (long long)ny * qd);
                p0d[i] = p0;
                p1d[i] = p1;
                p2d[i] = p2;
                r0d[i] = r0;
                r1d[i] = r1;
                r2d[i] = r2;
            }
        }
    }

    if (*abort_flag) {
        __syncthreads();
        if (tid == 0) {
            atomicExch(za.err, kErrTimeout);
            if (f > 0 && qlast < f) mbar_wait_tma(&bars[Z2_STAGES], 0);
            for (int q = qlast + 1; q < next_issue && q <= last; ++q)
                mbar_wait_tma(&bars[slot(q)], parity(q));
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

struct Zmarch2Plan {
    dim3 grid;
    int zc;
};

inline int zmarch2_plan(int nx, int ny, int nz, Zmarch2Plan *plan)
{
    const int tx = (nx + Z2_TX - 1) / Z2_TX, ty = (ny + Z2_TY - 1) / Z2_TY;
    plan->zc = 32;
    plan->grid = dim3(tx, ty, (nz + plan->zc - 1) / plan->zc);
    if (!zmarch_supported(nx, ny, nz)) return 0;
    if (zm_encoder() == nullptr) return 3;
    const void *fn = reinterpret_cast<const void *>(&fgp_step2_zmarch_tma);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, Z2_SMEM) != cudaSuccess) {
        cudaGetLastError();
        return 3;
    }
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, Z2_THREADS, Z2_SMEM) != cudaSuccess) {
        cudaGetLastError();
        return 3;
    }
    plan->zc = zmarch_pick_zc(tx * ty, nz, sms * (per_sm > 0 ? per_sm : 1));
    plan->grid = dim3(tx, ty, (nz + plan->zc - 1) / plan->zc);
    return 0;
}

inline const void *zmarch2_kernel() { return reinterpret_cast<const void *>(&fgp_step2_zmarch_tma); }
inline int zmarch2_threads() { return Z2_THREADS; }
inline size_t zmarch2_smem_bytes() { return Z2_SMEM; }

// Kernel arguments of one two-step launch.
inline bool zmarch2_fill(const Zmarch2Plan &plan, const float *b, const float *p_src, float *p_dst,
                         const float *r_src, float *r_dst, float lam, float s, float m0, float m1,
                         int nx, int ny, int nz, long long N, int *err, Zmarch2Args &za)
{
    za.p_dst = p_dst;
    za.r_dst = r_dst;
    za.lam = lam;
    za.s = s;
    za.m0 = m0;
    za.m1 = m1;
    za.nx = nx;
    za.ny = ny;
    za.nz = nz;
    za.N = N;
    za.err = err;
    za.zc = plan.zc;
    return zm_encode(&za.tb, b, nx, ny, nz, Z2_BW, Z2_HB) &&
           zm_encode(&za.tr0, r_src, nx, ny, nz, Z2_BW, Z2_HR) &&
           zm_encode(&za.tr1, r_src + N, nx, ny, nz, Z2_BW, Z2_HR) &&
           zm_encode(&za.tr2, r_src + 2 * N, nx, ny, nz, Z2_BW, Z2_HR) &&
           zm_encode(&za.tp0, p_src, nx, ny, nz, Z2_BW, Z2_HP) &&
           zm_encode(&za.tp1, p_src + N, nx, ny, nz, Z2_BW, Z2_HP) &&
           zm_encode(&za.tp2, p_src + 2 * N, nx, ny, nz, Z2_BW, Z2_HP);
}

}  // namespace tvfgp
