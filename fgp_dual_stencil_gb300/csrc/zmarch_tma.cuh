// ZMARCH_TMA variant of the FGP step: an x-y tile marching along z, with the
// planes of b and r staged in shared memory by TMA (page "TV solver: the FGP
// step on the GPU", section "Variants", the marching-tile row; rebuilt here
// around the Blackwell tensor memory accelerator instead of plain loads and
// barriers).
//
// A CTA owns the columns x0..x0+TX-1 (TX = 32 by default) and computes z
// for the ROWS = 16 rows y0..y0+15 of each plane; it updates the dual on the
// first 15 rows (the 16th row's z is the y+1 neighbour of the 15th).  It
// walks zc planes in z (chosen per volume at set-up).  For each plane q a
// TMA load brings, into one slot of a 4-deep ring:
//   b  at x0..x0+TX+3,   y0..y0+15        (z(x0+TX) is the x+1 neighbour)
//   r0 at x0-4..x0+TX+3, y0..y0+15        (r0(x-1) for L)
//   r1 at x0..x0+TX+3,   y0-1..y0+15      (r1(y-1) for L)
//   r2 at x0..x0+TX+3,   y0..y0+15
//   p0, p1, p2 at x0..x0+TX-1, y0..y0+14  (the voxels' own p)
// Coordinates outside the volume read as zero, which is the r_a(-1) = 0
// boundary of L.  A thread owns 4 consecutive x voxels of one row: it keeps
// its own r and z of the current and next plane in registers, so only the
// z of the x+1 and y+1 neighbours goes through shared memory (a 3-slot ring
// of z planes: one barrier per plane suffices).  Every load of the step is a
// TMA copy issued planes ahead, before any wait on it: the voxel's own p and
// r arrive with their plane, and no thread issues a global load.
//
// The kernel is a template on the storage of p and r: fp32, or binary16
// (TMA boxes of halves, widened exactly to fp32 on their way out of shared
// memory; the step's arithmetic is the same fp32 sequence, and stored
// values are rounded to nearest-even).  Half boxes start on 8-column
// boundaries, so the r0 box then starts at x0-8 and the r1, r2 boxes span
// x0..x0+TX+7.
//
// Every wait on a TMA barrier is bounded; on timeout the kernel sets the
// caller's error word, drains its outstanding copies (again bounded) and
// returns, so the context stays usable (tvfgp_check reports it).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "fgp_kernels.cuh"

namespace tvfgp {

// Tile shape of the fp32 march, and the _H twins for a binary16 dual.
#ifndef TVFGP_ZM_TX
#define TVFGP_ZM_TX 32
#endif
#ifndef TVFGP_ZM_ROWS
#define TVFGP_ZM_ROWS 16
#endif
#ifndef TVFGP_ZM_STAGES
#define TVFGP_ZM_STAGES 4
#endif
#ifndef TVFGP_ZM_MINB
#define TVFGP_ZM_MINB 3
#endif
#ifndef TVFGP_ZM_TX_H
#define TVFGP_ZM_TX_H 32
#endif
#ifndef TVFGP_ZM_ROWS_H
#define TVFGP_ZM_ROWS_H 16
#endif
#ifndef TVFGP_ZM_STAGES_H
#define TVFGP_ZM_STAGES_H 4
#endif
#ifndef TVFGP_ZM_MINB_H
#define TVFGP_ZM_MINB_H 4
#endif
#ifndef TVFGP_ZM_ZC_MAX
#define TVFGP_ZM_ZC_MAX 32        // most planes per CTA
#endif
#ifndef TVFGP_ZM_WAVES
#define TVFGP_ZM_WAVES 4          // fewest waves of CTAs over the resident slots
#endif
#ifndef TVFGP_ZM_L2PROMO
#define TVFGP_ZM_L2PROMO CU_TENSOR_MAP_L2_PROMOTION_L2_256B
#endif
constexpr int ZM_MAX_POLLS = 1 << 22;     // bound of every barrier wait, in polls ...
constexpr unsigned long long ZM_MAX_WAIT_NS = 1000000000ull;   // ... and in time (1 s)

constexpr int zm_round128(int v) { return (v + 127) / 128 * 128; }

// Tile and shared-memory layout of one z-march for a dual stored as TS
// (float or __half; b and z are always fp32).  A CTA owns TX columns and
// computes z on ROWS rows of each plane, updating the dual on the first
// TY = ROWS-1; a thread owns a quad of 4 x voxels of one row.  A TMA box
// starts on a 16-byte column, so the r0 box starts XO = 16 / sizeof(TS)
// columns left of the tile (its column XO-1 is r0(x0-1)) and the r1, r2
// boxes are XO columns wider than the tile (their column TX is the x+1
// halo): 4 columns for fp32, 8 for binary16.
template <typename TS>
struct ZmLayout {
    static constexpr bool F32 = sizeof(TS) == 4;
    static constexpr int TX = F32 ? TVFGP_ZM_TX : TVFGP_ZM_TX_H;          // tile width (voxels)
    static constexpr int ROWS = F32 ? TVFGP_ZM_ROWS : TVFGP_ZM_ROWS_H;    // rows whose z is computed
    static constexpr int TY = ROWS - 1;                                   // rows whose dual is updated
    static constexpr int QX = TX / 4;                                     // quads per row
    static constexpr int THREADS = QX * ROWS;
    static constexpr int STAGES = F32 ? TVFGP_ZM_STAGES : TVFGP_ZM_STAGES_H;  // planes in flight
    // resident CTAs per SM the registers are budgeted for
    static constexpr int MINB = F32 ? TVFGP_ZM_MINB : TVFGP_ZM_MINB_H;
    static constexpr int BW = TX + 4;           // width of the b box (fp32)
    static constexpr int HB = ROWS;             // height of the b, r0, r2 boxes
    static constexpr int H1 = ROWS + 1;         // height of the r1 box
    static constexpr int ZP = TX + 4;           // row pitch of a z plane
    static constexpr int ES = static_cast<int>(sizeof(TS));
    static constexpr int XO = 16 / ES;
    static constexpr int W0 = TX + 2 * XO;      // width of the r0 box
    static constexpr int RW = TX + XO;          // width of the r1, r2 boxes
    static constexpr int BYTES_B = BW * HB * 4;
    static constexpr int BYTES_R0 = W0 * HB * ES;
    static constexpr int BYTES_R1 = RW * H1 * ES;
    static constexpr int BYTES_R2 = RW * HB * ES;
    static constexpr int BYTES_P = TX * TY * ES;     // one component of p
    static constexpr int OFF_B = 0;
    static constexpr int OFF_R0 = zm_round128(OFF_B + BYTES_B);
    static constexpr int OFF_R1 = zm_round128(OFF_R0 + BYTES_R0);
    static constexpr int OFF_R2 = zm_round128(OFF_R1 + BYTES_R1);
    static constexpr int OFF_P0 = zm_round128(OFF_R2 + BYTES_R2);
    static constexpr int OFF_P1 = zm_round128(OFF_P0 + BYTES_P);
    static constexpr int OFF_P2 = zm_round128(OFF_P1 + BYTES_P);
    static constexpr int STAGE_STRIDE = zm_round128(OFF_P2 + BYTES_P);
    static constexpr int STAGE_TX_BR = BYTES_B + BYTES_R0 + BYTES_R1 + BYTES_R2;
    static constexpr int STAGE_TX = STAGE_TX_BR + 3 * BYTES_P;
    static constexpr int OFF_PREV = STAGES * STAGE_STRIDE;               // r2 of plane z0-1
    static constexpr int OFF_Z = zm_round128(OFF_PREV + BYTES_R2);       // 3 z planes
    static constexpr int BYTES_Z = 3 * ROWS * ZP * 4;
    static constexpr int OFF_BAR = zm_round128(OFF_Z + BYTES_Z);         // STAGES+1 barriers
    static constexpr int OFF_FLAG = OFF_BAR + 8 * (STAGES + 1);
    static constexpr int SMEM = OFF_FLAG + 16 + 128;                     // + base alignment

    static_assert(TX % 4 == 0 && W0 <= 256 && H1 <= 256 && THREADS <= 1024, "TMA box limits");
    static_assert((W0 * ES) % 16 == 0 && (RW * ES) % 16 == 0 && (TX * ES) % 16 == 0,
                  "TMA box rows are whole 16-byte units");
    static_assert(SMEM * MINB <= 227 * 1024, "CTAs per SM must fit in shared memory");
    // Plane q's slot holds its p until the dual update of q, one iteration
    // after its b and r were consumed; the next plane is loaded into the slot
    // of q-1, so a plane is issued S-1 iterations before its wait: S >= 3.
    static_assert(STAGES >= 3, "the ring needs three slots");
};

struct ZmarchPlan {
    dim3 grid;
    int zc;                       // planes per CTA
};

template <typename TS>
struct ZmarchArgsT {
    CUtensorMap tb, t0, t1, t2;   // b, r0, r1, r2 of the r read by this step
    CUtensorMap tp0, tp1, tp2;    // the three components of p
    StepArgsT<TS> a;
    int *err;
    int zc;                       // planes per CTA (grid.z = ceil(nz / zc))
    int max_polls;                // bound of the waits for data (the drain after a timeout keeps ZM_MAX_POLLS) ...
    int poll_from;                // ... for planes >= the CTA's first + poll_from
};
using ZmarchArgs = ZmarchArgsT<float>;

// ---------------------------------------------------------------------------
// device helpers (TMA, mbarrier)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long globaltimer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity, at most `polls` polls (a poll
// may suspend the thread for a hardware-defined time) and, from the 256th
// poll on, at most ZM_MAX_WAIT_NS of wall-clock time.  False: gave up.
__device__ __forceinline__ bool mbar_wait_tma(uint64_t *bar, uint32_t parity, int polls = ZM_MAX_POLLS)
{
    unsigned long long start = 0;
    for (int k = 0; k < polls; ++k) {
        if (mbar_try(bar, parity)) return true;
        if ((k & 255) == 255) {
            const unsigned long long now = globaltimer_ns();
            if (k == 255)
                start = now;
            else if (now - start > ZM_MAX_WAIT_NS)
                return false;
        }
    }
    return false;
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ float4 lds4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 lds4(const __half *p) { return widen4(*reinterpret_cast<const uint2 *>(p)); }
__device__ __forceinline__ float lds1(const float *p) { return *p; }
__device__ __forceinline__ float lds1(const __half *p) { return __half2float(*p); }

// z of the quad (row, 4*qx) of a staged plane; r2lo is r2 of the plane below.
template <typename TS>
__device__ __forceinline__ void zm_quad(const unsigned char *st, int row, int qx, float4 r2lo,
                                        float lam, float4 &R0, float4 &R1, float4 &R2, float4 &Z)
{
    using L = ZmLayout<TS>;
    const float *B = reinterpret_cast<const float *>(st + L::OFF_B);
    const TS *S0 = reinterpret_cast<const TS *>(st + L::OFF_R0);
    const TS *S1 = reinterpret_cast<const TS *>(st + L::OFF_R1);
    const TS *S2 = reinterpret_cast<const TS *>(st + L::OFF_R2);
    const int c = 4 * qx;
    const float4 Bq = lds4(B + row * L::BW + c);
    R0 = lds4(S0 + row * L::W0 + L::XO + c);
    const float left = lds1(S0 + row * L::W0 + L::XO - 1 + c);
    R1 = lds4(S1 + (row + 1) * L::RW + c);
    const float4 R1lo = lds4(S1 + row * L::RW + c);
    R2 = lds4(S2 + row * L::RW + c);
    Z = zquad(Bq, R0, R1, R2, left, R1lo, r2lo, lam, neg_zero(lam));
}

// z at column x0+TX of a row (the x+1 neighbour of the tile's last quad).
template <typename TS>
__device__ __forceinline__ float zm_halo(const unsigned char *st, int row, float r2lo, float lam,
                                         float &r2here)
{
    using L = ZmLayout<TS>;
    const float *B = reinterpret_cast<const float *>(st + L::OFF_B);
    const TS *S0 = reinterpret_cast<const TS *>(st + L::OFF_R0);
    const TS *S1 = reinterpret_cast<const TS *>(st + L::OFF_R1);
    const TS *S2 = reinterpret_cast<const TS *>(st + L::OFF_R2);
    r2here = lds1(S2 + row * L::RW + L::TX);
    return zval(B[row * L::BW + L::TX], lam,
                __fsub_rn(lds1(S0 + row * L::W0 + L::XO + L::TX), lds1(S0 + row * L::W0 + L::XO - 1 + L::TX)),
                __fsub_rn(lds1(S1 + (row + 1) * L::RW + L::TX), lds1(S1 + row * L::RW + L::TX)),
                __fsub_rn(r2here, r2lo));
}

template <typename TS>
__global__ void __launch_bounds__(ZmLayout<TS>::THREADS, ZmLayout<TS>::MINB)
    fgp_step_zmarch_tma(const __grid_constant__ ZmarchArgsT<TS> za)
{
    using L = ZmLayout<TS>;
    extern __shared__ unsigned char zm_raw[];
    unsigned char *smem = zm_raw + ((128 - (smem_addr(zm_raw) & 127)) & 127);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);   // [STAGES] + prev
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_FLAG);
    float *zpl = reinterpret_cast<float *>(smem + L::OFF_Z);

    const StepArgsT<TS> &a = za.a;
    const int nx = a.nx, ny = a.ny, nz = a.nz;
    const int tid = threadIdx.x;
    const int qx = tid % L::QX, row = tid / L::QX;
    const int x0 = blockIdx.x * L::TX, y0 = blockIdx.y * L::TY;
    const int z0 = blockIdx.z * za.zc;
    const int ze = min(z0 + za.zc, nz);            // planes updated: [z0, ze)
    const int qmax = min(ze, nz - 1);              // last plane whose z is needed
    const int x = x0 + 4 * qx, y = y0 + row;
    const bool upd = (row < L::TY) && (x < nx) && (y < ny);
    const bool hasY = (y + 1 < ny);
    const float lam = a.lam, s = a.s, m = a.m;

    if (tid == 0) {
        for (int k = 0; k <= L::STAGES; ++k) mbar_init(&bars[k], 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();

    auto issue = [&](int q) {                       // thread 0 only
        unsigned char *st = smem + ((q - z0) % L::STAGES) * L::STAGE_STRIDE;
        uint64_t *bar = &bars[(q - z0) % L::STAGES];
        const bool with_p = q < ze;                 // plane ze only feeds z(i+ez)
        mbar_expect_tx(bar, with_p ? L::STAGE_TX : L::STAGE_TX_BR);
        if (with_p) {
            tma_load_3d(st + L::OFF_P0, &za.tp0, x0, y0, q, bar);
            tma_load_3d(st + L::OFF_P1, &za.tp1, x0, y0, q, bar);
            tma_load_3d(st + L::OFF_P2, &za.tp2, x0, y0, q, bar);
        }
        tma_load_3d(st + L::OFF_B, &za.tb, x0, y0, q, bar);
        tma_load_3d(st + L::OFF_R0, &za.t0, x0 - L::XO, y0, q, bar);
        tma_load_3d(st + L::OFF_R1, &za.t1, x0, y0 - 1, q, bar);
        tma_load_3d(st + L::OFF_R2, &za.t2, x0, y0, q, bar);
    };
    if (tid == 0) {
        if (z0 > 0) {
            mbar_expect_tx(&bars[L::STAGES], L::BYTES_R2);
            tma_load_3d(smem + L::OFF_PREV, &za.t2, x0, y0, z0 - 1, &bars[L::STAGES]);
        }
        for (int q = z0; q <= qmax && q < z0 + L::STAGES; ++q) issue(q);
    }
    int next_issue = z0 + L::STAGES;               // next plane to load (thread 0)

    auto stage_of = [&](int q) { return smem + ((q - z0) % L::STAGES) * L::STAGE_STRIDE; };
    auto parity_of = [&](int q) { return static_cast<uint32_t>(((q - z0) / L::STAGES) & 1); };
    auto zrow = [&](int q, int rr) { return zpl + ((q % 3) * L::ROWS + rr) * L::ZP; };

    // prologue: z of plane z0, own r at z0.  The z at column x0+TX of every
    // row (the x+1 neighbour of the row's last quad) is computed by thread
    // hrow = tid for rows tid < ROWS: one warp does all rows at once.
    float4 Rc0, Rc1, Rc2, Zc;
    const bool do_halo = tid < L::ROWS;
    const int hrow = tid;
    float r2halo = 0.0f;                            // r2 at column x0+TX of row hrow, current plane
    bool ok = true;
    {
        float4 r2lo = f4zero();
        float r2lo_h = 0.0f;
        if (z0 > 0) {
            ok = mbar_wait_tma(&bars[L::STAGES], 0, za.poll_from <= 0 ? za.max_polls : ZM_MAX_POLLS);
            const TS *P2 = reinterpret_cast<const TS *>(smem + L::OFF_PREV);
            r2lo = lds4(P2 + row * L::RW + 4 * qx);
            if (do_halo) r2lo_h = lds1(P2 + hrow * L::RW + L::TX);
        }
        ok = ok && mbar_wait_tma(&bars[0], 0, za.poll_from <= 0 ? za.max_polls : ZM_MAX_POLLS);
        if (ok) {
            const unsigned char *st = stage_of(z0);
            zm_quad<TS>(st, row, qx, r2lo, lam, Rc0, Rc1, Rc2, Zc);
            float *zr = zrow(z0, row);
            *reinterpret_cast<float4 *>(zr + 4 * qx) = Zc;
            if (do_halo) zrow(z0, hrow)[L::TX] = zm_halo<TS>(st, hrow, r2lo_h, lam, r2halo);
        } else {
            *abort_flag = 1;
        }
    }
    __syncthreads();

    TS *p0 = a.p, *p1 = a.p + a.N, *p2 = a.p + 2 * a.N;
    TS *o0 = a.rd, *o1 = a.rd + a.N, *o2 = a.rd + 2 * a.N;

    int zlast = z0 - 1;                            // planes <= zlast+1 were waited for
    for (int z = z0; z < ze && *abort_flag == 0; ++z) {
        zlast = z;
        const long long i = x + (long long)nx * (y + (long long)ny * z);
        // (1) z of plane z+1 from its staged planes (own r2 of plane z is its
        //     z-lower neighbour)
        const bool hasZ = (z + 1 < nz);
        float4 Rn0 = f4zero(), Rn1 = f4zero(), Rn2 = f4zero(), Zn = f4zero();
        float r2halo_n = 0.0f;
        if (hasZ) {
            if (mbar_wait_tma(&bars[(z + 1 - z0) % L::STAGES], parity_of(z + 1),
                              z + 1 - z0 >= za.poll_from ? za.max_polls : ZM_MAX_POLLS)) {
                const unsigned char *st = stage_of(z + 1);
                zm_quad<TS>(st, row, qx, Rc2, lam, Rn0, Rn1, Rn2, Zn);
                float *zr = zrow(z + 1, row);
                *reinterpret_cast<float4 *>(zr + 4 * qx) = Zn;
                if (do_halo) zrow(z + 1, hrow)[L::TX] = zm_halo<TS>(st, hrow, r2halo, lam, r2halo_n);
            } else {
                *abort_flag = 1;
            }
        }
        __syncthreads();
        if (*abort_flag) break;
        // every thread finished plane z-1 (its dual update read that slot's
        // p): the slot takes the next plane
        if (tid == 0 && z > z0 && next_issue <= qmax) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(next_issue++);
        }
        // (2) dual update of plane z, with its own p from the staged plane
        if (upd) {
            const unsigned char *stz = stage_of(z);
            const int pofs = row * L::TX + 4 * qx;
            float4 P0 = lds4(reinterpret_cast<const TS *>(stz + L::OFF_P0) + pofs);
            float4 P1 = lds4(reinterpret_cast<const TS *>(stz + L::OFF_P1) + pofs);
            float4 P2 = lds4(reinterpret_cast<const TS *>(stz + L::OFF_P2) + pofs);
            const float *zr = zrow(z, row);
            const float zx = zr[4 * qx + 4];
            const float4 ZY = hasY ? lds4(zrow(z, row + 1) + 4 * qx) : f4zero();
            const float gx3 = (x + 3 < nx - 1) ? __fsub_rn(Zc.w, zx) : 0.0f;
            float4 G1 = f4zero(), G2 = f4zero();
            if (hasY) {
                G1.x = __fsub_rn(Zc.x, ZY.x); G1.y = __fsub_rn(Zc.y, ZY.y);
                G1.z = __fsub_rn(Zc.z, ZY.z); G1.w = __fsub_rn(Zc.w, ZY.w);
            }
            if (hasZ) {
                G2.x = __fsub_rn(Zc.x, Zn.x); G2.y = __fsub_rn(Zc.y, Zn.y);
                G2.z = __fsub_rn(Zc.z, Zn.z); G2.w = __fsub_rn(Zc.w, Zn.w);
            }
            float4 N0 = Rc0, N1 = Rc1, N2 = Rc2;
            const float4 G0 = make_float4(__fsub_rn(Zc.x, Zc.y), __fsub_rn(Zc.y, Zc.z), __fsub_rn(Zc.z, Zc.w), gx3);
            dual_update4(N0, N1, N2, G0, G1, G2, P0, P1, P2, s, m, neg_zero(lam));
            stv(p0 + i, P0);
            stv(p1 + i, P1);
            stv(p2 + i, P2);
            stv(o0 + i, N0);
            stv(o1 + i, N1);
            stv(o2 + i, N2);
        }
        Rc0 = Rn0;
        Rc1 = Rn1;
        Rc2 = Rn2;
        Zc = Zn;
        r2halo = r2halo_n;
    }

    if (*abort_flag) {
        // A wait gave up.  Record it, then drain (bounded) every copy this
        // CTA issued that is still in flight: plane zlast+1 (whose wait
        // failed, or z0 when the prologue failed) and all later ones.
        __syncthreads();
        if (tid == 0) {
            atomicExch(za.err, kErrTimeout);
            if (z0 > 0 && zlast < z0) mbar_wait_tma(&bars[L::STAGES], 0);
            for (int q = zlast + 1; q < next_issue && q <= qmax; ++q)
                mbar_wait_tma(&bars[(q - z0) % L::STAGES], parity_of(q));
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

inline PFN_cuTensorMapEncodeTiled_v12000 zm_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// The fp32 march needs rows of whole 16-byte units (nx % 4 == 0), the
// binary16 one nx % 8 == 0; both need 16-byte aligned base addresses.
template <typename TS = float>
inline bool zmarch_supported(int nx, int, int) { return nx % ZmLayout<TS>::XO == 0; }

// The variant needs the driver's tensor-map encoder.
inline bool zmarch_available() { return zm_encoder() != nullptr; }

// Planes per CTA: the deepest march, up to zc_max planes (fewest repeated
// prologue planes), that still gives at least `waves` waves of CTAs over the
// GPU's resident slots, so the last partial wave costs little.
inline int zmarch_pick_zc(int tiles_xy, int nz, int slots, int zc_max = 32, int waves = 4)
{
    static const int cand[] = {128, 96, 64, 48, 32, 24, 16, 12, 8};
    for (int zc : cand) {
        if (zc > zc_max) continue;
        const long long ctas = static_cast<long long>(tiles_xy) * ((nz + zc - 1) / zc);
        if (ctas >= static_cast<long long>(waves) * slots) return zc;
    }
    return 8;
}

template <typename TS = float>
inline const void *zmarch_kernel() { return reinterpret_cast<const void *>(&fgp_step_zmarch_tma<TS>); }
template <typename TS = float>
inline int zmarch_threads() { return ZmLayout<TS>::THREADS; }
inline dim3 zmarch_grid(const ZmarchPlan &p) { return p.grid; }
template <typename TS = float>
inline size_t zmarch_smem_bytes() { return ZmLayout<TS>::SMEM; }

template <typename TS = float>
inline int zmarch_plan(int nx, int ny, int nz, ZmarchPlan *plan)
{
    using L = ZmLayout<TS>;
    const int tx = (nx + L::TX - 1) / L::TX, ty = (ny + L::TY - 1) / L::TY;
    plan->zc = 32;
    plan->grid = dim3(tx, ty, (nz + plan->zc - 1) / plan->zc);
    if (!zmarch_supported<TS>(nx, ny, nz)) return 0;
    if (zm_encoder() == nullptr) return 3;
    const void *fn = zmarch_kernel<TS>();
    const int smem = ZmLayout<TS>::SMEM;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
        cudaGetLastError();
        return 3;
    }
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, L::THREADS, smem) != cudaSuccess) {
        cudaGetLastError();
        return 3;
    }
    plan->zc = zmarch_pick_zc(tx * ty, nz, sms * (per_sm > 0 ? per_sm : 1), TVFGP_ZM_ZC_MAX, TVFGP_ZM_WAVES);
    plan->grid = dim3(tx, ty, (nz + plan->zc - 1) / plan->zc);
    return 0;
}

template <typename T>
inline bool zm_encode(CUtensorMap *map, const T *base, int nx, int ny, int nz, int bw, int bh)
{
    constexpr cuuint64_t es = sizeof(T);
    const CUtensorMapDataType dt = es == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const cuuint64_t dims[3] = {(cuuint64_t)nx, (cuuint64_t)ny, (cuuint64_t)nz};
    const cuuint64_t strides[2] = {(cuuint64_t)nx * es, (cuuint64_t)nx * ny * es};
    const cuuint32_t box[3] = {(cuuint32_t)bw, (cuuint32_t)bh, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return zm_encoder()(map, dt, 3, const_cast<T *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, TVFGP_ZM_L2PROMO,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Fill the kernel arguments of one step: tensor maps of b, of the three
// components of p and of the three components of r_src.  Returns false if
// an encoding fails.
template <typename TS>
inline bool zmarch_fill(const ZmarchPlan &plan, const StepArgsT<TS> &a, int *err, ZmarchArgsT<TS> &za)
{
    using L = ZmLayout<TS>;
    za.a = a;
    za.err = err;
    za.zc = plan.zc;
    za.max_polls = ZM_MAX_POLLS;
    za.poll_from = 0;
    const TS *r = a.rs;
    return zm_encode(&za.tp0, a.p, a.nx, a.ny, a.nz, L::TX, L::TY) &&
           zm_encode(&za.tp1, a.p + a.N, a.nx, a.ny, a.nz, L::TX, L::TY) &&
           zm_encode(&za.tp2, a.p + 2 * a.N, a.nx, a.ny, a.nz, L::TX, L::TY) &&
           zm_encode(&za.tb, a.b, a.nx, a.ny, a.nz, L::BW, L::HB) &&
           zm_encode(&za.t0, r, a.nx, a.ny, a.nz, L::W0, L::HB) &&
           zm_encode(&za.t1, r + a.N, a.nx, a.ny, a.nz, L::RW, L::H1) &&
           zm_encode(&za.t2, r + 2 * a.N, a.nx, a.ny, a.nz, L::RW, L::HB);
}

}  // namespace tvfgp
