// ZMARCH2_TMA: two FGP steps per pass over HBM (temporal blocking of the
// z-march).
//
// The page ("TV solver: the FGP step on the GPU", "Profiler counters") shows
// the step at its compulsory 13 volumes, so a cheaper step has to move fewer
// bytes.  Without changing the result, that means computing two
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
//     B  step k  of plane q   on x0-1..x0+TX,   y0-1..y0+TY     (-> r_x, r_y^{k+1} shared, all in registers)
//     -- barrier
//     C  z^{k+1} of plane q   on x0..x0+TX,     y0..y0+TY       (b, own r^{k+1} in registers)
//     D  step k+1 of plane q-1 on the tile                      (-> p^{k+2}, r^{k+2} in HBM)
//
// One barrier per plane suffices.  Across it every phase reads what the
// phases before it wrote.  Without a second one, a thread may already run
// A and B of plane q+1 while another still runs C and D of plane q, so what
// the latter read must not be overwritten by the former: C and step k+1
// take the quad's own r^{k+1} (and step k+1 its p^{k+1}) from the registers
// of the thread that made them, and C reads from shared memory only r_x of
// plane q at x-1 and r_y at y-1, which B of plane q+1 writes into the other
// of two slots.  r_z^{k+1} is needed only at the quad's own column, so it
// never goes through shared memory.  The z rings and the stages are written
// only at points that one barrier already separates from their readers; a
// wait that gives up is reported through that barrier (its OR over the
// threads).
//
// Each thread owns one quad (four x voxels) and runs A and B, and C and D,
// on it: the voxel's own z^k, z^{k+1}, p^{k+1} and r^{k+1} stay in its
// registers from the phase that makes them to the phase that uses them, and
// only the x+1 / y+1 neighbours' z and the r^{k+1} halo go through shared
// memory (rings of two planes).  Voxels of the ring that
// lie outside the volume get r^{k+1} = 0: that is the r(-1) = 0 boundary step
// k+1 sees.
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

#include <type_traits>

#include "zmarch_tma.cuh"

namespace tvfgp {

#ifndef TVFGP_Z2_TX
#define TVFGP_Z2_TX 32
#endif
#ifndef TVFGP_Z2_TY
#define TVFGP_Z2_TY 12
#endif
#ifndef TVFGP_Z2_STAGES
#define TVFGP_Z2_STAGES 3
#endif
#ifndef TVFGP_Z2_CTAS
#define TVFGP_Z2_CTAS 3           // CTAs per SM the shared memory is sized for
#endif
// The minimum CTAs per SM given to the compiler: 2 leaves it up to 204
// registers a thread; it takes 110 to 118 (by version of the kernel), for
// a schedule measured 0.4-0.5% faster than the one it builds within the
// 136 that 3 CTAs allow.  Three CTAs still fit while it takes at most 136
// (3 x 160 x 136 <= 65536); the build log shows the count.
#ifndef TVFGP_Z2_MINB
#define TVFGP_Z2_MINB 2
#endif
#ifndef TVFGP_Z2_ZC_MAX
#define TVFGP_Z2_ZC_MAX 128       // most output planes per CTA
#endif
#ifndef TVFGP_Z2_WAVES
#define TVFGP_Z2_WAVES 2          // fewest waves of CTAs over the resident slots
#endif
#ifndef TVFGP_Z2_TAPER
#define TVFGP_Z2_TAPER 1          // the last chunk of planes split in 3 (1), 2 (2) or kept (0)
#endif
#ifndef TVFGP_Z2_EDGE_SPLIT
#define TVFGP_Z2_EDGE_SPLIT 1     // boundary tests in step k only in CTAs that touch a face
#endif

constexpr int Z2_TX = TVFGP_Z2_TX;          // output tile width
constexpr int Z2_TY = TVFGP_Z2_TY;          // output tile height
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

// Regions (local coordinates lx = x - x0, ly = y - y0), in quads of four x
// voxels so that shared memory moves float4s.  Each region covers what the
// next phase needs (and a few columns more, which nothing reads):
//   z^k      lx -4..TX+3 (needed -1..TX+1),  ly -1..TY+1
//   step k   lx -4..TX+3 (needed -1..TX),    ly -1..TY
//   z^{k+1}  lx  0..TX+3 (needed  0..TX),    ly  0..TY
//   step k+1 lx  0..TX-1,                    ly  0..TY-1
constexpr int Z2_QA = Z2_BW / 4;                          // quads per row, z^k and step k
constexpr int Z2_QC = (Z2_TX + 4) / 4;                    // quads per row, z^{k+1}
constexpr int Z2_QD = Z2_TX / 4;                          // quads per row, step k+1
constexpr int Z2_TASKS_A = Z2_QA * (Z2_TY + 3);
constexpr int Z2_TASKS_B = Z2_QA * (Z2_TY + 2);
constexpr int Z2_TASKS_C = Z2_QC * (Z2_TY + 1);
constexpr int Z2_TASKS_D = Z2_QD * Z2_TY;
// One thread per z^k quad.  Threads are numbered so that the phases after
// the first barrier run on as few warps as possible: threads
// [0, TASKS_D) own the tile's quads (row-major, QD per row) and run all four
// phases on them; threads [TASKS_D, TASKS_B) own the ring of the grown tile
// (its first and last rows, then its left and right quad columns) and run z^k
// and step k; threads [TASKS_B, TASKS_A) own z^k's extra last row.  Each
// z^{k+1} quad (the tile, its x+1 column and its y+1 row) is computed by the
// thread that computed z^k at the same place one plane earlier, which keeps
// that quad's b in registers: phase C reads no staged plane, so a stage is
// free for the next copy right after the first barrier.
constexpr int Z2_THREADS = (Z2_TASKS_A + 31) / 32 * 32;
// The thread that issues the copies of the next planes: the last one, in the
// warp with the least work (none of the tile's four phases).
#ifndef TVFGP_Z2_PRODUCER
#define TVFGP_Z2_PRODUCER (Z2_THREADS - 1)
#endif
constexpr int Z2_PRODUCER = TVFGP_Z2_PRODUCER;
constexpr int Z2_RING_B = Z2_TASKS_B - Z2_TASKS_D;        // 2 QA + 2 TY
static_assert(Z2_RING_B == 2 * Z2_QA + 2 * Z2_TY && Z2_TASKS_A - Z2_TASKS_B == Z2_QA, "thread roles");
static_assert(Z2_TASKS_B <= Z2_THREADS && Z2_TASKS_A <= Z2_THREADS, "thread roles");

// shared rings (z^k, z^{k+1}, and r_x, r_y of r^{k+1}: two slots each, see
// above); pitches in floats
constexpr int Z2_PK = Z2_BW;                              // z^k and r^{k+1}: columns lx+4
constexpr int Z2_P1 = Z2_TX + 4;                          // z^{k+1}: columns lx
constexpr int Z2_RING_ZK = (Z2_TY + 3) * Z2_PK;           // floats per slot
constexpr int Z2_MR_COMP = (Z2_TY + 2) * Z2_PK;
constexpr int Z2_MR_SLOTS = 2 + 2;                        // r_x, r_y: 2 slots each
constexpr int Z2_RING_Z1 = (Z2_TY + 1) * Z2_P1;
constexpr int Z2_OFF_ZK = Z2_STAGES * Z2_STAGE_STRIDE;
constexpr int Z2_OFF_MR = zm_round128(Z2_OFF_ZK + 2 * Z2_RING_ZK * 4);
constexpr int Z2_OFF_Z1 = zm_round128(Z2_OFF_MR + Z2_MR_SLOTS * Z2_MR_COMP * 4);
// r2^k of the plane below the first: read only by the prologue, before the
// z^{k+1} ring is first written, so it shares that ring's memory
constexpr int Z2_OFF_PREV = Z2_OFF_Z1;
constexpr int Z2_OFF_BAR = zm_round128(Z2_OFF_Z1 + 2 * Z2_RING_Z1 * 4);
constexpr int Z2_SMEM = Z2_OFF_BAR + 8 * (Z2_STAGES + 1) + 128;

static_assert(Z2_TX % 4 == 0 && Z2_BW <= 256 && Z2_HR <= 256, "TMA box limits");
static_assert(Z2_STAGES >= 2, "two stages at least");
static_assert(Z2_BYTES_R <= 2 * Z2_RING_Z1 * 4, "the prologue's r2 box fits in the z^{k+1} ring");
static_assert(Z2_SMEM * TVFGP_Z2_CTAS <= 227 * 1024, "CTAs per SM must fit in shared memory");

struct Zmarch2Args {
    CUtensorMap tb, tr0, tr1, tr2, tp0, tp1, tp2;   // b, r_src (3), p_src (3)
    float *p_dst, *r_dst;
    float lam, s, m0, m1;                           // m0: step k, m1: step k+1
    int nx, ny, nz;
    long long N;
    int *err;
    int zc;                                         // output planes per CTA ...
    int nbig;                                       // ... for blockIdx.z < nbig; then the
    int tap[4];                                     // pieces [tap[j], tap[j+1]) after nbig*zc
    int opx;                                        // row pitch of p_dst, r_dst (nx: dense)
    long long No;                                   // their elements per component
    int max_polls;                                  // bound of the waits for data (drain: ZM_MAX_POLLS) ...
    int poll_from;                                  // ... for planes >= the CTA's first + poll_from
};

// PADDED_OUT: p_dst and r_dst have rows of opx floats (even), written as
// 8-byte halves of quads; else they are dense.
template <bool PADDED_OUT>
__global__ void __launch_bounds__(Z2_THREADS, TVFGP_Z2_MINB)
fgp_step2_zmarch_tma(const __grid_constant__ Zmarch2Args za)
{
    extern __shared__ unsigned char z2_raw[];
    unsigned char *smem = z2_raw + ((128 - (smem_addr(z2_raw) & 127)) & 127);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Z2_OFF_BAR);   // [STAGES] + prev
    float *ZK = reinterpret_cast<float *>(smem + Z2_OFF_ZK);
    float *MR = reinterpret_cast<float *>(smem + Z2_OFF_MR);
    float *Z1 = reinterpret_cast<float *>(smem + Z2_OFF_Z1);

    const int nx = za.nx, ny = za.ny, nz = za.nz;
    const int tid = threadIdx.x;
    const int x0 = blockIdx.x * Z2_TX, y0 = blockIdx.y * Z2_TY;
    const int jz = blockIdx.z;
    const int zbase = jz < za.nbig ? 0 : za.nbig * za.zc;
    const int z0 = jz < za.nbig ? jz * za.zc : zbase + za.tap[jz - za.nbig];
    const int ze = min(jz < za.nbig ? z0 + za.zc : zbase + za.tap[jz - za.nbig + 1], nz);   // output planes [z0, ze)
    const int f = max(z0 - 1, 0);              // first plane of step k
    const int uk_last = min(ze, nz - 1);       // last plane of step k (and of z^{k+1})
    const int last = min(ze + 1, nz - 1);      // last staged plane (z^k of plane ze+1)
    const float lam = za.lam, s = za.s, m0 = za.m0, m1 = za.m1;
    const float nzero = neg_zero(lam);

    if (tid == 0) {
        for (int k = 0; k <= Z2_STAGES; ++k) mbar_init(&bars[k], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();

    auto slot = [&](int q) { return (q - f) % Z2_STAGES; };
    auto stage = [&](int q) { return smem + slot(q) * Z2_STAGE_STRIDE; };
    auto parity = [&](int q) { return static_cast<uint32_t>(((q - f) / Z2_STAGES) & 1); };
    auto polls = [&](int q) { return q - f >= za.poll_from ? za.max_polls : ZM_MAX_POLLS; };
    auto issue = [&](int q) {                   // the producer thread only
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

    auto F = [](const unsigned char *st, int off) { return reinterpret_cast<const float *>(st + off); };
    auto zkp = [&](int q) { return ZK + (q & 1) * Z2_RING_ZK; };
    auto mrp = [&](int q, int a) { return MR + ((q & 1) * 2 + a) * Z2_MR_COMP; };   // a = 0 (x), 1 (y)
    auto z1p = [&](int q) { return Z1 + (q & 1) * Z2_RING_Z1; };

    // this thread's quad in the z^k / step-k grid (c = lx + 4, row = ly + 1)
    int my_c = 0, my_row = 0;
    if (tid < Z2_TASKS_D) {                                      // tile
        my_c = 4 + 4 * (tid % Z2_QD);
        my_row = 1 + tid / Z2_QD;
    } else if (tid < Z2_TASKS_D + 2 * Z2_QA) {                   // ring: rows ly = -1 and TY
        const int j = tid - Z2_TASKS_D;
        my_c = 4 * (j % Z2_QA);
        my_row = j < Z2_QA ? 0 : Z2_TY + 1;
    } else if (tid < Z2_TASKS_B) {                               // ring: quad columns 0 and QA-1
        const int j = tid - Z2_TASKS_D - 2 * Z2_QA;
        my_c = (j & 1) ? 4 * (Z2_QA - 1) : 0;
        my_row = 1 + j / 2;
    } else if (tid < Z2_TASKS_A) {                               // z^k only: row ly = TY+1
        my_c = 4 * (tid - Z2_TASKS_B);
        my_row = Z2_TY + 2;
    }
    const bool doA = tid < Z2_TASKS_A;
    const bool doB = tid < Z2_TASKS_B;
    const bool my_tile = tid < Z2_TASKS_D;
    // z^{k+1} runs on lx 0..TX, ly 0..TY: the z^k quads of columns c >= 4
    // and rows 1..TY+1 (the tile, the ring's right column and its last row)
    const bool doC = doA && my_c >= 4 && my_row >= 1 && my_row <= Z2_TY + 1;
    // Step k's quads cover lx -4..TX+3, ly -1..TY.  When all of them lie
    // inside the volume and none touches the upper x face, neither step
    // needs a per-voxel boundary test, nor a y or x face test (most CTAs of
    // a large volume): the march below is compiled twice, with and without
    // the tests, and each CTA runs one of the two.
#if TVFGP_Z2_EDGE_SPLIT
    const bool edge_cta = !(x0 >= 4 && x0 + Z2_TX + 5 <= nx && y0 >= 1 && y0 + Z2_TY + 2 <= ny);
#else
    const bool edge_cta = true;
#endif

    // z^k of plane q for this thread's quad, from the staged plane st and the
    // r2 of the plane below (lo: a staged r2 box, or nullptr at plane 0);
    // stored for the neighbours and returned, with the quad's b in Bq
    auto zk_quad = [&](int q, const unsigned char *st, const float *lo, float4 &Bq) {
        const int rr = (my_row + 1) * Z2_BW + my_c;                  // r box row of ly
        const float *R0 = F(st, Z2_OFF_R0), *R1 = F(st, Z2_OFF_R1);
        const float left = my_c > 0 ? R0[rr - 1] : 0.0f;
        const float4 r2lo = lo ? lds4(lo + rr) : f4zero();
        Bq = lds4(F(st, Z2_OFF_B) + my_row * Z2_BW + my_c);
        const float4 Z = zquad(Bq, lds4(R0 + rr), lds4(R1 + rr), lds4(F(st, Z2_OFF_R2) + rr), left,
                               lds4(R1 + rr - Z2_BW), r2lo, lam, nzero);
        *reinterpret_cast<float4 *>(zkp(q) + my_row * Z2_PK + my_c) = Z;
        return Z;
    };
    // z^{k+1} of plane q for the quad at (c = lx, ly) whose b is Bq,
    // stored and returned
    // (the quad's own r^{k+1} of plane q, R0..R2, and r_z^{k+1} of plane q-1,
    // R2lo, come from the registers of this thread, which made them in step
    // k; only the x-1 and y-1 neighbours are read from the ring)
    auto z1_quad = [&](int q, int c, int ly, float4 Bq, float4 R0, float4 R1, float4 R2, float4 R2lo) {
        const float *M0 = mrp(q, 0), *M1 = mrp(q, 1);
        const int mo = (ly + 1) * Z2_PK + c + 4;                     // r^{k+1} at (lx = c, ly)
        const float4 Z = zquad(Bq, R0, R1, R2, M0[mo - 1], lds4(M1 + mo - Z2_PK), q > 0 ? R2lo : f4zero(), lam,
                               nzero);
        *reinterpret_cast<float4 *>(z1p(q) + ly * Z2_P1 + c) = Z;
        return Z;
    };

    if (tid == Z2_PRODUCER) {
        if (f > 0) {
            mbar_expect_tx(&bars[Z2_STAGES], Z2_BYTES_R);
            tma_load_3d(smem + Z2_OFF_PREV, &za.tr2, x0 - 4, y0 - 2, f - 1, &bars[Z2_STAGES]);
        }
        for (int q = f; q <= last && q < f + Z2_STAGES; ++q) issue(q);
    }
    int next_issue = f + Z2_STAGES;

    float4 ZKc = f4zero();                      // z^k of this quad, current plane
    float4 Bc = f4zero();                       // b of this quad, current plane
    // prologue: z^k of plane f.  A wait that gives up is reported through
    // the barrier itself (its OR over the threads), so every thread takes
    // the same decision with no flag in shared memory.
    bool ok = true;
    if (f > 0) ok = mbar_wait_tma(&bars[Z2_STAGES], 0, polls(f));
    ok = ok && mbar_wait_tma(&bars[slot(f)], parity(f), polls(f));
    if (ok && doA)
        ZKc = zk_quad(f, stage(f), f > 0 ? reinterpret_cast<const float *>(smem + Z2_OFF_PREV) : nullptr, Bc);
    bool aborted = __syncthreads_or(!ok) != 0;

    const long long No = PADDED_OUT ? za.No : za.N;
    const int opx = PADDED_OUT ? za.opx : nx;
    float *p0d = za.p_dst, *p1d = za.p_dst + No, *p2d = za.p_dst + 2 * No;
    float *r0d = za.r_dst, *r1d = za.r_dst + No, *r2d = za.r_dst + 2 * No;
    float4 cP0 = f4zero(), cP1 = f4zero(), cP2 = f4zero();   // p^{k+1} of plane q-1 (tile quads)
    float4 cR0 = f4zero(), cR1 = f4zero(), cR2 = f4zero();   // r^{k+1} of plane q-1 (tile quads)
    float4 Z1c = f4zero();                                    // z^{k+1} of plane q-1 (tile quads)

    int qlast = f - 1;                          // planes <= qlast+1 were waited for
    // The march over the CTA's planes, instantiated for edge = true (every
    // boundary test) and edge = false (none; interior CTAs only).
    auto march = [&](auto edge_tag) {
        constexpr bool edge = decltype(edge_tag)::value;
        for (int q = f; q <= ze && !aborted; ++q) {
            qlast = q;
            bool failed = false;
            // ---- A: z^k of plane q+1 -------------------------------------------
            float4 ZKn = f4zero(), Bn = f4zero();
            if (q + 1 <= last) {
                if (mbar_wait_tma(&bars[slot(q + 1)], parity(q + 1), polls(q + 1))) {
                    if (doA) ZKn = zk_quad(q + 1, stage(q + 1), F(stage(q), Z2_OFF_R2), Bn);
                } else {
                    failed = true;
                }
            }
            // ---- B: step k on plane q over the grown tile ----------------------
            float4 nP0 = f4zero(), nP1 = f4zero(), nP2 = f4zero(), nR0 = f4zero(), nR1 = f4zero(), nR2 = f4zero();
            if (q <= uk_last && doB) {
                const unsigned char *st = stage(q);
                const bool hasZ = q + 1 < nz;
                const float *Zq = zkp(q);
                const int c = my_c, row = my_row;                        // row = ly + 1
                const int ly = row - 1, lx = c - 4;
                const int x = x0 + lx, y = y0 + ly;
                const int zo = row * Z2_PK + c;
                const float4 zc = ZKc;
                const float zx = c + 4 < Z2_PK ? Zq[zo + 4] : 0.0f;
                const float4 zy = lds4(Zq + zo + Z2_PK);
                const float4 zz = hasZ ? ZKn : f4zero();
                const int ro = (row + 1) * Z2_BW + c, po = row * Z2_BW + c;
                float4 R0 = lds4(F(st, Z2_OFF_R0) + ro), R1 = lds4(F(st, Z2_OFF_R1) + ro),
                       R2 = lds4(F(st, Z2_OFF_R2) + ro);
                float4 P0 = lds4(F(st, Z2_OFF_P0) + po), P1 = lds4(F(st, Z2_OFF_P1) + po),
                       P2 = lds4(F(st, Z2_OFF_P2) + po);
                const bool gy = !edge || y < ny - 1;
                float4 G0 = make_float4(__fsub_rn(zc.x, zc.y), __fsub_rn(zc.y, zc.z), __fsub_rn(zc.z, zc.w),
                                        __fsub_rn(zc.w, zx));
                const float4 G1 = gy ? sub4_rn(zc, zy) : f4zero();
                const float4 G2 = hasZ ? sub4_rn(zc, zz) : f4zero();
                if (edge) {
                    float *g0 = &G0.x;
    #pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (!(x + e < nx - 1)) g0[e] = 0.0f;
                }
                dual_update4(R0, R1, R2, G0, G1, G2, P0, P1, P2, s, m0, nzero);
                // voxels of the ring outside the volume: r^{k+1} = 0, the r(-1) = 0
                // boundary of step k+1 (their p is never used)
                if (edge) {
                    const bool yin = y >= 0 && y < ny;
                    float *r0 = &R0.x, *r1 = &R1.x, *r2 = &R2.x;
    #pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int xe = x + e;
                        if (!(yin && xe >= 0 && xe < nx)) r0[e] = r1[e] = r2[e] = 0.0f;
                    }
                }
                const int mo = row * Z2_PK + c;
                *reinterpret_cast<float4 *>(mrp(q, 0) + mo) = R0;
                *reinterpret_cast<float4 *>(mrp(q, 1) + mo) = R1;
                nP0 = P0;
                nP1 = P1;
                nP2 = P2;
                nR0 = R0;
                nR1 = R1;
                nR2 = R2;
            }
            ZKc = ZKn;
            if (__syncthreads_or(failed)) {
                aborted = true;
                break;
            }
            // every read of plane q's stage is done (phase C takes b from
            // registers): the slot takes the next plane
            if (tid == Z2_PRODUCER && next_issue <= last && q <= uk_last) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue(next_issue++);
            }

            // ---- C: z^{k+1} of plane q on the tile, its x+1 column and y+1 row ---
            // (each quad by the thread that computed z^k there, which holds its b)
            float4 Z1n = f4zero();
            if (q >= z0 && q <= uk_last && doC) {
                const float4 Z = z1_quad(q, my_c - 4, my_row - 1, Bc, nR0, nR1, nR2, cR2);
                if (my_tile) Z1n = Z;
            }
            Bc = Bn;
            // ---- D: step k+1 on plane q-1 over the tile -> p^{k+2}, r^{k+2} -----
            const int qd = q - 1;
            if (my_tile && qd >= z0 && qd < ze) {
                const int c = my_c - 4, ly = my_row - 1;
                const int x = x0 + c, y = y0 + ly;
                if (!edge || (x < nx && y < ny)) {
                    const bool hasZ = qd + 1 < nz;
                    const float *Zd = z1p(qd);
                    const int zo = ly * Z2_P1 + c;
                    const float4 zc = Z1c;
                    const float zx = Zd[zo + 4];
                    const float4 zy = lds4(Zd + zo + Z2_P1);
                    const float4 zz = hasZ ? Z1n : f4zero();
                    float4 R0 = cR0, R1 = cR1, R2 = cR2;
                    float4 P0 = cP0, P1 = cP1, P2 = cP2;
                    const bool gy = !edge || y < ny - 1;
                    const float4 G1 = gy ? sub4_rn(zc, zy) : f4zero();
                    const float4 G2 = hasZ ? sub4_rn(zc, zz) : f4zero();
                    const float gx3 = (!edge || x + 3 < nx - 1) ? __fsub_rn(zc.w, zx) : 0.0f;
                    const float4 G0 =
                        make_float4(__fsub_rn(zc.x, zc.y), __fsub_rn(zc.y, zc.z), __fsub_rn(zc.z, zc.w), gx3);
                    dual_update4(R0, R1, R2, G0, G1, G2, P0, P1, P2, s, m1, nzero);
                    const long long i = x + (long long)opx * (y + (long long)ny * qd);
                    if (!PADDED_OUT) {
                        st4(p0d + i, P0);
                        st4(p1d + i, P1);
                        st4(p2d + i, P2);
                        st4(r0d + i, R0);
                        st4(r1d + i, R1);
                        st4(r2d + i, R2);
                    } else {
                        stq<2>(p0d + i, P0);
                        stq<2>(p1d + i, P1);
                        stq<2>(p2d + i, P2);
                        stq<2>(r0d + i, R0);
                        stq<2>(r1d + i, R1);
                        stq<2>(r2d + i, R2);
                    }
                }
            }
            Z1c = Z1n;
            cP0 = nP0;
            cP1 = nP1;
            cP2 = nP2;
            cR0 = nR0;
            cR1 = nR1;
            cR2 = nR2;
        }
    };
    if (edge_cta)
        march(std::true_type{});
    else
        march(std::false_type{});

    if (aborted) {
        // A wait gave up.  Record it, then drain (bounded) every copy this
        // CTA issued that is still in flight: plane qlast+1 (whose wait
        // failed, or f when the prologue failed) and every later plane
        // issued.  The producer issued them and alone knows how many.
        __syncthreads();
        if (tid == Z2_PRODUCER) {
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

// Planes per CTA: zc for z-chunks 0..nbig-1.  CTAs start in blockIdx
// order, z-chunk last, so the last chunk's CTAs set the launch's tail.  When
// the last round of CTAs over the resident slots is less than half full (the
// GPU idles for most of a CTA's time), the last chunk is cut into shorter
// pieces (tap): 512^3 with 64-plane chunks ran 12.07 rounds, and its
// launches got 1.7% shorter; fuller last rounds lose more to the pieces'
// prologues than the tail costs.  With the tail cut, longer chunks (up to
// 128 planes, fewer prologues) pay: 512^3 now runs 6.04 rounds of 128.
struct Zmarch2Plan {
    dim3 grid;
    int zc;
    int nbig;
    int tap[4];
};

inline void zmarch2_chunks(int nz, long long tiles_xy, long long slots, Zmarch2Plan *plan)
{
    const int zc = plan->zc;
    const int chunks = (nz + zc - 1) / zc;
    const int last = nz - (chunks - 1) * zc;
    plan->nbig = chunks;
    plan->tap[0] = 0;
    plan->tap[1] = plan->tap[2] = plan->tap[3] = 0;
    const long long ctas = tiles_xy * chunks;
    const bool ragged = slots > 0 && (ctas % slots) * 2 < slots;
    int pieces = 0;
    if (!ragged) {
    } else if (TVFGP_Z2_TAPER == 1 && chunks > 1 && last >= 24) {
        const int a = (last + 1) / 2, b2 = (last - a + 1) / 2;
        plan->tap[1] = a;
        plan->tap[2] = a + b2;
        plan->tap[3] = last;
        pieces = 3;
    } else if (TVFGP_Z2_TAPER == 2 && chunks > 1 && last >= 16) {
        plan->tap[1] = (last + 1) / 2;
        plan->tap[2] = last;
        pieces = 2;
    }
    if (pieces > 0) plan->nbig = chunks - 1;
    plan->grid.z = plan->nbig + pieces;
}

inline int zmarch2_plan(int nx, int ny, int nz, Zmarch2Plan *plan)
{
    const int tx = (nx + Z2_TX - 1) / Z2_TX, ty = (ny + Z2_TY - 1) / Z2_TY;
    plan->zc = 32;
    plan->grid = dim3(tx, ty, (nz + plan->zc - 1) / plan->zc);
    zmarch2_chunks(nz, 0, 0, plan);
    if (!zmarch_supported(nx, ny, nz)) return 0;
    if (zm_encoder() == nullptr) return 3;
    const void *fn = reinterpret_cast<const void *>(&fgp_step2_zmarch_tma<false>);
    const void *fn_padded = reinterpret_cast<const void *>(&fgp_step2_zmarch_tma<true>);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, Z2_SMEM) != cudaSuccess ||
        cudaFuncSetAttribute(fn_padded, cudaFuncAttributeMaxDynamicSharedMemorySize, Z2_SMEM) != cudaSuccess) {
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
    const int slots = sms * (per_sm > 0 ? per_sm : 1);
    plan->zc = zmarch_pick_zc(tx * ty, nz, slots, TVFGP_Z2_ZC_MAX, TVFGP_Z2_WAVES);
    plan->grid = dim3(tx, ty, (nz + plan->zc - 1) / plan->zc);
    zmarch2_chunks(nz, static_cast<long long>(tx) * ty, slots, plan);
    return 0;
}

inline const void *zmarch2_kernel(bool padded_out = false)
{
    return padded_out ? reinterpret_cast<const void *>(&fgp_step2_zmarch_tma<true>)
                      : reinterpret_cast<const void *>(&fgp_step2_zmarch_tma<false>);
}
inline int zmarch2_threads() { return Z2_THREADS; }
inline size_t zmarch2_smem_bytes() { return Z2_SMEM; }

// Kernel arguments of one two-step launch (outputs dense; a caller that
// writes padded rows sets opx and No afterwards).
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
    za.nbig = plan.nbig;
    for (int k = 0; k < 4; ++k) za.tap[k] = plan.tap[k];
    za.opx = nx;
    za.No = N;
    za.max_polls = ZM_MAX_POLLS;
    za.poll_from = 0;
    return zm_encode(&za.tb, b, nx, ny, nz, Z2_BW, Z2_HB) &&
           zm_encode(&za.tr0, r_src, nx, ny, nz, Z2_BW, Z2_HR) &&
           zm_encode(&za.tr1, r_src + N, nx, ny, nz, Z2_BW, Z2_HR) &&
           zm_encode(&za.tr2, r_src + 2 * N, nx, ny, nz, Z2_BW, Z2_HR) &&
           zm_encode(&za.tp0, p_src, nx, ny, nz, Z2_BW, Z2_HP) &&
           zm_encode(&za.tp1, p_src + N, nx, ny, nz, Z2_BW, Z2_HP) &&
           zm_encode(&za.tp2, p_src + 2 * N, nx, ny, nz, Z2_BW, Z2_HP);
}

}  // namespace tvfgp
