// Kernels of the FGP step on the 3D isotropic TV dual (sm_103a).
//
// The step (page "TV solver: the FGP step on the GPU", section "What one step
// does"): z(j) = max(b(j) - lambda L(r)(j), 0) with L(r)(j) = sum_a r_a(j) -
// r_a(j - e_a); g_a = z(i) - z(i + e_a); q = r(i) + g/(12 lambda);
// p' = q / max(1, |q|); r(i) = p' + m (p' - p(i)); p(i) = p'.  Boundaries:
// r_a(-1) = 0, and g_a = 0 where i + e_a leaves the volume.
//
// Every kernel here evaluates exactly the same fp32 expressions in the same
// order (explicit __f*_rn intrinsics, so no multiply-add is ever contracted),
// which makes all variants bitwise identical to each other and to a CPU
// evaluation of the same canonical order:
//   L   = ((r0(j) - r0(j-ex)) + (r1(j) - r1(j-ey))) + (r2(j) - r2(j-ez))
//   z   = max(b - lambda*L, 0)
//   q_a = r_a + g_a*s,  s = 1/(12 lambda) rounded to float once
//   |q| = sqrt((q0*q0 + q1*q1) + q2*q2);  p'_a = q_a / max(1, |q|)
//   r_a = p'_a + m*(p'_a - p_a)
// Dividing by max(1,|q|) equals q itself when |q| <= 1, so the square root
// and the division are only issued when |q|^2 > 1 (IEEE x/1 == x); they are
// then evaluated by a shorter sequence with the same correctly rounded
// results (project_unit_ball below).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace tvfgp {

// Arguments of one FGP step.  Volumes are fp32, x fastest; dual fields are
// planar [3][N] (component a at a*N + i), stored as TS: float, or __half for
// the half-precision storage of the dual (arithmetic stays fp32: a stored
// value is widened exactly on load and rounded once, to nearest even, on
// store).
template <typename TS>
struct StepArgsT {
    const float *b;
    TS *p;
    const TS *rs;      // r read by this step
    TS *rd;            // r written by this step (distinct buffer: neighbours still read rs)
    float lam;
    float s;           // 1/(12 lambda) rounded once to float
    float m;           // momentum weight of this step
    int nx, ny, nz;
    long long N;       // elements per volume: px*ny*nz
    int px = 0;        // row pitch in elements (0: nx); only the scalar kernels take px != nx
    // packing step (fused kernel only): p' goes to po and r to rd as dense
    // volumes of No elements each, and b is copied to bo (dense)
    TS *po = nullptr;
    float *bo = nullptr;
    long long No = 0;
};
using StepArgs = StepArgsT<float>;

template <typename TS>
struct PrimalArgsT {
    const float *b;
    const TS *d;       // dual field [3][N]
    float *z;
    float lam;
    int nx, ny, nz;
    long long N;       // elements per volume: px*ny*nz
    int px = 0;        // row pitch in elements (0: nx); only the scalar kernels take px != nx
};
using PrimalArgs = PrimalArgsT<float>;

constexpr unsigned kFull = 0xffffffffu;
constexpr int kErrTimeout = 5;   // value written to the device error word

// ---------------------------------------------------------------------------
// packed fp32 pairs (sm_100 and later)
// ---------------------------------------------------------------------------
//
// One packed instruction rounds two independent lanes, each exactly as the
// scalar __fadd_rn / __fsub_rn / __fmul_rn / __fmaf_rn would (IEEE binary32,
// nearest even, subnormals kept).  A quad (x, y, z, w) of four x voxels is
// the two aligned register pairs (x, y) and (z, w) of its float4, so every
// per-voxel operation of the step that pairs voxels lane for lane runs as two
// packed instructions instead of four scalar ones, with the same bits.  Only
// the x differences inside a quad (voxel minus its x-1 neighbour) do not pair
// lane for lane; they stay scalar.

__device__ __forceinline__ float2 lo2(float4 v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 hi2(float4 v) { return make_float2(v.z, v.w); }
__device__ __forceinline__ float4 join2(float2 a, float2 b) { return make_float4(a.x, a.y, b.x, b.y); }
__device__ __forceinline__ float4 splat4(float v) { return make_float4(v, v, v, v); }

// Each packed operation is written as PTX with an explicit .rn rounding
// modifier: like the scalar __f*_rn intrinsics, such an add or multiply is
// never contracted with a neighbouring operation into a fused multiply-add.
__device__ __forceinline__ float2 add2_rn(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 pa, pb, pd;\n\t"
        "mov.b64 pa, {%2, %3};\n\t"
        "mov.b64 pb, {%4, %5};\n\t"
        "add.rn.f32x2 pd, pa, pb;\n\t"
        "mov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 sub2_rn(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 pa, pb, pd;\n\t"
        "mov.b64 pa, {%2, %3};\n\t"
        "mov.b64 pb, {%4, %5};\n\t"
        "sub.rn.f32x2 pd, pa, pb;\n\t"
        "mov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 mul2_rn(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 pa, pb, pd;\n\t"
        "mov.b64 pa, {%2, %3};\n\t"
        "mov.b64 pb, {%4, %5};\n\t"
        "mul.rn.f32x2 pd, pa, pb;\n\t"
        "mov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 fma2_rn(float2 a, float2 b, float2 c)   // a*b + c, one rounding
{
    float2 d;
    asm("{\n\t.reg .b64 pa, pb, pc, pd;\n\t"
        "mov.b64 pa, {%2, %3};\n\t"
        "mov.b64 pb, {%4, %5};\n\t"
        "mov.b64 pc, {%6, %7};\n\t"
        "fma.rn.f32x2 pd, pa, pb, pc;\n\t"
        "mov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float4 add4_rn(float4 a, float4 b)
{
    return join2(add2_rn(lo2(a), lo2(b)), add2_rn(hi2(a), hi2(b)));
}
__device__ __forceinline__ float4 sub4_rn(float4 a, float4 b)
{
    return join2(sub2_rn(lo2(a), lo2(b)), sub2_rn(hi2(a), hi2(b)));
}
__device__ __forceinline__ float4 mul4_rn(float4 a, float4 b)
{
    return join2(mul2_rn(lo2(a), lo2(b)), mul2_rn(hi2(a), hi2(b)));
}
__device__ __forceinline__ float4 fma4_rn(float4 a, float4 b, float4 c)   // a*b + c, one rounding
{
    return join2(fma2_rn(lo2(a), lo2(b), lo2(c)), fma2_rn(hi2(a), hi2(b), hi2(c)));
}
__device__ __forceinline__ float4 neg4(float4 a) { return make_float4(-a.x, -a.y, -a.z, -a.w); }

// A product that feeds a packed add or subtract.  ptxas merges a packed
// multiply whose only use is a packed add or subtract into one fused
// multiply-add, even when both are written with an explicit .rn (measured
// with nvcc 13.0 for sm_103a: a third of random products then round
// differently), which would change the step's bits.  The product is
// therefore formed as a fused multiply-add with a -0 addend,
// RN(a*b + (-0)) = RN(a*b) for every a and b, signed zeros included, which
// is not merged further.  nz must be -0 at run time, made from a kernel
// argument by neg_zero(): a -0 literal would be folded back into a multiply.
__device__ __forceinline__ float4 prod4_rn(float4 a, float4 b, float4 nz) { return fma4_rn(a, b, nz); }

// -0.0f from a kernel argument x that the host has checked to be finite and
// positive (lambda, or the step 1/(12 lambda)).
__device__ __forceinline__ float neg_zero(float x) { return __fmul_rn(-0.0f, x); }

// ---------------------------------------------------------------------------
// scalar pieces of the step (the single definition every kernel uses)
// ---------------------------------------------------------------------------

// z = max(b - lambda * ((d0 + d1) + d2), 0)
__device__ __forceinline__ float zval(float b, float lam, float d0, float d1, float d2)
{
    const float L = __fadd_rn(__fadd_rn(d0, d1), d2);
    return fmaxf(__fsub_rn(b, __fmul_rn(lam, L)), 0.0f);
}

// ---------------------------------------------------------------------------
// projection onto the unit ball, p' = q / max(1, |q|)
// ---------------------------------------------------------------------------
//
// Where |q|^2 = nn > 1 the canonical result is n = RN(sqrt(nn)) followed by
// RN(q_a / n) for each component (IEEE square root and division).  The fast
// path reaches the same bits with one hardware estimate and fused
// multiply-adds:
//   k = rsqrt.approx(nn)                          estimate of 1/sqrt(nn)
//   g = RN(nn k), e = RN(nn - g^2), n = RN(g + e k/2)
//                                                 Newton correction of sqrt
//   v = rcp.approx(n), t = RN(1 - n v), y = RN(v + t v)
//                                                 Newton correction of 1/n
//   c = RN(q y), w = RN(c n - q), d = RN(c - w y) corrected quotient
// The last line is Markstein's FMA division (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990; the FMA-based division of Muller et al., "Handbook of
// Floating-Point Arithmetic"): when y = RN(1/n) and c is within one ulp of
// q/n, w is exact and d = RN(q/n), as long as nothing under- or overflows.
// That n = RN(sqrt(nn)) and y = RN(1/n) for every float nn in [1, 2^100) is
// not a theorem about the estimates but a measured fact (a reciprocal
// corrected from k instead of from its own estimate misses 200 of them):
// tvfgp_debug_projection_check compares all of them with __fsqrt_rn and
// __frcp_rn, and compares whole projections with the IEEE ones on random
// and near-binade-edge inputs.  Range guard: the fast path runs only for
// nn < 2^100 and components that are zero or at least 2^-75 in magnitude,
// which keeps every intermediate a normal number; other inputs take the IEEE
// operations.  Forming w = c n - q (not q - c n) and d = c - w y returns a
// zero component with its sign, as the IEEE division does.

__device__ __forceinline__ float rsqrt_estimate(float x)
{
    float y;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_estimate(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// n = RN(sqrt(nn)) and y = RN(1/n), for nn in [1, 2^100).
__device__ __forceinline__ void sqrt_recip_rn(float nn, float &n, float &y)
{
    const float k = rsqrt_estimate(nn);
    const float g = __fmul_rn(nn, k);
    const float e = __fmaf_rn(-g, g, nn);
    n = __fmaf_rn(e, __fmul_rn(0.5f, k), g);
    const float v = rcp_estimate(n);
    const float t = __fmaf_rn(-n, v, 1.0f);
    y = __fmaf_rn(t, v, v);
}

// RN(q / n) given y = RN(1/n), in the range the guard admits.
__device__ __forceinline__ float div_by_recip_rn(float q, float n, float y)
{
    const float c = __fmul_rn(q, y);
    const float w = __fmaf_rn(c, n, -q);
    return __fmaf_rn(-w, y, c);
}

// A component outside the fast path's range: non-zero and below 2^-75 in
// magnitude.  (2|q| as bits) - 2 wraps to the top for q = +-0, so the key
// of a component is below kTinyLim exactly when it is tiny and non-zero.
constexpr uint32_t kTinyLim = 0x1a000000u * 2u - 2u;    // 2^-75 has the bits 0x1a000000
__device__ __forceinline__ uint32_t tiny_key(float q) { return (__float_as_uint(q) << 1) - 2u; }
__device__ __forceinline__ bool tiny_nonzero(float q) { return tiny_key(q) < kTinyLim; }

// The canonical IEEE projection (also the reference of the self-check).
__device__ __forceinline__ void project_unit_ball_ieee(float &q0, float &q1, float &q2, float nn)
{
    if (nn > 1.0f) {
        const float n = __fsqrt_rn(nn);
        q0 = __fdiv_rn(q0, n);
        q1 = __fdiv_rn(q1, n);
        q2 = __fdiv_rn(q2, n);
    }
}

__device__ __forceinline__ void project_unit_ball(float &q0, float &q1, float &q2, float nn)
{
    if (nn > 1.0f) {
        if (nn < 0x1p100f && !(tiny_nonzero(q0) | tiny_nonzero(q1) | tiny_nonzero(q2))) {
            float n, y;
            sqrt_recip_rn(nn, n, y);
            q0 = div_by_recip_rn(q0, n, y);
            q1 = div_by_recip_rn(q1, n, y);
            q2 = div_by_recip_rn(q2, n, y);
        } else {
            project_unit_ball_ieee(q0, q1, q2, nn);
        }
    }
}

// q = r + g*s, projection onto the unit ball, extrapolation.  Writes p' into
// (p0,p1,p2) and the new r into (r0,r1,r2).
__device__ __forceinline__ void dual_update(float &r0, float &r1, float &r2,
                                            float g0, float g1, float g2,
                                            float &p0, float &p1, float &p2,
                                            float s, float m)
{
    float q0 = __fadd_rn(r0, __fmul_rn(g0, s));
    float q1 = __fadd_rn(r1, __fmul_rn(g1, s));
    float q2 = __fadd_rn(r2, __fmul_rn(g2, s));
    const float nn = __fadd_rn(__fadd_rn(__fmul_rn(q0, q0), __fmul_rn(q1, q1)), __fmul_rn(q2, q2));
    // max(1, |q|) > 1 exactly when |q|^2 > 1 (a correctly rounded square root
    // is monotone and sqrt(1) = 1); where |q|^2 > 1 but |q| rounds to 1, the
    // division by 1 leaves q unchanged, as the definition does.
    project_unit_ball(q0, q1, q2, nn);
    r0 = __fadd_rn(q0, __fmul_rn(m, __fsub_rn(q0, p0)));
    r1 = __fadd_rn(q1, __fmul_rn(m, __fsub_rn(q1, p1)));
    r2 = __fadd_rn(q2, __fmul_rn(m, __fsub_rn(q2, p2)));
    p0 = q0;
    p1 = q1;
    p2 = q2;
}

// RN(q / n) for the four voxels of a quad, given Y = RN(1/n) (packed form of
// div_by_recip_rn, the same three roundings per lane).
__device__ __forceinline__ float4 div4_by_recip_rn(float4 Q, float4 N, float4 Y)
{
    const float4 C = mul4_rn(Q, Y);
    const float4 W = fma4_rn(C, N, neg4(Q));
    return fma4_rn(neg4(W), Y, C);
}

// dual_update on the four voxels of a quad (component a of the quad in Ra,
// Ga, Pa): the same operations per voxel, as packed pairs where the lanes
// pair up.  q and |q|^2 of all four first; one branch to the projection when
// any of the four needs it, one to the IEEE operations when any value of the
// quad lies outside the fast path's range; then the four extrapolations.
// The fast path divides every voxel by RN(sqrt(max(1, |q|^2))): the voxels
// with |q|^2 <= 1 get n = RN(sqrt(1)) = 1 and y = 1 (checked on the GPU with
// the other square roots), and c = q*1, w = c*1 - q = +0, d = c - 0*1 return
// their q unchanged, signed zeros and subnormals included.  nzero: -0 at run
// time (neg_zero).
__device__ __forceinline__ void dual_update4(float4 &R0, float4 &R1, float4 &R2, float4 G0, float4 G1,
                                             float4 G2, float4 &P0, float4 &P1, float4 &P2, float s,
                                             float m, float nzero)
{
    const float4 S = splat4(s), NZ = splat4(nzero);
    float4 Q0 = add4_rn(R0, prod4_rn(G0, S, NZ));
    float4 Q1 = add4_rn(R1, prod4_rn(G1, S, NZ));
    float4 Q2 = add4_rn(R2, prod4_rn(G2, S, NZ));
    const float4 NN = add4_rn(add4_rn(prod4_rn(Q0, Q0, NZ), prod4_rn(Q1, Q1, NZ)), prod4_rn(Q2, Q2, NZ));
    const float4 NC = make_float4(fmaxf(NN.x, 1.0f), fmaxf(NN.y, 1.0f), fmaxf(NN.z, 1.0f), fmaxf(NN.w, 1.0f));
    if (fmaxf(fmaxf(NC.x, NC.y), fmaxf(NC.z, NC.w)) > 1.0f) {
        // The fast path's range for the whole quad: the rounded sum of the
        // four |q|^2 (none of which exceeds it; NaN if one is NaN) below
        // 2^100, and every component zero or at least 2^-75.
        const float2 half = add2_rn(lo2(NN), hi2(NN));
        const float sum = __fadd_rn(half.x, half.y);
        uint32_t key = min(min(tiny_key(Q0.x), tiny_key(Q0.y)), min(tiny_key(Q0.z), tiny_key(Q0.w)));
        key = min(key, min(min(tiny_key(Q1.x), tiny_key(Q1.y)), min(tiny_key(Q1.z), tiny_key(Q1.w))));
        key = min(key, min(min(tiny_key(Q2.x), tiny_key(Q2.y)), min(tiny_key(Q2.z), tiny_key(Q2.w))));
        if (sum < 0x1p100f && key >= kTinyLim) {
            // sqrt_recip_rn on the four voxels, packed where the lanes pair up
            const float4 K = make_float4(rsqrt_estimate(NC.x), rsqrt_estimate(NC.y), rsqrt_estimate(NC.z),
                                         rsqrt_estimate(NC.w));
            const float4 Gq = mul4_rn(NC, K);
            const float4 E = fma4_rn(neg4(Gq), Gq, NC);
            const float4 N = fma4_rn(E, mul4_rn(splat4(0.5f), K), Gq);
            const float4 V = make_float4(rcp_estimate(N.x), rcp_estimate(N.y), rcp_estimate(N.z),
                                         rcp_estimate(N.w));
            const float4 T = fma4_rn(neg4(N), V, splat4(1.0f));
            const float4 Y = fma4_rn(T, V, V);
            Q0 = div4_by_recip_rn(Q0, N, Y);
            Q1 = div4_by_recip_rn(Q1, N, Y);
            Q2 = div4_by_recip_rn(Q2, N, Y);
        } else {
            project_unit_ball(Q0.x, Q1.x, Q2.x, NN.x);
            project_unit_ball(Q0.y, Q1.y, Q2.y, NN.y);
            project_unit_ball(Q0.z, Q1.z, Q2.z, NN.z);
            project_unit_ball(Q0.w, Q1.w, Q2.w, NN.w);
        }
    }
    const float4 M = splat4(m);
    R0 = add4_rn(Q0, prod4_rn(M, sub4_rn(Q0, P0), NZ));
    R1 = add4_rn(Q1, prod4_rn(M, sub4_rn(Q1, P1), NZ));
    R2 = add4_rn(Q2, prod4_rn(M, sub4_rn(Q2, P2), NZ));
    P0 = Q0;
    P1 = Q1;
    P2 = Q2;
}

// ---------------------------------------------------------------------------
// memory helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ float4 ld_ro4(const float *p)      // read-only for the kernel
{
    return __ldg(reinterpret_cast<const float4 *>(p));
}
__device__ __forceinline__ float4 ld_once4(const float *p)    // read once, then overwritten
{
    return __ldcs(reinterpret_cast<const float4 *>(p));
}
__device__ __forceinline__ void st4(float *p, float4 v)
{
    *reinterpret_cast<float4 *>(p) = v;
}
__device__ __forceinline__ float4 f4zero()
{
    return make_float4(0.f, 0.f, 0.f, 0.f);
}
__device__ __forceinline__ float2 ld_ro2(const float *p) { return __ldg(reinterpret_cast<const float2 *>(p)); }
__device__ __forceinline__ float2 ld_once2(const float *p) { return __ldcs(reinterpret_cast<const float2 *>(p)); }
__device__ __forceinline__ void st2(float *p, float2 v) { *reinterpret_cast<float2 *>(p) = v; }
__device__ __forceinline__ float2 f2zero() { return make_float2(0.f, 0.f); }

// A quad of four x values moved as one 16-byte access (VW = 4) or as two
// 8-byte halves (VW = 2: rows padded to a pitch that is even but not a
// multiple of four, where a quad is only 8-byte aligned).
template <int VW>
__device__ __forceinline__ float4 ldq_ro(const float *p)
{
    if (VW == 4) return ld_ro4(p);
    const float2 a = ld_ro2(p), b = ld_ro2(p + 2);
    return make_float4(a.x, a.y, b.x, b.y);
}
template <int VW>
__device__ __forceinline__ float4 ldq_once(const float *p)
{
    if (VW == 4) return ld_once4(p);
    const float2 a = ld_once2(p), b = ld_once2(p + 2);
    return make_float4(a.x, a.y, b.x, b.y);
}
template <int VW>
__device__ __forceinline__ void stq(float *p, float4 v)
{
    if (VW == 4) {
        st4(p, v);
    } else {
        st2(p, make_float2(v.x, v.y));
        st2(p + 2, make_float2(v.z, v.w));
    }
}


// Four consecutive values of a dual component, widened to float4, and back.
__device__ __forceinline__ float4 ldv_ro(const float *p) { return ld_ro4(p); }
__device__ __forceinline__ float4 ldv_once(const float *p) { return ld_once4(p); }
__device__ __forceinline__ void stv(float *p, float4 v) { st4(p, v); }
__device__ __forceinline__ float ld1_ro(const float *p) { return __ldg(p); }
__device__ __forceinline__ float ld1_once(const float *p) { return __ldcs(p); }
__device__ __forceinline__ void st1(float *p, float v) { *p = v; }

__device__ __forceinline__ float4 widen4(uint2 u)
{
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ float4 ldv_ro(const __half *p) { return widen4(__ldg(reinterpret_cast<const uint2 *>(p))); }
__device__ __forceinline__ float4 ldv_once(const __half *p) { return widen4(__ldcs(reinterpret_cast<const uint2 *>(p))); }
__device__ __forceinline__ void stv(__half *p, float4 v)
{
    const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<const unsigned *>(&a);
    u.y = *reinterpret_cast<const unsigned *>(&b);
    *reinterpret_cast<uint2 *>(p) = u;
}
__device__ __forceinline__ float ld1_ro(const __half *p) { return __half2float(__ldg(p)); }
__device__ __forceinline__ float ld1_once(const __half *p) { return __half2float(__ldcs(p)); }
__device__ __forceinline__ void st1(__half *p, float v) { *p = __float2half_rn(v); }

// Dual quads by storage type: binary16 quads are 8 bytes and keep VW = 4.
template <int VW> __device__ __forceinline__ float4 ldvq_ro(const float *p) { return ldq_ro<VW>(p); }
template <int VW> __device__ __forceinline__ float4 ldvq_once(const float *p) { return ldq_once<VW>(p); }
template <int VW> __device__ __forceinline__ void stvq(float *p, float4 v) { stq<VW>(p, v); }
template <int VW> __device__ __forceinline__ float4 ldvq_ro(const __half *p)
{
    static_assert(VW == 4, "binary16 quads are moved whole");
    return ldv_ro(p);
}
template <int VW> __device__ __forceinline__ float4 ldvq_once(const __half *p)
{
    static_assert(VW == 4, "binary16 quads are moved whole");
    return ldv_once(p);
}
template <int VW> __device__ __forceinline__ void stvq(__half *p, float4 v)
{
    static_assert(VW == 4, "binary16 quads are moved whole");
    stv(p, v);
}


// z at four consecutive x voxels from their b and r, the r0 of the voxel left
// of the first one, and r1, r2 of the lower neighbours in y and z (nzero: -0
// at run time, neg_zero(lam)).
__device__ __forceinline__ float4 zquad(float4 B, float4 R0, float4 R1, float4 R2, float r0left,
                                        float4 R1lo, float4 R2lo, float lam, float nzero)
{
    // zval on each voxel: the x differences pair a voxel with its left
    // neighbour (scalar); the rest runs as packed pairs, in the same order
    const float4 D0 = make_float4(__fsub_rn(R0.x, r0left), __fsub_rn(R0.y, R0.x), __fsub_rn(R0.z, R0.y),
                                  __fsub_rn(R0.w, R0.z));
    const float4 L = add4_rn(add4_rn(D0, sub4_rn(R1, R1lo)), sub4_rn(R2, R2lo));
    const float4 t = sub4_rn(B, prod4_rn(splat4(lam), L, splat4(nzero)));
    return make_float4(fmaxf(t.x, 0.0f), fmaxf(t.y, 0.0f), fmaxf(t.z, 0.0f), fmaxf(t.w, 0.0f));
}

// ---------------------------------------------------------------------------
// FUSED: one kernel per step, float4 along x, z carried along z in registers
// ---------------------------------------------------------------------------
//
// Block (32, BY): a warp is 32 consecutive x-quads (128 voxels) of one row
// (y, z); the block stacks BY rows in y.  Each thread walks ZC planes in z.
// At plane z it needs z(i), z(i+ex), z(i+ey), z(i+ez) for its 4 voxels:
//   z(i)     was computed at the previous plane as that plane's z(i+ez);
//   z(i+ex)  is the neighbour lane's z(i) (shuffle; lane 31 computes it);
//   z(i+ey)  is recomputed from row y+1 (whose r1 lower neighbour is the
//            thread's own r1, and whose r2 lower neighbour was loaded at the
//            previous plane);
//   z(i+ez)  is recomputed from the next plane's own data, which is the
//            prefetch of the next iteration.
// The voxel's own p loads are issued first in every iteration, then the
// next plane's own b and r, then row y+1: no barrier exists in this kernel.
// Requirements: nx % 4 == 0 and 16-byte aligned b, p, rs, rd.
// With PACK, the step reads padded rows (pitch px, 8-byte halves of quads)
// and writes p', r and a copy of b as dense volumes (16-byte stores), so the
// first step of a run on the real-to-complex FFT layout also packs it.
#ifndef TVFGP_FUSED_MINB
#define TVFGP_FUSED_MINB 5
#endif
// IT: the voxel index type, int unless px*ny*(nz+1) exceeds its range (the
// 64-bit instance runs one block per SM fewer, so that it does not spill).
template <int BY, int ZC, typename TS = float, int VW = 4, bool PACK = false, typename IT = int>
__global__ void __launch_bounds__(32 * BY, sizeof(IT) == 4 ? TVFGP_FUSED_MINB : TVFGP_FUSED_MINB - 1)
fgp_step_fused4(const StepArgsT<TS> a)
{
    static_assert(!PACK || (VW == 2 && sizeof(TS) == 4), "packing reads padded fp32 rows");
    const int lane = threadIdx.x;
    const int x0 = (blockIdx.x * 32 + lane) * 4;
    const int y = blockIdx.y * BY + threadIdx.y;
    const int nx = a.nx, ny = a.ny, nz = a.nz;
    const int px = a.px > 0 ? a.px : nx;         // row pitch
    if (y >= ny) return;                         // whole warp: y is warp-uniform
    const int zb = blockIdx.z * ZC;
    const int ze = min(zb + ZC, nz);
    const bool xin = x0 < nx;
    const bool hasY = (y + 1 < ny);              // warp-uniform
    const int sz = px * ny;
    const float lam = a.lam, s = a.s, m = a.m;
    const float nzero = neg_zero(lam);

    const float *__restrict__ b = a.b;
    const TS *__restrict__ r0 = a.rs;
    const TS *__restrict__ r1 = a.rs + a.N;
    const TS *__restrict__ r2 = a.rs + 2 * a.N;
    TS *__restrict__ p0 = a.p;
    TS *__restrict__ p1 = a.p + a.N;
    TS *__restrict__ p2 = a.p + 2 * a.N;
    // outputs: in place (p) and at the input's layout (r), or dense when packing
    const long long No = PACK ? a.No : a.N;
    TS *__restrict__ q0 = PACK ? a.po : a.p;
    TS *__restrict__ q1 = q0 + No;
    TS *__restrict__ q2 = q0 + 2 * No;
    TS *__restrict__ o0 = a.rd;
    TS *__restrict__ o1 = a.rd + No;
    TS *__restrict__ o2 = a.rd + 2 * No;
    constexpr int VO = PACK ? 4 : VW;            // store width
    const int szo = PACK ? nx * ny : px * ny;

    int z = zb;
    IT i = x0 + (IT)px * (y + (IT)ny * z);
    IT io = PACK ? x0 + (IT)nx * (y + (IT)ny * z) : i;

    // prologue: own r at plane zb and z(i) there
    float4 R0c = f4zero(), R1c = f4zero(), R2c = f4zero(), Zc;
    {
        float4 Bc = f4zero(), R1lo = f4zero(), R2lo = f4zero();
        if (xin) {
            Bc = ldq_ro<VW>(b + i);
            R0c = ldvq_ro<VW>(r0 + i);
            R1c = ldvq_ro<VW>(r1 + i);
            R2c = ldvq_ro<VW>(r2 + i);
            if (y > 0) R1lo = ldvq_ro<VW>(r1 + i - px);
            if (z > 0) R2lo = ldvq_ro<VW>(r2 + i - sz);
        }
        float left = __shfl_up_sync(kFull, R0c.w, 1);
        if (lane == 0) left = (x0 > 0) ? ld1_ro(r0 + i - 1) : 0.0f;
        Zc = zquad(Bc, R0c, R1c, R2c, left, R1lo, R2lo, lam, nzero);
        if (PACK && xin) stq<4>(a.bo + io, Bc);
    }
    // r2 of row y+1 one plane below (the z-lower neighbour of z(i+ey))
    float4 R2yp = f4zero();
    if (xin && hasY && z > 0) R2yp = ldvq_ro<VW>(r2 + i + px - sz);

    for (; z < ze; ++z, i += sz, io += szo) {
        const bool hasZ = (z + 1 < nz);          // block-uniform

        // (1) the voxel's own p, first
        float4 P0 = f4zero(), P1 = f4zero(), P2 = f4zero();
        if (xin) {
            P0 = ldvq_once<VW>(p0 + i);
            P1 = ldvq_once<VW>(p1 + i);
            P2 = ldvq_once<VW>(p2 + i);
        }
        // (2) the next plane's own b, r (and r1 of its y-lower row)
        float4 Bn = f4zero(), R0n = f4zero(), R1n = f4zero(), R2n = f4zero(), R1lon = f4zero();
        if (xin && hasZ) {
            Bn = ldq_ro<VW>(b + i + sz);
            R0n = ldvq_ro<VW>(r0 + i + sz);
            R1n = ldvq_ro<VW>(r1 + i + sz);
            R2n = ldvq_ro<VW>(r2 + i + sz);
            if (y > 0) R1lon = ldvq_ro<VW>(r1 + i + sz - px);
        }
        // (3) row y+1 of this plane
        float4 By = f4zero(), R0y = f4zero(), R1y = f4zero(), R2y = f4zero();
        if (xin && hasY) {
            By = ldq_ro<VW>(b + i + px);
            R0y = ldvq_ro<VW>(r0 + i + px);
            R1y = ldvq_ro<VW>(r1 + i + px);
            R2y = ldvq_ro<VW>(r2 + i + px);
        }

        // z(i+ey)
        float4 ZY = f4zero();
        if (hasY) {
            float left = __shfl_up_sync(kFull, R0y.w, 1);
            if (lane == 0) left = (x0 > 0) ? ld1_ro(r0 + i + px - 1) : 0.0f;
            ZY = zquad(By, R0y, R1y, R2y, left, R1c, R2yp, lam, nzero);
        }
        // z(i+ez)
        float4 ZZ = f4zero();
        if (hasZ) {
            float left = __shfl_up_sync(kFull, R0n.w, 1);
            if (lane == 0) left = (x0 > 0) ? ld1_ro(r0 + i + sz - 1) : 0.0f;
            ZZ = zquad(Bn, R0n, R1n, R2n, left, R1lon, R2c, lam, nzero);
        }
        // z(i+ex) of the last voxel: the next lane's first z
        float zx = __shfl_down_sync(kFull, Zc.x, 1);
        if (lane == 31 && x0 + 4 < nx) {
            const IT j = i + 4;
            const float d0 = __fsub_rn(ld1_ro(r0 + j), R0c.w);
            const float d1 = __fsub_rn(ld1_ro(r1 + j), y > 0 ? ld1_ro(r1 + j - px) : 0.0f);
            const float d2 = __fsub_rn(ld1_ro(r2 + j), z > 0 ? ld1_ro(r2 + j - sz) : 0.0f);
            zx = zval(__ldg(b + j), lam, d0, d1, d2);
        }

        if (xin) {
            const float gx3 = (x0 + 3 < nx - 1) ? __fsub_rn(Zc.w, zx) : 0.0f;
            float4 G1 = f4zero(), G2 = f4zero();
            if (hasY) {
                G1.x = __fsub_rn(Zc.x, ZY.x); G1.y = __fsub_rn(Zc.y, ZY.y);
                G1.z = __fsub_rn(Zc.z, ZY.z); G1.w = __fsub_rn(Zc.w, ZY.w);
            }
            if (hasZ) {
                G2.x = __fsub_rn(Zc.x, ZZ.x); G2.y = __fsub_rn(Zc.y, ZZ.y);
                G2.z = __fsub_rn(Zc.z, ZZ.z); G2.w = __fsub_rn(Zc.w, ZZ.w);
            }
            float4 N0 = R0c, N1 = R1c, N2 = R2c;
            const float4 G0 = make_float4(__fsub_rn(Zc.x, Zc.y), __fsub_rn(Zc.y, Zc.z), __fsub_rn(Zc.z, Zc.w), gx3);
            dual_update4(N0, N1, N2, G0, G1, G2, P0, P1, P2, s, m, nzero);
            stvq<VO>(q0 + io, P0);
            stvq<VO>(q1 + io, P1);
            stvq<VO>(q2 + io, P2);
            stvq<VO>(o0 + io, N0);
            stvq<VO>(o1 + io, N1);
            stvq<VO>(o2 + io, N2);
            if (PACK && z + 1 < ze) stq<4>(a.bo + io + szo, Bn);
        }

        R0c = R0n;
        R1c = R1n;
        R2c = R2n;
        Zc = ZZ;
        R2yp = R2y;
    }
}

// ---------------------------------------------------------------------------
// FUSED2: the fused kernel's plan on pairs of x voxels (float2), for volumes
// whose rows are padded to an even pitch that is not a multiple of four
// floats (the in-place real-to-complex FFT layout: rows of nx+2 floats)
// ---------------------------------------------------------------------------
//
// A warp is 32 consecutive x-pairs (64 voxels) of one row; z(i+ex) of the
// pair's second voxel is the next lane's first z (lane 31 computes it);
// z(i+ey) and z(i+ez) are recomputed from row y+1 and from the next plane,
// whose own data is the prefetch of the next iteration.  Requirements: nx
// and the pitch even, every pointer 8-byte aligned.

// z of a pair of x voxels, in the canonical order
__device__ __forceinline__ float2 zpair(float2 B, float2 R0, float2 R1, float2 R2, float r0left, float2 R1lo,
                                        float2 R2lo, float lam)
{
    float2 z;
    z.x = zval(B.x, lam, __fsub_rn(R0.x, r0left), __fsub_rn(R1.x, R1lo.x), __fsub_rn(R2.x, R2lo.x));
    z.y = zval(B.y, lam, __fsub_rn(R0.y, R0.x), __fsub_rn(R1.y, R1lo.y), __fsub_rn(R2.y, R2lo.y));
    return z;
}

template <int BY, int ZC>
__global__ void __launch_bounds__(32 * BY) fgp_step_fused2(const StepArgs a)
{
    const int lane = threadIdx.x;
    const int x0 = (blockIdx.x * 32 + lane) * 2;
    const int y = blockIdx.y * BY + threadIdx.y;
    const int nx = a.nx, ny = a.ny, nz = a.nz;
    const int px = a.px > 0 ? a.px : nx;         // row pitch
    if (y >= ny) return;                         // whole warp: y is warp-uniform
    const int zb = blockIdx.z * ZC;
    const int ze = min(zb + ZC, nz);
    const bool xin = x0 < nx;
    const bool hasY = (y + 1 < ny);
    const long long sz = (long long)px * ny;
    const float lam = a.lam, s = a.s, m = a.m;

    const float *__restrict__ b = a.b;
    const float *__restrict__ r0 = a.rs;
    const float *__restrict__ r1 = a.rs + a.N;
    const float *__restrict__ r2 = a.rs + 2 * a.N;
    float *__restrict__ p0 = a.p;
    float *__restrict__ p1 = a.p + a.N;
    float *__restrict__ p2 = a.p + 2 * a.N;
    float *__restrict__ o0 = a.rd;
    float *__restrict__ o1 = a.rd + a.N;
    float *__restrict__ o2 = a.rd + 2 * a.N;

    int z = zb;
    long long i = x0 + (long long)px * y + sz * z;

    // prologue: own r at plane zb and z(i) there
    float2 R0c = f2zero(), R1c = f2zero(), R2c = f2zero(), Zc;
    {
        float2 Bc = f2zero(), R1lo = f2zero(), R2lo = f2zero();
        if (xin) {
            Bc = ld_ro2(b + i);
            R0c = ld_ro2(r0 + i);
            R1c = ld_ro2(r1 + i);
            R2c = ld_ro2(r2 + i);
            if (y > 0) R1lo = ld_ro2(r1 + i - px);
            if (z > 0) R2lo = ld_ro2(r2 + i - sz);
        }
        float left = __shfl_up_sync(kFull, R0c.y, 1);
        if (lane == 0) left = (x0 > 0) ? __ldg(r0 + i - 1) : 0.0f;
        Zc = zpair(Bc, R0c, R1c, R2c, left, R1lo, R2lo, lam);
    }
    float2 R2yp = f2zero();                      // r2 of row y+1 one plane below
    if (xin && hasY && z > 0) R2yp = ld_ro2(r2 + i + px - sz);

    for (; z < ze; ++z, i += sz) {
        const bool hasZ = (z + 1 < nz);
        // the voxel's own p, first
        float2 P0 = f2zero(), P1 = f2zero(), P2 = f2zero();
        if (xin) {
            P0 = ld_once2(p0 + i);
            P1 = ld_once2(p1 + i);
            P2 = ld_once2(p2 + i);
        }
        // the next plane's own b, r (and r1 of its y-lower row)
        float2 Bn = f2zero(), R0n = f2zero(), R1n = f2zero(), R2n = f2zero(), R1lon = f2zero();
        if (xin && hasZ) {
            Bn = ld_ro2(b + i + sz);
            R0n = ld_ro2(r0 + i + sz);
            R1n = ld_ro2(r1 + i + sz);
            R2n = ld_ro2(r2 + i + sz);
            if (y > 0) R1lon = ld_ro2(r1 + i + sz - px);
        }
        // row y+1 of this plane
        float2 By = f2zero(), R0y = f2zero(), R1y = f2zero(), R2y = f2zero();
        if (xin && hasY) {
            By = ld_ro2(b + i + px);
            R0y = ld_ro2(r0 + i + px);
            R1y = ld_ro2(r1 + i + px);
            R2y = ld_ro2(r2 + i + px);
        }
        float2 ZY = f2zero();
        if (hasY) {
            float left = __shfl_up_sync(kFull, R0y.y, 1);
            if (lane == 0) left = (x0 > 0) ? __ldg(r0 + i + px - 1) : 0.0f;
            ZY = zpair(By, R0y, R1y, R2y, left, R1c, R2yp, lam);
        }
        float2 ZZ = f2zero();
        if (hasZ) {
            float left = __shfl_up_sync(kFull, R0n.y, 1);
            if (lane == 0) left = (x0 > 0) ? __ldg(r0 + i + sz - 1) : 0.0f;
            ZZ = zpair(Bn, R0n, R1n, R2n, left, R1lon, R2c, lam);
        }
        // z(i+ex) of the second voxel: the next lane's first z
        float zx = __shfl_down_sync(kFull, Zc.x, 1);
        if (lane == 31 && x0 + 2 < nx) {
            const long long j = i + 2;
            const float d0 = __fsub_rn(__ldg(r0 + j), R0c.y);
            const float d1 = __fsub_rn(__ldg(r1 + j), y > 0 ? __ldg(r1 + j - px) : 0.0f);
            const float d2 = __fsub_rn(__ldg(r2 + j), z > 0 ? __ldg(r2 + j - sz) : 0.0f);
            zx = zval(__ldg(b + j), lam, d0, d1, d2);
        }
        if (xin) {
            const float gx1 = (x0 + 1 < nx - 1) ? __fsub_rn(Zc.y, zx) : 0.0f;
            const float g1x = hasY ? __fsub_rn(Zc.x, ZY.x) : 0.0f, g1y = hasY ? __fsub_rn(Zc.y, ZY.y) : 0.0f;
            const float g2x = hasZ ? __fsub_rn(Zc.x, ZZ.x) : 0.0f, g2y = hasZ ? __fsub_rn(Zc.y, ZZ.y) : 0.0f;
            float2 N0 = R0c, N1 = R1c, N2 = R2c;
            dual_update(N0.x, N1.x, N2.x, __fsub_rn(Zc.x, Zc.y), g1x, g2x, P0.x, P1.x, P2.x, s, m);
            dual_update(N0.y, N1.y, N2.y, gx1, g1y, g2y, P0.y, P1.y, P2.y, s, m);
            st2(p0 + i, P0);
            st2(p1 + i, P1);
            st2(p2 + i, P2);
            st2(o0 + i, N0);
            st2(o1 + i, N1);
            st2(o2 + i, N2);
        }
        R0c = R0n;
        R1c = R1n;
        R2c = R2n;
        Zc = ZZ;
        R2yp = R2y;
    }
}

// ---------------------------------------------------------------------------
// rows between a padded and a dense layout
// ---------------------------------------------------------------------------
//
// One block per row: copies the row's nx floats (nx % 4 == 0) from src, row
// pitch spitch, to dst, row pitch dpitch, as 8-byte halves of quads (both
// pitches even, both buffers 8-byte aligned); x >= nx is never touched.
__global__ void __launch_bounds__(128) repack_rows(float *__restrict__ dst, int dpitch,
                                                   const float *__restrict__ src, int spitch, int nx)
{
    const long long row = blockIdx.x;
    const float *s = src + row * spitch;
    float *d = dst + row * dpitch;
    for (int x = 4 * threadIdx.x; x < nx; x += 4 * blockDim.x) {
        const float2 lo = __ldcs(reinterpret_cast<const float2 *>(s + x));
        const float2 hi = __ldcs(reinterpret_cast<const float2 *>(s + x + 2));
        st2(d + x, lo);
        st2(d + x + 2, hi);
    }
}

// ---------------------------------------------------------------------------
// SCALAR: one voxel per thread, any shape and alignment
// ---------------------------------------------------------------------------

template <typename TS>
__device__ __forceinline__ float zpoint(const float *__restrict__ b, const TS *__restrict__ r0,
                                        const TS *__restrict__ r1, const TS *__restrict__ r2,
                                        int x, int y, int z, long long j, int px, long long sz,
                                        float lam)
{
    const float d0 = __fsub_rn(ld1_ro(r0 + j), x > 0 ? ld1_ro(r0 + j - 1) : 0.0f);
    const float d1 = __fsub_rn(ld1_ro(r1 + j), y > 0 ? ld1_ro(r1 + j - px) : 0.0f);
    const float d2 = __fsub_rn(ld1_ro(r2 + j), z > 0 ? ld1_ro(r2 + j - sz) : 0.0f);
    return zval(__ldg(b + j), lam, d0, d1, d2);
}

template <typename TS = float>
__global__ void __launch_bounds__(256) fgp_step_scalar(const StepArgsT<TS> a)
{
    const int x = blockIdx.x * 32 + threadIdx.x;
    const int y = blockIdx.y * 8 + threadIdx.y;
    const int z = blockIdx.z;
    const int nx = a.nx, ny = a.ny, nz = a.nz;
    const int px = a.px > 0 ? a.px : nx;             // row pitch
    if (x >= nx || y >= ny) return;
    const long long sz = (long long)px * ny;
    const long long i = x + (long long)px * y + sz * z;
    const TS *r0 = a.rs, *r1 = a.rs + a.N, *r2 = a.rs + 2 * a.N;

    // the voxel's own p and r first
    float P0 = ld1_once(a.p + i), P1 = ld1_once(a.p + a.N + i), P2 = ld1_once(a.p + 2 * a.N + i);
    float R0 = ld1_ro(r0 + i), R1 = ld1_ro(r1 + i), R2 = ld1_ro(r2 + i);

    const float zc = zpoint(a.b, r0, r1, r2, x, y, z, i, px, sz, a.lam);
    const float g0 = (x < nx - 1) ? __fsub_rn(zc, zpoint(a.b, r0, r1, r2, x + 1, y, z, i + 1, px, sz, a.lam)) : 0.0f;
    const float g1 = (y < ny - 1) ? __fsub_rn(zc, zpoint(a.b, r0, r1, r2, x, y + 1, z, i + px, px, sz, a.lam)) : 0.0f;
    const float g2 = (z < nz - 1) ? __fsub_rn(zc, zpoint(a.b, r0, r1, r2, x, y, z + 1, i + sz, px, sz, a.lam)) : 0.0f;
    dual_update(R0, R1, R2, g0, g1, g2, P0, P1, P2, a.s, a.m);
    st1(a.p + i, P0);
    st1(a.p + a.N + i, P1);
    st1(a.p + 2 * a.N + i, P2);
    st1(a.rd + i, R0);
    st1(a.rd + a.N + i, R1);
    st1(a.rd + 2 * a.N + i, R2);
}

// ---------------------------------------------------------------------------
// primal z = max(b - lambda L(dual), 0)
// ---------------------------------------------------------------------------

template <int BY, typename TS = float>
__global__ void __launch_bounds__(32 * BY) primal_vec4(const PrimalArgsT<TS> a)
{
    const int lane = threadIdx.x;
    const int x0 = (blockIdx.x * 32 + lane) * 4;
    const int y = blockIdx.y * BY + threadIdx.y;
    const int z = blockIdx.z;
    const int nx = a.nx, ny = a.ny;
    if (y >= ny) return;
    const bool xin = x0 < nx;
    const int sz = nx * ny;
    const long long i = x0 + (long long)nx * (y + (long long)ny * z);
    const TS *d0 = a.d, *d1 = a.d + a.N, *d2 = a.d + 2 * a.N;
    float4 B = f4zero(), D0 = f4zero(), D1 = f4zero(), D2 = f4zero(), D1lo = f4zero(), D2lo = f4zero();
    if (xin) {
        B = ld_ro4(a.b + i);
        D0 = ldv_ro(d0 + i);
        D1 = ldv_ro(d1 + i);
        D2 = ldv_ro(d2 + i);
        if (y > 0) D1lo = ldv_ro(d1 + i - nx);
        if (z > 0) D2lo = ldv_ro(d2 + i - sz);
    }
    float left = __shfl_up_sync(kFull, D0.w, 1);
    if (lane == 0) left = (x0 > 0) ? ld1_ro(d0 + i - 1) : 0.0f;
    const float4 Z = zquad(B, D0, D1, D2, left, D1lo, D2lo, a.lam, neg_zero(a.lam));
    if (xin) st4(a.z + i, Z);
}

template <typename TS = float>
__global__ void __launch_bounds__(256) primal_scalar(const PrimalArgsT<TS> a)
{
    const int x = blockIdx.x * 32 + threadIdx.x;
    const int y = blockIdx.y * 8 + threadIdx.y;
    const int z = blockIdx.z;
    const int nx = a.nx, ny = a.ny;
    const int px = a.px > 0 ? a.px : nx;             // row pitch
    if (x >= nx || y >= ny) return;
    const long long sz = (long long)px * ny;
    const long long i = x + (long long)px * y + sz * z;
    a.z[i] = zpoint(a.b, a.d, a.d + a.N, a.d + 2 * a.N, x, y, z, i, px, sz, a.lam);
}

// ---------------------------------------------------------------------------
// SEPARATE: the step as two kernels, z written by one and read by the next
// (page "TV solver: the FGP step on the GPU", section "Variants", first row:
// 18 volumes per step).  The first kernel is primal_vec4 / primal_scalar on
// r_src; this one reads z at the voxel and at its +x, +y, +z neighbours.
// ---------------------------------------------------------------------------

struct DualArgs {
    const float *z;    // primal of r_src, [N]
    float *p;
    const float *rs;
    float *rd;
    float s, m;
    int nx, ny, nz;
    long long N;       // elements per volume: px*ny*nz
    int px = 0;        // row pitch in elements (0: nx); only the scalar kernel takes px != nx
};

template <int BY>
__global__ void __launch_bounds__(32 * BY) dual_from_z_vec4(const DualArgs a)
{
    const int lane = threadIdx.x;
    const int x0 = (blockIdx.x * 32 + lane) * 4;
    const int y = blockIdx.y * BY + threadIdx.y;
    const int z = blockIdx.z;
    const int nx = a.nx, ny = a.ny, nz = a.nz;
    if (y >= ny) return;                         // whole warp: y is warp-uniform
    const bool xin = x0 < nx;
    const int sz = nx * ny;
    const long long i = x0 + (long long)nx * (y + (long long)ny * z);
    const bool hasY = y + 1 < ny, hasZ = z + 1 < nz;
    float4 P0 = f4zero(), P1 = f4zero(), P2 = f4zero(), R0 = f4zero(), R1 = f4zero(), R2 = f4zero();
    float4 Zc = f4zero(), ZY = f4zero(), ZZ = f4zero();
    if (xin) {
        // the voxel's own p and r first
        P0 = ld_once4(a.p + i);
        P1 = ld_once4(a.p + a.N + i);
        P2 = ld_once4(a.p + 2 * a.N + i);
        R0 = ld_ro4(a.rs + i);
        R1 = ld_ro4(a.rs + a.N + i);
        R2 = ld_ro4(a.rs + 2 * a.N + i);
        Zc = ld_ro4(a.z + i);
        if (hasY) ZY = ld_ro4(a.z + i + nx);
        if (hasZ) ZZ = ld_ro4(a.z + i + sz);
    }
    float zx = __shfl_down_sync(kFull, Zc.x, 1);
    if (lane == 31 && x0 + 4 < nx) zx = __ldg(a.z + i + 4);
    if (!xin) return;
    const float gx3 = (x0 + 3 < nx - 1) ? __fsub_rn(Zc.w, zx) : 0.0f;
    float4 G1 = f4zero(), G2 = f4zero();
    if (hasY) {
        G1.x = __fsub_rn(Zc.x, ZY.x); G1.y = __fsub_rn(Zc.y, ZY.y);
        G1.z = __fsub_rn(Zc.z, ZY.z); G1.w = __fsub_rn(Zc.w, ZY.w);
    }
    if (hasZ) {
        G2.x = __fsub_rn(Zc.x, ZZ.x); G2.y = __fsub_rn(Zc.y, ZZ.y);
        G2.z = __fsub_rn(Zc.z, ZZ.z); G2.w = __fsub_rn(Zc.w, ZZ.w);
    }
    dual_update(R0.x, R1.x, R2.x, __fsub_rn(Zc.x, Zc.y), G1.x, G2.x, P0.x, P1.x, P2.x, a.s, a.m);
    dual_update(R0.y, R1.y, R2.y, __fsub_rn(Zc.y, Zc.z), G1.y, G2.y, P0.y, P1.y, P2.y, a.s, a.m);
    dual_update(R0.z, R1.z, R2.z, __fsub_rn(Zc.z, Zc.w), G1.z, G2.z, P0.z, P1.z, P2.z, a.s, a.m);
    dual_update(R0.w, R1.w, R2.w, gx3, G1.w, G2.w, P0.w, P1.w, P2.w, a.s, a.m);
    st4(a.p + i, P0);
    st4(a.p + a.N + i, P1);
    st4(a.p + 2 * a.N + i, P2);
    st4(a.rd + i, R0);
    st4(a.rd + a.N + i, R1);
    st4(a.rd + 2 * a.N + i, R2);
}

__global__ void __launch_bounds__(256) dual_from_z_scalar(const DualArgs a)
{
    const int x = blockIdx.x * 32 + threadIdx.x;
    const int y = blockIdx.y * 8 + threadIdx.y;
    const int z = blockIdx.z;
    const int nx = a.nx, ny = a.ny, nz = a.nz;
    const int px = a.px > 0 ? a.px : nx;             // row pitch
    if (x >= nx || y >= ny) return;
    const long long sz = (long long)px * ny;
    const long long i = x + (long long)px * y + sz * z;
    float P0 = __ldcs(a.p + i), P1 = __ldcs(a.p + a.N + i), P2 = __ldcs(a.p + 2 * a.N + i);
    float R0 = __ldg(a.rs + i), R1 = __ldg(a.rs + a.N + i), R2 = __ldg(a.rs + 2 * a.N + i);
    const float zc = __ldg(a.z + i);
    const float g0 = (x < nx - 1) ? __fsub_rn(zc, __ldg(a.z + i + 1)) : 0.0f;
    const float g1 = (y < ny - 1) ? __fsub_rn(zc, __ldg(a.z + i + px)) : 0.0f;
    const float g2 = (z < nz - 1) ? __fsub_rn(zc, __ldg(a.z + i + sz)) : 0.0f;
    dual_update(R0, R1, R2, g0, g1, g2, P0, P1, P2, a.s, a.m);
    a.p[i] = P0;
    a.p[a.N + i] = P1;
    a.p[2 * a.N + i] = P2;
    a.rd[i] = R0;
    a.rd[a.N + i] = R1;
    a.rd[2 * a.N + i] = R2;
}

// ---------------------------------------------------------------------------
// bounded waits
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Poll the barrier phase with a bounded number of polls (with a short sleep
// between them).  Returns false when the limit is reached.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, int max_polls)
{
    for (int k = 0; k < max_polls; ++k) {
        if (mbar_test(bar, parity)) return true;
        __nanosleep(32);
    }
    return false;
}

// Test hook: wait on a barrier that nobody arrives at, give up after
// `polls` polls, record the timeout in the error word and return.
__global__ void timeout_probe(int *err, int polls)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const bool ok = mbar_wait_bounded(&bar, 0, polls);
    if (!ok && threadIdx.x == 0) atomicExch(err, kErrTimeout);
}

}  // namespace tvfgp
