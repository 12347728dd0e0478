// Self-check of the fast projection onto the unit ball (project_unit_ball in
// fgp_kernels.cuh) against CUDA's correctly rounded operations, on the GPU
// that runs it.  Plain grid-stride loops: no waits, every index in range.
//
//   mode 0  every float nn in [1, 2^100): the fast n equals __fsqrt_rn(nn)
//           and the fast y equals __frcp_rn(n);
//   mode 1  `count` pseudo-random triples q: project_unit_ball equals
//           project_unit_ball_ieee bit for bit (components spread over
//           exponents -130..48, with zeros and values below the guard);
//   mode 2  `count` quotients q / n: div_by_recip_rn(q, n, __frcp_rn(n))
//           equals __fdiv_rn(q, n) for q / n placed within a few ulps of a
//           power of two (half the samples) or anywhere (the other half).
//   mode 3  `count` quads: dual_update4 equals four updates built on the
//           IEEE projection, bit for bit (r, g, p drawn so that about half
//           the voxels project, with zero and tiny components mixed in).
//
// out[0] counts mismatches; out[1] is lowered (atomicMin) to the index of
// the first one.  The caller sets out to {0, ~0} beforehand.
#pragma once

#include "fgp_kernels.cuh"

namespace tvfgp {

constexpr uint32_t kNnFirst = 0x3f800000u;   // 1
constexpr uint32_t kNnEnd = 0x71800000u;     // 2^100 (excluded)

__device__ __forceinline__ uint64_t splitmix64(uint64_t x)
{
    x += 0x9e3779b97f4a7c15ull;
    x = (x ^ (x >> 30)) * 0xbf58476d1ce4e5b9ull;
    x = (x ^ (x >> 27)) * 0x94d049bb133111ebull;
    return x ^ (x >> 31);
}

// A float with the given sign bit, unbiased exponent e (normal range, or 0
// for e < -126: a subnormal with a random fraction) and 23 random fraction bits.
__device__ __forceinline__ float make_float(uint32_t sign, int e, uint32_t frac)
{
    frac &= 0x7fffffu;
    if (e < -126) return __uint_as_float((sign << 31) | (frac >> min(23, -126 - e)));
    return __uint_as_float((sign << 31) | (static_cast<uint32_t>(e + 127) << 23) | frac);
}

__device__ __forceinline__ void record_mismatch(unsigned long long *out, unsigned long long i)
{
    atomicAdd(&out[0], 1ull);
    atomicMin(&out[1], i);
}

// One voxel of the update with the IEEE projection (the reference of mode 3).
__device__ __forceinline__ void dual_update_ieee(float &r0, float &r1, float &r2, float g0, float g1,
                                                 float g2, float &p0, float &p1, float &p2, float s, float m)
{
    float q0 = __fadd_rn(r0, __fmul_rn(g0, s));
    float q1 = __fadd_rn(r1, __fmul_rn(g1, s));
    float q2 = __fadd_rn(r2, __fmul_rn(g2, s));
    const float nn = __fadd_rn(__fadd_rn(__fmul_rn(q0, q0), __fmul_rn(q1, q1)), __fmul_rn(q2, q2));
    project_unit_ball_ieee(q0, q1, q2, nn);
    r0 = __fadd_rn(q0, __fmul_rn(m, __fsub_rn(q0, p0)));
    r1 = __fadd_rn(q1, __fmul_rn(m, __fsub_rn(q1, p1)));
    r2 = __fadd_rn(q2, __fmul_rn(m, __fsub_rn(q2, p2)));
    p0 = q0;
    p1 = q1;
    p2 = q2;
}

// A value for mode 3: mostly of order one, sometimes zero, tiny or large.
__device__ __forceinline__ float quad_value(uint64_t h)
{
    const uint32_t kind = static_cast<uint32_t>(h >> 60);
    const uint32_t sign = static_cast<uint32_t>(h >> 59) & 1u;
    const uint32_t frac = static_cast<uint32_t>(h);
    if (kind == 0) return sign ? -0.0f : 0.0f;
    if (kind == 1) return make_float(sign, -140 + static_cast<int>((h >> 40) % 70), frac);   // tiny
    if (kind == 2) return make_float(sign, 10 + static_cast<int>((h >> 40) % 50), frac);     // large
    return make_float(sign, -3 - static_cast<int>((h >> 40) % 4), frac);                      // 2^-6 .. 2^-2
}

__global__ void projection_check(int mode, unsigned long long count, unsigned long long seed,
                                 unsigned long long *out)
{
    const unsigned long long stride = static_cast<unsigned long long>(gridDim.x) * blockDim.x;
    for (unsigned long long i = static_cast<unsigned long long>(blockIdx.x) * blockDim.x + threadIdx.x;
         i < count; i += stride) {
        if (mode == 0) {
            const float nn = __uint_as_float(kNnFirst + static_cast<uint32_t>(i));
            float n, y;
            sqrt_recip_rn(nn, n, y);
            if (__float_as_uint(n) != __float_as_uint(__fsqrt_rn(nn)) ||
                __float_as_uint(y) != __float_as_uint(__frcp_rn(n)))
                record_mismatch(out, i);
        } else if (mode == 1) {
            const uint64_t h0 = splitmix64(seed ^ (2 * i)), h1 = splitmix64(seed ^ (2 * i + 1));
            const int base = -2 + static_cast<int>((h0 >> 58) % 51);          // -2 .. 48
            float q[3];
            for (int a = 0; a < 3; ++a) {
                const uint32_t bits = static_cast<uint32_t>(h1 >> (21 * a));
                const uint32_t sel = (bits >> 18) & 15u;
                const int span = sel < 12 ? 41 : 179;                         // mostly near the base
                const int e = base - static_cast<int>(((h0 >> (14 * a)) & 0x3fffu) % span);
                q[a] = sel == 15 ? 0.0f : make_float((bits >> 17) & 1u, e, static_cast<uint32_t>(h0 >> 40) ^ bits);
                if (sel == 14 && a == 1) q[a] = -0.0f;
            }
            const float nn = __fadd_rn(__fadd_rn(__fmul_rn(q[0], q[0]), __fmul_rn(q[1], q[1])),
                                       __fmul_rn(q[2], q[2]));
            float f0 = q[0], f1 = q[1], f2 = q[2], r0 = q[0], r1 = q[1], r2 = q[2];
            project_unit_ball(f0, f1, f2, nn);
            project_unit_ball_ieee(r0, r1, r2, nn);
            if (__float_as_uint(f0) != __float_as_uint(r0) || __float_as_uint(f1) != __float_as_uint(r1) ||
                __float_as_uint(f2) != __float_as_uint(r2))
                record_mismatch(out, i);
        } else if (mode == 3) {
            float4 v[9];
            float *f = &v[0].x;
            for (int k = 0; k < 36; ++k) f[k] = quad_value(splitmix64(seed ^ (36 * i + k)));
            const float sc = make_float(0, static_cast<int>(splitmix64(~seed ^ i) % 5) + 1, 0u);   // s: 2 .. 32
            const float m = 0.25f;
            float4 R0 = v[0], R1 = v[1], R2 = v[2], P0 = v[6], P1 = v[7], P2 = v[8];
            dual_update4(R0, R1, R2, v[3], v[4], v[5], P0, P1, P2, sc, m, neg_zero(sc));
            bool same = true;
            const float *g0 = &v[3].x, *g1 = &v[4].x, *g2 = &v[5].x;
            const float *o[6] = {&R0.x, &R1.x, &R2.x, &P0.x, &P1.x, &P2.x};
            for (int e = 0; e < 4; ++e) {
                float r0 = f[e], r1 = f[4 + e], r2 = f[8 + e], p0 = f[24 + e], p1 = f[28 + e], p2 = f[32 + e];
                dual_update_ieee(r0, r1, r2, g0[e], g1[e], g2[e], p0, p1, p2, sc, m);
                const float ref[6] = {r0, r1, r2, p0, p1, p2};
                for (int c = 0; c < 6; ++c) same &= __float_as_uint(o[c][e]) == __float_as_uint(ref[c]);
            }
            if (!same) record_mismatch(out, i);
        } else {
            const uint64_t h = splitmix64(seed ^ i), g = splitmix64(~seed ^ i);
            const float n = make_float(0, static_cast<int>((h >> 58) % 50), static_cast<uint32_t>(h));
            if (!(n > 1.0f)) continue;
            float q;
            if (h & (1ull << 57)) {
                // q / n within a few ulps of +-2^j
                const int j = -40 + static_cast<int>((g >> 58) % 61);
                const float t = make_float(static_cast<uint32_t>(g >> 57) & 1u, j, 0u);
                q = __fmul_rn(t, n);
                const int d = static_cast<int>((g >> 32) & 15u) - 8;            // -8 .. 7 ulps
                q = __uint_as_float(__float_as_uint(q) + d);
            } else {
                q = make_float(static_cast<uint32_t>(g >> 57) & 1u, -75 + static_cast<int>((g >> 50) % 125),
                               static_cast<uint32_t>(g));
            }
            const float aq = fabsf(q);
            if (!(aq >= 0x1p-75f) || !(aq < 0x1p50f)) continue;             // the guard's range
            const float d = div_by_recip_rn(q, n, __frcp_rn(n));
            if (__float_as_uint(d) != __float_as_uint(__fdiv_rn(q, n))) record_mismatch(out, i);
        }
    }
}

}  // namespace tvfgp
