// fp8.cuh -- per-row FP8 (OCP E4M3) quantisation helpers shared by the
// dispatch with FP8 rows, the combine with FP8 output and the standalone row
// quantiser.
//
// A row v[0..H) is stored as codes q_h = e4m3(RN32(v_h / scale)) with
// scale = RN32(amax / 448) (1 for an all-zero row): binary32 quotient,
// then round-to-nearest-even into E4M3 with saturation to +-448.
//
// The quotient.  All elements of a row share the divisor s, so instead of
// one IEEE division per element the row computes y = RN(1/s') once and every
// element takes the FMA remainder refinement of x' * y twice:
//   q0 = RN(x'*y);  r0 = x' - q0*s' (FMA);  q1 = RN(q0 + r0*y)
//                   r1 = x' - q1*s' (FMA);  q2 = RN(q1 + r1*y).
// q0 is within 1.5 ulp of x'/s' (y is within half an ulp of 1/s'), the first
// step brings the estimate within one ulp, and Markstein's theorem
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with y the
// correctly rounded reciprocal and q1 within one ulp of x'/s', the
// remainder r1 is exact and RN(q1 + r1*y) is the correctly rounded quotient.
// The theorem needs no overflow and no underflow, so rows whose s lies
// outside [2^-100, 2^100] divide the scaled pair x' = x*m, s' = s*m with
// m = 2^100 or 2^-100 (exact power-of-two scalings: x/s = x'/s'); elsewhere
// m = 1.  Quotients below 2^-126 (including every x' that underflows) are
// far below half the smallest E4M3 subnormal (2^-10) and become a zero with
// the sign of x either way, which the result is given explicitly.
#pragma once

#include <cuda_fp8.h>

#include <cstdint>

#include "f32x2.cuh"

namespace moe {
namespace fp8 {

constexpr float kMax = 448.0f;  // largest finite E4M3 value

struct RowScale {
    float s;   // the row's scale (what is stored)
    float m;   // power-of-two scaling of the pair (1 for most rows)
    float sd;  // s * m
    float y;   // RN(1 / sd)
};

__device__ __forceinline__ RowScale row_scale(float amax) {
    RowScale r;
    r.s = amax > 0.0f ? __fdiv_rn(amax, kMax) : 1.0f;
    r.m = r.s < 0x1p-100f ? 0x1p100f : (r.s > 0x1p100f ? 0x1p-100f : 1.0f);
    r.sd = __fmul_rn(r.s, r.m);
    r.y = __frcp_rn(r.sd);
    return r;
}

// RN32(a / s) and RN32(b / s), two elements per instruction (paired fp32,
// each lane rounded as the scalar operation would be; x' - q*s' is formed as
// fma(q, -s', x'), the same exact product).  SCALED: the pair is prescaled
// by r.m (rows whose scale is outside [2^-100, 2^100]); otherwise r.m = 1
// and r.sd = r.s.
template <bool SCALED>
__device__ __forceinline__ void quotient2(float a, float b, const RowScale &r, float &qa,
                                          float &qb) {
    x2::f2 xs = x2::pack(a, b);
    if (SCALED) xs = x2::mul(xs, x2::pack(r.m, r.m));
    const x2::f2 y = x2::pack(r.y, r.y), nsd = x2::pack(-r.sd, -r.sd);
    x2::f2 q = x2::mul(xs, y);
    x2::f2 e = x2::fma(q, nsd, xs);
    q = x2::fma(e, y, q);
    e = x2::fma(q, nsd, xs);
    q = x2::fma(e, y, q);
    x2::unpack(q, qa, qb);
    qa = copysignf(qa, a);
    qb = copysignf(qb, b);
}

// Two binary32 values -> two E4M3 codes (low byte first), RN, saturating.
__device__ __forceinline__ uint32_t cvt2(float a, float b) {
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// Eight values of a row -> eight codes packed in 8 bytes.
template <bool SCALED>
__device__ __forceinline__ uint2 quantize8(const float (&v)[8], const RowScale &r) {
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float qa, qb;
        quotient2<SCALED>(v[2 * i], v[2 * i + 1], r, qa, qb);
        c[i] = cvt2(qa, qb);
    }
    return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

template <int VPT>
__device__ __forceinline__ void quantize_row(const float (&v)[VPT][8], const RowScale &r,
                                             uint2 (&q)[VPT]) {
    if (r.m == 1.0f) {  // the row is uniform: one branch for all lanes
#pragma unroll
        for (int j = 0; j < VPT; ++j) q[j] = quantize8<false>(v[j], r);
    } else {
#pragma unroll
        for (int j = 0; j < VPT; ++j) q[j] = quantize8<true>(v[j], r);
    }
}

}  // namespace fp8
}  // namespace moe
