// s5_ff.cuh -- float-float ("double-single") arithmetic for the per-mode
// factors of the discretisation.
//
// A value is the unevaluated sum hi + lo of two floats with |lo| <= ulp(hi)/2:
// about 48 bits of significand from FP32 instructions only, which GB300 runs
// at full rate (its float64 units are few and slow).  The building blocks are
// the error-free transformations of the published literature:
//   TwoSum      Knuth, The Art of Computer Programming vol. 2, 4.2.2 (Moller's
//               algorithm): s + e = a + b exactly, for any a, b;
//   Fast2Sum    Dekker, "A floating-point technique for extending the
//               available precision", Numer. Math. 18 (1971): the same when
//               |a| >= |b|;
//   TwoProduct  Dekker (1971), in its fused-multiply-add form: p + e = a * b
//               exactly, e = fma(a, b, -p);
// and the float-float sum and product built from them (Dekker 1971; the
// "accurate" sum that adds the low parts separately).  Every operation uses
// the explicitly rounded intrinsics so that the compiler neither contracts
// nor reassociates the steps the transformations depend on.
//
// Elementary functions here are written from their Taylor series (the
// coefficients 1/n! are exact rationals, stored as float-float pairs) after a
// Cody-Waite argument reduction (Cody and Waite, "Software Manual for the
// Elementary Functions", 1980): x = k*c + r with the constant c = ln 2 or pi/2
// split into three floats, the first with 12 significant bits; every k*c_i is
// formed with TwoProduct, so r is exact to float-float precision.
#pragma once

#include <cuda_runtime.h>

namespace s5 {
namespace ff {

struct F2 {
    float hi, lo;
};

__device__ __forceinline__ F2 make(float hi) { return {hi, 0.f}; }

__device__ __forceinline__ F2 two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return {s, e};
}

__device__ __forceinline__ F2 fast_two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

__device__ __forceinline__ F2 two_prod(float a, float b) {
    const float p = __fmul_rn(a, b);
    return {p, __fmaf_rn(a, b, -p)};
}

__device__ __forceinline__ F2 neg(F2 a) { return {-a.hi, -a.lo}; }

// (a.hi + a.lo) + (b.hi + b.lo), relative error a few units of 2^-48
__device__ __forceinline__ F2 add(F2 a, F2 b) {
    F2 s = two_sum(a.hi, b.hi);
    const F2 t = two_sum(a.lo, b.lo);
    s.lo = __fadd_rn(s.lo, t.hi);
    s = fast_two_sum(s.hi, s.lo);
    s.lo = __fadd_rn(s.lo, t.lo);
    return fast_two_sum(s.hi, s.lo);
}

__device__ __forceinline__ F2 sub(F2 a, F2 b) { return add(a, neg(b)); }

__device__ __forceinline__ F2 mul(F2 a, F2 b) {
    F2 p = two_prod(a.hi, b.hi);
    p.lo = __fmaf_rn(a.hi, b.lo, p.lo);
    p.lo = __fmaf_rn(a.lo, b.hi, p.lo);
    return fast_two_sum(p.hi, p.lo);
}

__device__ __forceinline__ F2 mul(F2 a, float b) {
    F2 p = two_prod(a.hi, b);
    p.lo = __fmaf_rn(a.lo, b, p.lo);
    return fast_two_sum(p.hi, p.lo);
}

// a * 2^k (exact unless the result leaves the normal range)
__device__ __forceinline__ F2 ldexp2(F2 a, int k) { return {ldexpf(a.hi, k), ldexpf(a.lo, k)}; }

// 1 / a: the correctly rounded float reciprocal, then one Newton step
// y + y (1 - a y) carried out in float-float
__device__ __forceinline__ F2 recip(F2 a) {
    const float y = __frcp_rn(a.hi);
    const F2 r = sub(make(1.f), mul(a, y));
    return add(make(y), mul(r, y));
}

__device__ __forceinline__ float to_float(F2 a) { return __fadd_rn(a.hi, a.lo); }

// ---------------------------------------------------------------------------
// Constants: 1/n! as float-float pairs and the three-part splits of ln 2 and
// pi/2 (each part the float nearest the remainder of the exact constant;
// the parts add up to the constant within 2^-64 of it, relative).
// ---------------------------------------------------------------------------
__device__ __forceinline__ F2 inv_fact(int n) {
    switch (n) {
        case 0: return {0x1p+0f, 0.f};
        case 1: return {0x1p+0f, 0.f};
        case 2: return {0x1p-1f, 0.f};
        case 3: return {0x1.555556p-3f, -0x1.555556p-28f};
        case 4: return {0x1.555556p-5f, -0x1.555556p-30f};
        case 5: return {0x1.111112p-7f, -0x1.ddddep-32f};
        case 6: return {0x1.6c16c2p-10f, -0x1.27d27ep-35f};
        case 7: return {0x1.a01a02p-13f, -0x1.7f97fap-39f};
        case 8: return {0x1.a01a02p-16f, -0x1.7f97fap-42f};
        case 9: return {0x1.71de3ap-19f, 0x1.55b1ccp-45f};
        case 10: return {0x1.27e4fcp-22f, -0x1.10ec14p-47f};
        case 11: return {0x1.ae6456p-26f, 0x1.fd5138p-52f};
        case 12: return {0x1.1eed8ep-29f, 0x1.ff1b12p-54f};
        case 13: return {0x1.612462p-33f, -0x1.8af25ep-58f};
        case 14: return {0x1.93974ap-37f, 0x1.180f94p-62f};
        case 15: return {0x1.ae7f3ep-41f, 0x1.ccee08p-67f};
        case 16: return {0x1.ae7f3ep-45f, 0x1.ccee08p-71f};
        default: return {0.f, 0.f};
    }
}
constexpr float LN2_1 = 0x1.62ep-1f, LN2_2 = 0x1.0bfbe8p-15f, LN2_3 = 0x1.cf79acp-40f;
constexpr float INV_LN2 = 0x1.715476p+0f;
constexpr float PIO2_1 = 0x1.922p+0f, PIO2_2 = -0x1.2aeef4p-18f, PIO2_3 = -0x1.73dcb4p-43f;
constexpr float TWO_OVER_PI = 0x1.45f306p-1f;

// x - k*(c1 + c2 + c3) in float-float, every product error-free
__device__ __forceinline__ F2 reduce(F2 x, float k, float c1, float c2, float c3) {
    F2 r = add(x, neg(two_prod(k, c1)));
    r = add(r, neg(two_prod(k, c2)));
    return add(r, neg(two_prod(k, c3)));
}

// e^r - 1 for |r| <= ln2/2 + a little: r * sum_{m>=0} r^m/(m+1)!, the series
// cut after m = 12 (the next term is below 4e-18).  Terms m >= 8 add up to
// less than 3e-10 and are summed in float.
__device__ __forceinline__ F2 expm1_reduced(F2 r) {
    float t = inv_fact(13).hi;
#pragma unroll
    for (int m = 11; m >= 8; --m) t = __fmaf_rn(t, r.hi, inv_fact(m + 1).hi);
    F2 acc = make(t);
#pragma unroll
    for (int m = 7; m >= 0; --m) acc = add(mul(acc, r), inv_fact(m + 1));
    return mul(acc, r);
}

// e^x and e^x - 1 of a float-float x (x >= -87, x <= 88)
__device__ __forceinline__ void exp_expm1(F2 x, F2 &ex, F2 &em1) {
    const float k = rintf(__fmul_rn(x.hi, INV_LN2));
    const F2 r = reduce(x, k, LN2_1, LN2_2, LN2_3);
    const F2 e = expm1_reduced(r);
    const int ki = (int)k;
    ex = ldexp2(add(make(1.f), e), ki);
    em1 = ki == 0 ? e : add(ex, make(-1.f));
}

// sin x, cos x and 1 - cos x of a float-float x: x = k*pi/2 + r, |r| <= pi/4
// (+ a little); with y = r^2,
//   sin r = r * sum (-1)^m y^m/(2m+1)!,   1 - cos r = y * sum (-1)^m y^m/(2m+2)!,
// both cut after m = 7 (next terms below 2e-15 of the leading one); terms
// m >= 4 are summed in float.  1 - cos x is taken from the versine series in
// quadrant 0 (no cancellation near x = 0) and as 1 -+ sin r / 1 + cos r in
// the others, where it is at least 1 - cos(pi/4).
__device__ __forceinline__ void sincos_vers(F2 x, F2 &s, F2 &c, F2 &v) {
    const float k = rintf(__fmul_rn(x.hi, TWO_OVER_PI));
    const F2 r = reduce(x, k, PIO2_1, PIO2_2, PIO2_3);
    const F2 y = mul(r, r);
    // Horner from m = 7 (coefficient (-1)^7/15!, resp. /16!) down to m = 4 in
    // float: ts = sum_{m=4..7} (-1)^m y^(m-4)/(2m+1)!, tv the versine analogue
    float ts = -inv_fact(15).hi, tv = -inv_fact(16).hi;
#pragma unroll
    for (int m = 6; m >= 4; --m) {
        const float sg = (m & 1) ? -1.f : 1.f;
        ts = __fmaf_rn(ts, y.hi, sg * inv_fact(2 * m + 1).hi);
        tv = __fmaf_rn(tv, y.hi, sg * inv_fact(2 * m + 2).hi);
    }
    F2 as = make(ts), av = make(tv);
#pragma unroll
    for (int m = 3; m >= 0; --m) {
        const F2 cs = (m & 1) ? neg(inv_fact(2 * m + 1)) : inv_fact(2 * m + 1);
        const F2 cv = (m & 1) ? neg(inv_fact(2 * m + 2)) : inv_fact(2 * m + 2);
        as = add(mul(as, y), cs);
        av = add(mul(av, y), cv);
    }
    const F2 sr = mul(as, r);          // sin r
    const F2 vr = mul(av, y);          // 1 - cos r
    const F2 cr = sub(make(1.f), vr);  // cos r
    switch (((int)k) & 3) {
        case 0: s = sr; c = cr; v = vr; break;
        case 1: s = cr; c = neg(sr); v = add(make(1.f), sr); break;
        case 2: s = neg(sr); c = neg(cr); v = add(make(1.f), cr); break;
        default: s = neg(cr); c = sr; v = sub(make(1.f), sr); break;
    }
}

}  // namespace ff
}  // namespace s5
