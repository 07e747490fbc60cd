// Double-float ("dd") arithmetic on the fp32 pipes: a value is hi + lo with
// |lo| <= ulp(hi)/2, about 48 significant bits.  Used where a floating-point
// result decides an integer (the token a uniform selects), so that decision
// is taken at close to float64 precision without the GB300's slow FP64 path.
//
// Error-free transformations: Knuth's TwoSum, Dekker's Fast2Sum and the
// FMA-based TwoProd (Dekker 1971; Knuth, TAOCP vol. 2, 4.2.2).  The
// exponential follows Tang's table-driven method (Tang 1989, ACM TOMS
// 15(2)) in base e with a Cody-Waite reduction (Cody and Waite 1980):
//   y = k ln2/64 + s,  |s| <= ln2/128,  e^y = 2^(k>>6) * 2^((k&63)/64) * e^s,
//   e^s = 1 + s + s^2/2 + s^3/6 + s^4/24 + s^5/120 (the next term is below
//   4e-17).  ln2/64 is held in three parts, the first with 11 significant
//   bits, so that k*c1 is exact for |k| < 2^13 and y - k*c1 is exact
//   (Sterbenz); the 2^(j/64) values come from the host in double and are
//   split into dd pairs.
#pragma once

#include <cuda_runtime.h>

namespace specv {

struct dd {
    float hi, lo;
};

__device__ __forceinline__ dd two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return dd{s, e};
}

// requires |a| >= |b| (or a == 0)
__device__ __forceinline__ dd fast_two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float e = __fsub_rn(b, __fsub_rn(s, a));
    return dd{s, e};
}

__device__ __forceinline__ dd two_prod(float a, float b) {
    const float p = __fmul_rn(a, b);
    const float e = __fmaf_rn(a, b, -p);
    return dd{p, e};
}

__device__ __forceinline__ dd dd_add(dd x, dd y) {
    const dd s = two_sum(x.hi, y.hi);
    const dd t = two_sum(x.lo, y.lo);
    dd r = fast_two_sum(s.hi, __fadd_rn(s.lo, t.hi));
    return fast_two_sum(r.hi, __fadd_rn(r.lo, t.lo));
}

__device__ __forceinline__ dd dd_add_f(dd x, float y) {
    const dd s = two_sum(x.hi, y);
    return fast_two_sum(s.hi, __fadd_rn(s.lo, x.lo));
}

__device__ __forceinline__ dd dd_neg(dd x) { return dd{-x.hi, -x.lo}; }

__device__ __forceinline__ dd dd_mul(dd x, dd y) {
    const dd p = two_prod(x.hi, y.hi);
    const float e = __fadd_rn(p.lo, __fmaf_rn(x.hi, y.lo, __fmul_rn(x.lo, y.hi)));
    return fast_two_sum(p.hi, e);
}

__device__ __forceinline__ dd dd_mul_f(dd x, float f) {
    const dd p = two_prod(x.hi, f);
    return fast_two_sum(p.hi, __fmaf_rn(x.lo, f, p.lo));
}

// 1/x by one Newton step on the fp32 reciprocal (x > 0)
__device__ __forceinline__ dd dd_recip(dd x) {
    const float q = __fdiv_rn(1.0f, x.hi);
    const dd t = dd_mul_f(x, q);                  // x*q, close to 1
    const dd r = dd_add(dd{1.0f, 0.0f}, dd_neg(t));  // 1 - x*q
    return fast_two_sum(q, __fmul_rn(q, r.hi));
}

__device__ __forceinline__ bool dd_gt(dd a, dd b) { return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo); }
__device__ __forceinline__ bool dd_le(dd a, dd b) { return !dd_gt(a, b); }
__device__ __forceinline__ bool dd_pos(dd a) { return a.hi > 0.0f || (a.hi == 0.0f && a.lo > 0.0f); }
__device__ __forceinline__ dd dd_max0(dd a) { return dd_pos(a) ? a : dd{0.0f, 0.0f}; }
__device__ __forceinline__ float dd_to_f(dd a) { return __fadd_rn(a.hi, a.lo); }

// acc + v for non-negative terms: TwoSum on the high parts, the low parts
// added in fp32, then renormalised (Dekker's add; relative error ~2^-45 for
// terms of one sign).  Cheaper than dd_add, which also serves mixed signs.
__device__ __forceinline__ dd dd_acc(dd acc, dd v) {
    const dd s = two_sum(acc.hi, v.hi);
    return fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(acc.lo, v.lo)));
}

// Constants of the double-float exponential: 1/T as a dd pair, ln2/64 in
// three parts, and 2^(j/64), j = 0..63, as dd pairs.
struct DdExpTables {
    float2 it;           // 1 / temperature, (hi, lo)
    float c1, c2, c3;    // ln2/64 = c1 + c2 + c3, c1 with 11 significant bits
    float2 tab[64];      // 2^(j/64) as (hi, lo)
};

// e^((x - m)/T) for x <= m: a dd pair with relative error below ~1e-13 where
// (x - m)/T > -30 (the terms that carry probability mass); values below
// e^-86.6 flush to 0, -inf gives 0.
__device__ __forceinline__ dd dd_expw(float x, float m, const DdExpTables &K) {
    if (!(x > -INFINITY)) return dd{0.0f, 0.0f};
    const dd d = two_sum(x, -m);  // exact
    // y = d / T as an unnormalised pair (yh, yl)
    const float yh = __fmul_rn(d.hi, K.it.x);
    const float yl = __fadd_rn(__fmaf_rn(d.hi, K.it.x, -yh),
                               __fmaf_rn(d.hi, K.it.y, __fmul_rn(d.lo, K.it.x)));
    const float kf = rintf(__fmul_rn(yh, 92.332482616893657f));  // 64 / ln 2
    if (kf < -8000.0f) return dd{0.0f, 0.0f};
    // s = y - k ln2/64 as a dd pair
    const float s1 = __fmaf_rn(-kf, K.c1, yh);  // exact
    const dd t2 = two_prod(kf, K.c2);
    dd s = two_sum(s1, -t2.hi);
    s = dd_add_f(s, yl);
    s.lo = __fadd_rn(s.lo, -__fmaf_rn(kf, K.c3, t2.lo));
    // e^s: 1 + h + h^2/2 exactly, the rest in fp32
    const float h = s.hi;
    const dd sq = two_prod(h, h);
    const float cub = __fmul_rn(__fmul_rn(h, sq.hi),
                                __fmaf_rn(h, __fmaf_rn(h, 1.0f / 120.0f, 1.0f / 24.0f), 1.0f / 6.0f));
    const float tail = __fadd_rn(__fadd_rn(s.lo, __fmul_rn(h, s.lo)), __fmaf_rn(0.5f, sq.lo, cub));
    const dd e1 = fast_two_sum(1.0f, h);
    const dd e2 = fast_two_sum(e1.hi, __fmul_rn(0.5f, sq.hi));
    dd e = fast_two_sum(e2.hi, __fadd_rn(__fadd_rn(e1.lo, e2.lo), tail));
    // times 2^(k/64)
    const int ki = (int)kf;
    const float2 t = K.tab[ki & 63];
    e = dd_mul(e, dd{t.x, t.y});
    const float scale = __int_as_float(((ki >> 6) + 127) << 23);  // 2^(k>>6), k>>6 >= -125
    return dd{__fmul_rn(e.hi, scale), __fmul_rn(e.lo, scale)};
}

// warp-level dd sum in a fixed butterfly order (every lane gets the result)
__device__ __forceinline__ dd warp_dd_sum(dd v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const dd w{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
        v = dd_add(v, w);
    }
    return v;
}

}  // namespace specv
