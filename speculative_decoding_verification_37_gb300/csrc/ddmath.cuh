// Double-float ("dd") arithmetic on the fp32 pipes: a value is hi + lo with
// |lo| <= ulp(hi)/2, about 48 significant bits.  Used where a floating-point
// result decides an integer (the token a uniform selects), so that decision
// is taken at close to float64 precision without the GB300's slow FP64 path.
//
// Error-free transformations: Knuth's TwoSum, Dekker's Fast2Sum and the
// FMA-based TwoProd (Dekker 1971; Knuth, TAOCP vol. 2, 4.2.2).  exp2 follows
// Tang's table-driven reduction (Tang 1989, ACM TOMS 15(2)):
//   2^y = 2^n * 2^(j/64) * e^(r ln 2),  n = rint(y), j = rint(64 (y - n)),
//   |r| <= 1/128, with e^z = 1 + z + z^2/2 + z^3/6 + z^4/24 + z^5/120
//   (the next term is below 4e-17 for |z| <= 0.0055).  The 2^(j/64) values
//   and ln 2 come from the host in double and are split into dd pairs.
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

// Constants a kernel needs for dd exp2: ln 2 and 2^(j/64), j = -32..32.
struct DdExpTables {
    float2 ln2;          // (hi, lo)
    float2 tab[65];      // 2^((j-32)/64) as (hi, lo)
};

// 2^y for y <= 0 (values below 2^-125 flush to 0, far below any tolerance here).
__device__ __forceinline__ dd dd_exp2(dd y, const float2 *tab, float2 ln2) {
    const float n = rintf(y.hi);
    if (n < -125.0f) return dd{0.0f, 0.0f};
    const dd f = fast_two_sum(__fsub_rn(y.hi, n), y.lo);   // y.hi - n is exact
    const float jf = rintf(__fmul_rn(f.hi, 64.0f));
    const dd r = fast_two_sum(__fsub_rn(f.hi, __fmul_rn(jf, 0.015625f)), f.lo);  // exact subtraction
    const dd z = dd_mul(r, dd{ln2.x, ln2.y});
    const dd z2 = dd_mul(z, z);
    const float zh = z.hi;
    const float tail = __fmul_rn(__fmul_rn(zh, __fmul_rn(zh, zh)),
                                 __fmaf_rn(zh, __fmaf_rn(zh, 1.0f / 120.0f, 1.0f / 24.0f), 1.0f / 6.0f));
    dd s = dd_add_f(z, 1.0f);
    s = dd_add(s, dd{__fmul_rn(z2.hi, 0.5f), __fmul_rn(z2.lo, 0.5f)});
    s = dd_add_f(s, tail);
    const float2 t = tab[(int)jf + 32];
    s = dd_mul(s, dd{t.x, t.y});
    const float scale = __int_as_float(((int)n + 127) << 23);  // 2^n, exact for n >= -126
    return dd{__fmul_rn(s.hi, scale), __fmul_rn(s.lo, scale)};
}

// e^((x - m)/T) = 2^((x - m) * c2) with c2 = log2(e)/T given as a dd pair.
__device__ __forceinline__ dd dd_expw(float x, float m, dd c2, const float2 *tab, float2 ln2) {
    if (x == -INFINITY) return dd{0.0f, 0.0f};
    const dd d = two_sum(x, -m);
    return dd_exp2(dd_mul(d, c2), tab, ln2);
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
