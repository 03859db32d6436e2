// Double-float ("df") arithmetic on the float32 pipes: a value is hi + lo with |lo| <= ulp(hi)/2,
// about 48 significant bits.  The per-stream scalars of the verify rules (ratios, running
// products, thresholds, CDF positions) are carried in df so that their rounding stays far below
// the 1e-6 relative window in which a decision counts as a near tie, without float64 (whose
// dependent-operation latency on this part is hundreds of cycles).
//
// Building blocks are the classical error-free transformations (Knuth's TwoSum, Dekker's
// Fast2Sum, and the FMA-based exact product); every operation uses explicit _rn intrinsics so
// that the compiler cannot contract or reassociate them.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

struct df {
    float hi, lo;
};

__device__ __forceinline__ df df_make(float a) { return df{a, 0.f}; }

// s + e == a + b exactly (any magnitudes)
__device__ __forceinline__ df two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return df{s, e};
}
// s + e == a + b exactly when |a| >= |b| (or a == 0)
__device__ __forceinline__ df fast_two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    return df{s, __fsub_rn(b, __fsub_rn(s, a))};
}
// p + e == a * b exactly (barring under/overflow)
__device__ __forceinline__ df two_prod(float a, float b) {
    const float p = __fmul_rn(a, b);
    return df{p, __fmaf_rn(a, b, -p)};
}

__device__ __forceinline__ df df_add(df a, df b) {
    const df s = two_sum(a.hi, b.hi);
    const df t = two_sum(a.lo, b.lo);
    df r = fast_two_sum(s.hi, __fadd_rn(s.lo, t.hi));
    return fast_two_sum(r.hi, __fadd_rn(r.lo, t.lo));
}
__device__ __forceinline__ df df_add_f(df a, float b) {
    const df s = two_sum(a.hi, b);
    return fast_two_sum(s.hi, __fadd_rn(s.lo, a.lo));
}
__device__ __forceinline__ df df_neg(df a) { return df{-a.hi, -a.lo}; }
__device__ __forceinline__ df df_sub(df a, df b) { return df_add(a, df_neg(b)); }

__device__ __forceinline__ df df_mul(df a, df b) {
    const df p = two_prod(a.hi, b.hi);
    const float c = __fmaf_rn(a.hi, b.lo, __fmul_rn(a.lo, b.hi));
    return fast_two_sum(p.hi, __fadd_rn(p.lo, c));
}
__device__ __forceinline__ df df_mul_f(df a, float b) {
    const df p = two_prod(a.hi, b);
    return fast_two_sum(p.hi, __fmaf_rn(a.lo, b, p.lo));
}
// exact scaling by a power of two held in a float
__device__ __forceinline__ df df_scale(df a, float pow2) {
    return df{__fmul_rn(a.hi, pow2), __fmul_rn(a.lo, pow2)};
}

__device__ __forceinline__ df df_div(df a, df b) {
    const float q1 = __fdiv_rn(a.hi, b.hi);
    const df r = df_sub(a, df_mul_f(b, q1));
    const float q2 = __fdiv_rn(r.hi, b.hi);
    const df r2 = df_sub(r, df_mul_f(b, q2));
    const float q3 = __fdiv_rn(r2.hi, b.hi);
    return df_add_f(fast_two_sum(q1, q2), q3);
}

__device__ __forceinline__ float df_to_f(df a) { return __fadd_rn(a.hi, a.lo); }

// a <= b, a < b, sign tests on the exact difference
__device__ __forceinline__ bool df_le(df a, df b) {
    const df d = df_sub(a, b);
    return d.hi < 0.f || (d.hi == 0.f && d.lo <= 0.f);
}
__device__ __forceinline__ bool df_lt(df a, df b) { return !df_le(b, a); }
__device__ __forceinline__ bool df_is_zero(df a) { return a.hi == 0.f && a.lo == 0.f; }
__device__ __forceinline__ df df_min(df a, df b) { return df_le(a, b) ? a : b; }

// 2^d for an integer-valued float d (d may be -inf): exact power of two, 0 below 2^-126
__device__ __forceinline__ float pow2_int(float d) {
    if (!(d >= -126.f)) return 0.f;
    if (d > 127.f) return __int_as_float(0x7f800000);
    return __int_as_float(((int)d + 127) << 23);
}

// The uniform U(x) = ((x >> 8) + 0.5) * 2^-24 as an exact df.
__device__ __forceinline__ df uniform24_df(uint32_t x) {
    const float k = (float)(x >> 8) * 0x1p-24f;   // exact: x >> 8 < 2^24
    return two_sum(k, 0x1p-25f);
}

// 2^x for a df argument, to about 3e-10 relative: x = n + f with n = rint(x.hi),
// |f| <= 0.5 + tiny; 2^f = e^(f ln 2) by its Taylor series (terms up to g^9/9!, |g| <= 0.35),
// evaluated in df by Horner's rule; then an exact scaling by 2^n.  Arguments are clamped to
// [-150, 126], which maps to 0 and to 2^126 respectively.
__device__ __forceinline__ df df_exp2(df x) {
    if (!(x.hi > -150.f)) return df{0.f, 0.f};
    if (x.hi > 126.f) x = df{126.f, 0.f};
    const float n = rintf(x.hi);
    const df f = df_add_f(df{__fsub_rn(x.hi, n), 0.f}, x.lo);
    // ln 2 = LN2_HI + LN2_LO
    const df ln2{0.6931471824645996f, -1.9046542121259336e-09f};
    const df g = df_mul(f, ln2);
    // 1/k! for k = 0 .. 12 as df constants (float nearest, then the rounded remainder)
    const df inv_fact[13] = {
        {1.0f, 0.0f},
        {1.0f, 0.0f},
        {0.5f, 0.0f},
        {0.1666666716337204f, -4.967053879312289e-09f},
        {0.0416666679084301f, -1.2417634698280722e-09f},
        {0.008333333767950535f, -4.34617203337595e-10f},
        {0.0013888889225199819f, -3.3631094437103215e-11f},
        {0.00019841270113829523f, -2.725596874933456e-12f},
        {2.4801587642286904e-05f, -3.40699609366682e-13f},
        {2.7557318844628753e-06f, 3.793571224297229e-14f},
        {2.755731998149713e-07f, -7.575112209051195e-15f},
        {2.5052107943679403e-08f, 4.4176230446483665e-16f},
        {2.0876755879584152e-09f, 1.1082839147459852e-16f},
    };
    df p = inv_fact[9];
#pragma unroll
    for (int k = 8; k >= 0; --k) p = df_add(df_mul(p, g), inv_fact[k]);
    // exact 2^n (n in [-150, 126]) as up to two float factors
    if (n >= -126.f) return df_scale(p, pow2_int(n));
    return df_scale(df_scale(p, pow2_int(n + 64.f)), 0x1p-64f);
}

// log2(e) / T as a df (T > 0) whose low part is strictly positive, so that x (hi + lo) with
// x = -inf is -inf in both products: a low part of either sign, or zero, would give
// -inf + inf = NaN for a -inf logit (a masked column, or one outside a reduced draft
// vocabulary).  A non-positive low part takes one unit in the last place from the high part
// (an exact move up to the low part's own rounding, ~2^-48 relative).
__device__ __forceinline__ df temperature_scale(float T) {
    const df l2e{1.4426950216293335f, 1.925963033500011e-08f};
    df a = df_div(l2e, df_make(T));
    if (!(a.lo > 0.f)) {
        const float h = __int_as_float(__float_as_int(a.hi) - 1);   // hi > 0: the next float toward 0
        a.lo = a.lo + (a.hi - h);
        a.hi = h;
    }
    return a;
}

}  // namespace sv
