// precise.cuh -- double-float arithmetic and the sampling weights of one row,
// accurate enough that the GPU's inverse-CDF pick agrees with a float64
// evaluation except within ~1e-10 of a CDF edge.
//
// Why: the sampled token is the first index j whose running weight sum
// exceeds u * Z. A vocabulary of V tokens puts V CDF edges in [0, 1), so a
// CDF error of e flips about 2 e V draws; fp32 weights and sums (e ~ 1e-8)
// would flip ~1e-3 of the draws at V = 128k. Here every weight is
// w_j = 2^((l_j - l_max) * k), k = log2(e) / T, with
//   - the exponent (l_j - l_max) * k carried as an unevaluated pair hi + lo
//     (Dekker's error-free product via FMA),
//   - "heavy" weights (w_j > 2^-13 of the row maximum) evaluated in
//     double-float: 2^x = 2^n * 2^(i/64) * e^(r ln 2), |r| <= 1/128, with the
//     table 2^(i/64) held as float pairs and a degree-4 Taylor polynomial for
//     e^a - 1 (Tang's table-driven method, ACM TOMS 15(2), 1989),
//   - light weights from the SFU's 2^x of the high part, corrected to first
//     order by the low part (their rounding errors average out in the sums),
//   - all sums, normalisers and prefix sums in double-float (Knuth's TwoSum,
//     Dekker's Fast2Sum and TwoProduct).
#pragma once

#include "common.cuh"

namespace specv {

struct df {
    float hi, lo;
};

__device__ __forceinline__ df df_make(float h, float l = 0.f) { return df{h, l}; }

// s + e == a + b exactly (Knuth).
__device__ __forceinline__ df two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return df{s, e};
}
// s + e == a + b exactly when |a| >= |b| (Dekker).
__device__ __forceinline__ df fast_two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    return df{s, __fsub_rn(b, __fsub_rn(s, a))};
}
// p + e == a * b exactly (FMA).
__device__ __forceinline__ df two_prod(float a, float b) {
    const float p = __fmul_rn(a, b);
    return df{p, __fmaf_rn(a, b, -p)};
}
__device__ __forceinline__ df df_add(df a, df b) {
    df s = two_sum(a.hi, b.hi);
    return fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}
__device__ __forceinline__ df df_mul(df a, df b) {
    df p = two_prod(a.hi, b.hi);
    return fast_two_sum(p.hi, __fadd_rn(p.lo, __fmaf_rn(a.hi, b.lo, __fmul_rn(a.lo, b.hi))));
}
__device__ __forceinline__ df df_mul_f(df a, float b) {
    df p = two_prod(a.hi, b);
    return fast_two_sum(p.hi, __fmaf_rn(a.lo, b, p.lo));
}
__device__ __forceinline__ df df_sub(df a, df b) { return df_add(a, df{-b.hi, -b.lo}); }
// 1 / a with one Newton correction.
__device__ __forceinline__ df df_recip(df a) {
    const float y = 1.0f / a.hi;
    // e = 1 - a * y, evaluated exactly enough in double-float
    df ay = df_mul_f(a, y);
    df e = df_sub(df{1.f, 0.f}, ay);
    return fast_two_sum(y, __fmul_rn(y, e.hi));
}
// a > b for normalised pairs
__device__ __forceinline__ bool df_gt(df a, df b) { return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo); }
__device__ __forceinline__ bool df_pos(df a) { return a.hi > 0.f || (a.hi == 0.f && a.lo > 0.f); }

// The residual's normaliser Z = sum max(0, p - q) lies in [0, 1]. When p and
// q agree exactly (one-hot rows of the same column, say) the double-float
// evaluation leaves a rounding residue of a few units of 2^-48 instead of 0;
// a Z below 2^-40 is that residue, and the draw then takes p as the
// float64 reading does for Z = 0.
constexpr float kZeroResidual = 9.094947017729282e-13f;  // 2^-40
__device__ __forceinline__ bool residual_empty(df Z) { return !(Z.hi > kZeroResidual); }

// Running sum with the error term kept apart; normalise with df_norm.
__device__ __forceinline__ void acc_add(df& acc, float v) {
    df s = two_sum(acc.hi, v);
    acc.hi = s.hi;
    acc.lo = __fadd_rn(acc.lo, s.lo);
}
__device__ __forceinline__ void acc_add(df& acc, df v) {
    df s = two_sum(acc.hi, v.hi);
    acc.hi = s.hi;
    acc.lo = __fadd_rn(acc.lo, __fadd_rn(s.lo, v.lo));
}
__device__ __forceinline__ df df_norm(df a) { return fast_two_sum(a.hi, a.lo); }

__device__ __forceinline__ df shfl_xor_df(df v, int o) {
    return df{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
}
__device__ __forceinline__ df shfl_up_df(df v, int o) {
    return df{__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
}
__device__ __forceinline__ df shfl_df(df v, int src) {
    return df{__shfl_sync(0xffffffffu, v.hi, src), __shfl_sync(0xffffffffu, v.lo, src)};
}

// ------------------------------------------------------------ constants
// ln 2 and log2(e) as float pairs (hi = nearest float, lo = remainder).
constexpr double kLn2D = 0.69314718055994530941723212145818;
constexpr double kLog2eD = 1.4426950408889634073599246810019;
constexpr float kLn2Hi = (float)kLn2D;
constexpr float kLn2Lo = (float)(kLn2D - (double)(float)kLn2D);
constexpr float kHeavyExp = -13.0f;  // weights above 2^-13 of the row maximum are evaluated in double-float

// k = log2(e) / T as a float pair, by float arithmetic only (the GPU's
// float64 rate is low): q = fl(L_hi / T), then the remainder L - q T, exact
// by FMA up to L_lo, divided by T gives the low part.
constexpr float kLog2eHi = (float)kLog2eD;
constexpr float kLog2eLo = (float)(kLog2eD - (double)(float)kLog2eD);
__device__ __forceinline__ df k_of_temperature(float T) {
    const float q = __fdiv_rn(kLog2eHi, T);
    const float r = __fadd_rn(__fmaf_rn(-q, T, kLog2eHi), kLog2eLo);
    return fast_two_sum(q, __fdiv_rn(r, T));
}

// The same k as a pair whose low part is positive (at least the smallest
// normal float), for the weights of the residual draw: then (l - m) * hi +
// (l - m) * lo is -inf rather than NaN for a logit of -inf, with no separate
// test. The pair still equals k to within about 2^-47 of k (one rounding of
// the low part). k.hi > 0.
__device__ __forceinline__ df k_pos_lo(df k) {
    float hi = k.hi, lo = k.lo;
    if (!(lo > 0.f)) {
        const float h2 = __int_as_float(__float_as_int(hi) - 1);  // the float below hi
        lo = __fadd_rn(lo, __fsub_rn(hi, h2));                  // hi - h2 is exact
        hi = h2;
    }
    return df{hi, fmaxf(lo, 1.17549435e-38f)};
}

// Table 2^(i/64), i = 0..63, as float pairs.
using Exp2Table = Exp2Pairs;
static __device__ __noinline__ void exp2_table_init(Exp2Table& t) {
    for (int i = threadIdx.x; i < 64; i += blockDim.x) {
        const double v = exp2((double)i / 64.0);
        const float h = (float)v;
        t.hi[i] = h;
        t.lo[i] = (float)(v - (double)h);
    }
}

// 2^(xh + xl) in double-float for |xh| < 2^16 (the heavy range is [-13, ~0]).
// The out-of-line exp2_df below is the one most call sites use: heavy
// weights are rare, and inlining this at every call site would overflow the
// instruction cache. A site that evaluates heavy columns in one place of its
// own (already out of line) uses the inline body directly.
__device__ __forceinline__ df exp2_df_inline(float xh, float xl, const Exp2Table& tab) {
    const float t = rintf(xh * 64.0f);                  // x = t/64 + r
    const int ti = (int)t;
    const int i = ti & 63;
    const int n = ti >> 6;                              // floor(t / 64)
    const float rh = __fmaf_rn(t, -0.015625f, xh);      // exact: |rh| <= 1/128
    // a = (rh + xl) * ln2 as a pair
    df a = two_prod(rh, kLn2Hi);
    a.lo = __fadd_rn(a.lo, __fmaf_rn(rh, kLn2Lo, __fmul_rn(xl, kLn2Hi)));
    // e^a - 1 = a + a^2 (1/2 + a (1/6 + a/24)), |a| < 0.0055
    const float a2 = __fmul_rn(a.hi, a.hi);
    const float poly = __fmul_rn(a2, __fmaf_rn(a.hi, __fmaf_rn(a.hi, 1.0f / 24.0f, 1.0f / 6.0f), 0.5f));
    df e = fast_two_sum(1.0f, a.hi);
    e.lo = __fadd_rn(e.lo, __fadd_rn(a.lo, poly));
    df w = df_mul(df{tab.hi[i], tab.lo[i]}, e);
    const float sc = __int_as_float((n + 127) << 23);   // 2^n, n in [-126, 127] here
    return df{__fmul_rn(w.hi, sc), __fmul_rn(w.lo, sc)};
}
static __device__ __noinline__ df exp2_df(float xh, float xl, const Exp2Table& tab) {
    return exp2_df_inline(xh, xl, tab);
}

// Mean relative error of the SFU's 2^x over the light range x <= -13,
// measured on GB300 (-5.1e-8, std 3.0e-8). A single fp32 weight cannot carry
// a correction that small (it is under half an ulp), so light weights are
// used as the SFU returns them and the correction is applied to their fp32
// sums, which join double-float sums as (s, s * kEx2LightBias). A GPU test
// re-measures the mean error of corrected sums against exact 2^x.
constexpr float kEx2LightBias = 5.1e-8f;
__device__ __forceinline__ float light_exp2(float x) { return ex2(x); }
__device__ __forceinline__ df light_sum_df(float s, float bias) { return df{s, __fmul_rn(s, bias)}; }

// 2^((dh + dl) * k) in double-float, the exponent carried as a pair.
template <bool INL>
__device__ __forceinline__ df heavy_weight_t(float dh, float dl, df k, const Exp2Table& tab) {
    const float xh = __fmul_rn(dh, k.hi);
    float xl = __fmaf_rn(dh, k.hi, -xh);
    xl = __fmaf_rn(dh, k.lo, xl);
    xl = __fmaf_rn(dl, k.hi, xl);
    return INL ? exp2_df_inline(xh, xl, tab) : exp2_df(xh, xl, tab);
}
static __device__ __noinline__ df heavy_weight(float dh, float dl, df k, const Exp2Table& tab) {
    return heavy_weight_t<false>(dh, dl, k, tab);
}

// Weight of one logit relative to the row maximum: 2^((l - lmax) * k).
// Light weights (exponent <= -13) are the SFU's 2^x of the exponent rounded
// once to fp32 (fma of the float-pair product); their errors stay below 2e-7
// relative and average out in the sums. Heavy weights carry the exponent as a
// pair (for fp32 logits, l - lmax itself is carried as a pair) and go through
// the double-float exp2.
// INL: the heavy path inline (for sites that are themselves out of line).
template <bool FP32IN, bool INL = false>
__device__ __forceinline__ df logit_weight(float l, float lmax, df k, const Exp2Table& tab) {
    const float dh = __fsub_rn(l, lmax);
    if (!(dh > -INFINITY)) return df{0.f, 0.f};  // -inf logits (and masked columns) weigh nothing
    float dl = 0.f;
    if constexpr (FP32IN) dl = two_sum(l, -lmax).lo;  // fp32 logits: l - lmax exactly, as a pair
    const float x = __fmaf_rn(dh, k.hi, __fmaf_rn(dl, k.hi, __fmul_rn(dh, k.lo)));
    if (!(x > kHeavyExp)) return df{light_exp2(x), 0.f};
    if constexpr (INL) return heavy_weight_t<true>(dh, dl, k, tab);
    return heavy_weight(dh, dl, k, tab);
}

static __device__ __noinline__ df resid_weight_df(df a, df b, df It, df Id) {
    df d = df_sub(df_mul(a, It), df_mul(b, Id));
    return df_pos(d) ? d : df{0.f, 0.f};
}

// Light-path weight 2^((l - lmax) k) as one float, and whether the weight is
// heavy (then the float is not used: the caller evaluates it with
// heavy_logit_weight). Branch-free: -inf logits clamp to a huge negative
// exponent, whose 2^x is 0.
template <bool FP32IN>
__device__ __forceinline__ float light_weight(float l, float lmax, df k, bool& heavy) {
    const float dh = fmaxf(__fsub_rn(l, lmax), -1e30f);
    float lo = __fmul_rn(dh, k.lo);
    if constexpr (FP32IN) lo = __fmaf_rn((dh > -1e30f) ? two_sum(l, -lmax).lo : 0.f, k.hi, lo);
    const float x = __fmaf_rn(dh, k.hi, lo);
    heavy = x > kHeavyExp;
    return light_exp2(x);
}

// The double-float weight of a heavy logit (INL: the exp2 inline).
template <bool FP32IN, bool INL = false>
__device__ __forceinline__ df heavy_logit_weight(float l, float lmax, df k, const Exp2Table& tab) {
    const float dh = __fsub_rn(l, lmax);
    const float dl = FP32IN ? two_sum(l, -lmax).lo : 0.f;
    if constexpr (INL) return heavy_weight_t<true>(dh, dl, k, tab);
    return heavy_weight(dh, dl, k, tab);
}

// Residual weight of one column: max(0, Wt * It - Wd * Id).
__device__ __forceinline__ df resid_weight(df a, df b, df It, df Id) {
    if (a.lo == 0.f && b.lo == 0.f) {
        // both weights light (single floats): the difference of two small
        // products, each rounded once
        const float p = __fmaf_rn(a.hi, It.hi, __fmul_rn(a.hi, It.lo));
        const float q = __fmaf_rn(b.hi, Id.hi, __fmul_rn(b.hi, Id.lo));
        const float r = __fsub_rn(p, q);
        return df{r > 0.f ? r : 0.f, 0.f};
    }
    return resid_weight_df(a, b, It, Id);
}

}  // namespace specv
