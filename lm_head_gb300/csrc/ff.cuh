// Float-float arithmetic for exact threshold decisions on fp32 data: a value is the
// unevaluated sum hi + lo of two floats (|lo| <= ulp(hi) / 2), about 2^-48 relative.
// Built on the error-free transformations TwoSum (Knuth) and FMA TwoProduct; e^x by
// Tang's table-driven method.  fp64 is a slow pipe on this part, so the exact decisions
// of the elementwise paths use this instead.
#pragma once

#include <cmath>

#include "common.cuh"

namespace rl {

// ----------------------------------------------------------------------------------
// Float-float arithmetic (value = hi + lo, |lo| <= ulp(hi) / 2)
// ----------------------------------------------------------------------------------
struct FF {
    float hi, lo;
};
RL_DEVINL FF two_sum(float a, float b) {   // exact: a + b = s + e
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return {s, e};
}
RL_DEVINL FF fast_two_sum(float a, float b) {   // exact when |a| >= |b|
    const float s = __fadd_rn(a, b);
    return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
RL_DEVINL FF two_prod(float a, float b) {   // exact: a * b = p + e
    const float p = __fmul_rn(a, b);
    return {p, fmaf(a, b, -p)};
}
RL_DEVINL FF ff_add(FF a, FF b) {
    const FF s = two_sum(a.hi, b.hi);
    return fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}
RL_DEVINL FF ff_mul(FF a, FF b) {
    const FF p = two_prod(a.hi, b.hi);
    return fast_two_sum(p.hi, fmaf(a.hi, b.lo, fmaf(a.lo, b.hi, p.lo)));
}
RL_DEVINL bool ff_gt(FF a, FF b) { return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo); }
RL_DEVINL bool ff_lt(FF a, FF b) { return ff_gt(b, a); }

// 2^(j/64), j = 0..63, as float-float pairs
static __device__ __constant__ float kExp2Hi[64] = {
    1.000000000e+00f, 1.010889292e+00f, 1.021897197e+00f, 1.033024907e+00f, 1.044273734e+00f, 1.055645227e+00f,
    1.067140460e+00f, 1.078760743e+00f, 1.090507746e+00f, 1.102382541e+00f, 1.114386797e+00f, 1.126521587e+00f,
    1.138788581e+00f, 1.151189208e+00f, 1.163724899e+00f, 1.176396966e+00f, 1.189207077e+00f, 1.202156782e+00f,
    1.215247393e+00f, 1.228480577e+00f, 1.241857767e+00f, 1.255380750e+00f, 1.269050956e+00f, 1.282870054e+00f,
    1.296839595e+00f, 1.310961246e+00f, 1.325236678e+00f, 1.339667559e+00f, 1.354255557e+00f, 1.369002461e+00f,
    1.383909941e+00f, 1.398979664e+00f, 1.414213538e+00f, 1.429613352e+00f, 1.445180774e+00f, 1.460917830e+00f,
    1.476826191e+00f, 1.492907763e+00f, 1.509164453e+00f, 1.525598168e+00f, 1.542210817e+00f, 1.559004426e+00f,
    1.575980902e+00f, 1.593142152e+00f, 1.610490322e+00f, 1.628027439e+00f, 1.645755529e+00f, 1.663676620e+00f,
    1.681792855e+00f, 1.700106382e+00f, 1.718619347e+00f, 1.737333894e+00f, 1.756252170e+00f, 1.775376439e+00f,
    1.794709086e+00f, 1.814252138e+00f, 1.834008098e+00f, 1.853979111e+00f, 1.874167681e+00f, 1.894575953e+00f,
    1.915206552e+00f, 1.936061740e+00f, 1.957144141e+00f, 1.978456020e+00f};
static __device__ __constant__ float kExp2Lo[64] = {
    0.000000000e+00f, -5.711605411e-09f, -4.811559862e-08f, -2.809089317e-08f, 4.833470157e-08f,
    -4.907169426e-08f, -5.933751979e-08f, 5.461594554e-08f, -1.307753994e-08f, 4.260501996e-08f,
    -5.435540018e-08f, 3.123641434e-08f, 5.386222313e-08f, 2.192228266e-08f, -4.051441493e-08f,
    2.566975077e-08f, 3.797635273e-08f, -5.069756526e-08f, -3.267394888e-08f, -4.136200360e-08f,
    4.496838102e-08f, 7.322237483e-09f, 1.419333318e-09f, -3.816621685e-08f, -4.018999533e-08f,
    -3.496571566e-08f, -3.496373324e-08f, -3.461673970e-08f, -1.012334927e-08f, -3.845881835e-08f,
    -5.875577358e-08f, 8.689434061e-09f, 2.420323497e-08f, -1.342992917e-08f, 3.324199938e-08f,
    -3.628657552e-08f, -4.500898854e-08f, -3.423620143e-08f, -2.495937323e-08f, -1.762856883e-08f,
    8.070904833e-09f, -2.576466507e-08f, -5.661025426e-08f, -4.903136785e-10f, 9.836217174e-09f,
    -1.726008314e-08f, -5.124972091e-08f, -3.920298752e-08f, -2.475532668e-08f, -2.865147231e-08f,
    -4.849617596e-08f, -5.850223417e-08f, -9.235770371e-09f, 5.343197884e-08f, -1.141504491e-08f,
    3.736258236e-08f, -1.123927795e-08f, 1.436561181e-08f, -4.663005626e-08f, 2.810338451e-08f,
    9.845328108e-09f, 5.357072297e-08f, -1.702180441e-08f, 6.032726318e-09f};

// e^x (x an fp32 value) as a float-float pair, about 2^-46 relative (Tang's table-driven
// method): x = (64 k + j) ln2/64 + s with ln2/64 = C1 + C2 + C3 (C1, C2 with 10 significant
// bits, so n C1 and n C2 are exact for |n| < 2^14), |s| <= ln2/128; e^s by a degree-5
// Taylor polynomial; e^x = 2^k 2^(j/64) e^s.
RL_DEVINL FF exp_ff(float x) {
    if (x < -103.f) return {0.f, 0.f};
    if (x > 88.f) return {INFINITY, 0.f};
    const float n = rintf(x * 92.33248138427734f);   // 64 / ln 2
    const float C1 = 0.0108184814453125f, C2 = 1.1935830116271973e-05f, C3 = 7.420820402614936e-09f;
    FF r = two_sum(x, -(n * C1));
    r = ff_add(r, {-(n * C2), 0.f});
    r = ff_add(r, two_prod(-n, C3));
    // 1 + s + s^2/2 + s^3/6 + s^4/24 + s^5/120 by Horner (1/6, 1/24, 1/120 as float-float)
    FF p = {8.333333768e-03f, -4.346172033e-10f};
    p = ff_add(ff_mul(p, r), {4.166666791e-02f, -1.241763470e-09f});
    p = ff_add(ff_mul(p, r), {1.666666716e-01f, -4.967053879e-09f});
    p = ff_add(ff_mul(p, r), {0.5f, 0.f});
    p = ff_add(ff_mul(p, r), {1.f, 0.f});
    p = ff_add(ff_mul(p, r), {1.f, 0.f});
    const int ni = static_cast<int>(n);
    const int k = ni >> 6, j = ni - (k << 6);
    p = ff_mul(p, {kExp2Hi[j], kExp2Lo[j]});
    return {ldexpf(p.hi, k), ldexpf(p.lo, k)};
}

// ln t as a float-float pair (host): hi = the float nearest ln t, lo = the float nearest
// the rest; -inf for t <= 0.
inline FF ln_ff(double t) {
    if (!(t > 0.0)) return {-INFINITY, 0.f};
    const double l = std::log(t);
    const float hi = static_cast<float>(l);
    return {hi, static_cast<float>(l - static_cast<double>(hi))};
}

}  // namespace rl
