// Elementwise PPO / dual-clip / decoupled-TIS losses and mismatch statistics on per-token
// log-probabilities ("Rollout Correction Methods": standard, bypass and decoupled
// 3-policy PPO, "Mismatch Metrics"; "10-KL-clip-entropy" section 2: clip, dual clip,
// pg_clipfrac / ppo_kl / pg_clipfrac_lower; "IPO (INTELLECT Policy Optimization)",
// "Choosing eps": masked fraction vs eps against the IcePop ratio band).
//
// Every count predicate must equal the exact predicate on the fp32 inputs (the oracle's
// fp64 evaluation).  Decisions are taken in fp32; a token whose fp32 value lies within
// 1e-5 (relative to max(1, |threshold|)) of a threshold is re-decided exactly.  fp64 is a
// slow pipe on this part, so the exact decisions use float-float arithmetic instead:
//   * a ratio against a threshold, e^x > t, is x > ln t with x = a - b formed exactly as a
//     float-float pair and ln t prepared on the host as one;
//   * the IPO curve's |e^lo - e^ls| > eps evaluates both exponentials in float-float
//     (about 2^-46 relative: Tang's table-driven method, a reduction by ln2/64 in three
//     parts and a degree-5 Taylor polynomial), built on the error-free TwoSum (Knuth) and
//     FMA TwoProduct.
//
//  1. policy_fast_kernel   one streaming pass, two tokens per thread and round with the
//                          next round's loads in flight (registers), branch-free fp32
//                          math, thresholds and their bands prepared on the host, the IPO
//                          curve as a per-thread histogram over the sorted eps (binary
//                          search; only the two neighbouring eps are band-checked).  A token
//                          inside a band goes to its block's list in shared memory (or, if
//                          that is full, to a global spill list); after its loop the block
//                          takes its listed tokens with exact decisions (outputs rewritten,
//                          contributions added in 2^-16 fixed point, exact and so
//                          independent of the list order) and writes its partial.
//  2. policy_slow_kernel   the whole pass with exact decisions in the bands, for inputs the
//                          fast pass does not take (odd length, unaligned, T >= 2^31).
//  3. policy_final_kernel  one block of 1024 threads: the spill list's tokens, then the
//                          block partials in fixed order into the metrics.  If the spill
//                          list overflowed, it redoes the whole batch with exact decisions
//                          instead (slow, correct).
//
// Results are bitwise reproducible for a given device and T.
#include <cmath>
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace rl {

constexpr int kPgThreads = 256;
constexpr int kPgSums = 6;
constexpr int kPgCounts = 6 + RL_PG_MAX_CURVE;
constexpr int kPgFields = kPgSums + kPgCounts;
constexpr int kPgBins = RL_PG_MAX_CURVE + 1;
constexpr int kPgFastPerSm = 4;   // resident blocks per SM of the fast pass
constexpr int kPgSlowPerSm = 2;
constexpr float kPgFix = 65536.f;   // 2^16: fixed-point scale of the band-token sums
constexpr int kPgBlockBand = 1024;  // band tokens a fast-pass block keeps in shared memory
constexpr int kPgBandRows = 64;     // band tokens taken per step (one shared-memory row each)
constexpr int kPgFinalThreads = 1024;

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
__device__ __constant__ float kExp2Hi[64] = {
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
__device__ __constant__ float kExp2Lo[64] = {
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

// ----------------------------------------------------------------------------------
// Parameters
// ----------------------------------------------------------------------------------
// Thresholds and band half-widths prepared on the host; ln of each ratio threshold as a
// float-float pair (-inf for a threshold <= 0); the curve eps sorted ascending with perm
// mapping sorted position -> caller's index.
struct PgPrep {
    float lo_b, hi_b, cc, tis, ice_lo, ice_hi;
    float w_lo_b, w_hi_b, w_cc, w_tis, w_ice_lo, w_ice_hi;
    FF ln_lo_b, ln_hi_b, ln_cc, ln_tis, ln_ice_lo, ln_ice_hi;
    int n;
    float eps[RL_PG_MAX_CURVE];
    float weps[RL_PG_MAX_CURVE];
    int perm[RL_PG_MAX_CURVE];
};

struct PgArgs {
    const float* lt;
    const float* lo;
    const float* ls;
    const float* adv;
    const uint8_t* mask;
    int64_t T;
    rl_pg_params p;
    PgPrep q;
    float* loss_ppo;
    float* loss_dec;
    float* grad_ppo;
    float* grad_dec;
    float* psum;                  // block partials, field-major: psum[k * nb + block]
    int* pcnt;                    // pcnt[k * nb + block]
    int nb;                       // blocks of the pass that wrote them
    int64_t rot_step;             // per-round rotation of the thread -> slot map (warp-aligned)
    int* count;                   // global spill list: length (may exceed cap: overflow)
    int* list;
    int cap;
    rl_pg_metrics* metrics;       // or nullptr
};

struct PgAcc {
    float sum[kPgSums];
    int cnt[kPgCounts];   // valid, clip, dual-clip, icepop low / high, tis truncated, curve[caller's k]
};


RL_DEVINL void pg_zero(PgAcc& acc) {
#pragma unroll
    for (int k = 0; k < kPgSums; ++k) acc.sum[k] = 0.f;
#pragma unroll
    for (int k = 0; k < kPgCounts; ++k) acc.cnt[k] = 0;
}

RL_DEVINL bool near(float x, float thr) { return fabsf(x - thr) <= 1e-5f * fmaxf(1.f, fabsf(thr)); }

// e^x as 2^(x log2 e) on the hardware EX2 unit: relative error about 2^-22 plus the rounding
// of x log2 e (|x| < 25 here: under 2e-6), well inside the 1e-5 bands around thresholds.
RL_DEVINL float exp_fast(float x) { return exp2_approx(x * kLog2e); }

// ----------------------------------------------------------------------------------
// Exact decisions
// ----------------------------------------------------------------------------------
struct PgExact {
    bool clip, dual, tis_trunc, ice_lo, ice_hi;
    unsigned curve;   // bit k: |p_old - p_samp| > curve_eps[k] (caller's order)
};

// With x = lp_theta - lp_old and d = lp_old - lp_samp exact:
//   clip    (l2 > l1):         A > 0 and x > ln(1 + high), or A < 0 and x < ln(1 - low)
//   dual    (A < 0, l3 < lc):  A < 0 and x > ln c           (c > 1 >= 1 - low)
//   tis / icepop:              d against ln tis_upper, ln low, ln high
//   curve:                     |e^lo - e^ls| > eps_k (both exponentials in float-float)
RL_DEVINL PgExact pg_exact(float lt, float lo, float ls, float A, const PgPrep& q) {
    PgExact e;
    const FF x = two_sum(lt, -lo);
    const FF d = two_sum(lo, -ls);
    e.clip = (A > 0.f && ff_gt(x, q.ln_hi_b)) || (A < 0.f && ff_lt(x, q.ln_lo_b));
    e.dual = A < 0.f && ff_gt(x, q.ln_cc);
    e.tis_trunc = ff_gt(d, q.ln_tis);
    e.ice_lo = ff_lt(d, q.ln_ice_lo);
    e.ice_hi = ff_gt(d, q.ln_ice_hi);
    const FF eo = exp_ff(lo), es = exp_ff(ls);
    FF diff = ff_add(eo, {-es.hi, -es.lo});
    if (diff.hi < 0.f) diff = {-diff.hi, -diff.lo};
    e.curve = 0u;
    for (int k = 0; k < q.n; ++k)
        if (ff_gt(diff, {q.eps[k], 0.f})) e.curve |= 1u << q.perm[k];
    return e;
}

// One token of the exact path (slow pass, band tokens): fp32 values and decisions, the
// decisions re-taken exactly when some value lies inside a band.  Adds to acc.
RL_DEVINL void pg_token(float lt, float lo, float ls, float A, bool valid, const PgPrep& q, float& out_lp,
                        float& out_ld, float& out_gp, float& out_gd, PgAcc& acc) {
    if (!valid) {
        out_lp = out_ld = out_gp = out_gd = 0.f;
        return;
    }
    const float r = exp_fast(lt - lo);
    const float l1 = -A * r;
    const float l2 = -A * fminf(fmaxf(r, q.lo_b), q.hi_b);
    const float lc = fmaxf(l1, l2);
    const float l3 = -A * q.cc;
    // decided on the ratio (the sign of A alone picks the side), so a tiny |A| does not
    // put the token in a band: l2 > l1 <=> (A > 0, r > 1 + high) or (A < 0, r < 1 - low);
    // A < 0 and l3 < lc <=> A < 0 and r > c (c > 1 >= 1 - low)
    bool dual = (A < 0.f) && (r > q.cc);
    bool clip = (A > 0.f && r > q.hi_b) || (A < 0.f && r < q.lo_b);
    const float d = lo - ls;
    const float rho_raw = exp_fast(d);
    bool tis_trunc = rho_raw > q.tis;
    bool ice_lo = rho_raw < q.ice_lo;
    bool ice_hi = rho_raw > q.ice_hi;
    const float adiff = fabsf(exp_fast(lo) - exp_fast(ls));
    unsigned curve = 0u;
    bool band = (A < 0.f && (near(r, q.lo_b) || near(r, q.cc))) || (A > 0.f && near(r, q.hi_b)) || near(rho_raw, q.tis) ||
                near(rho_raw, q.ice_lo) || near(rho_raw, q.ice_hi);
    for (int k = 0; k < q.n; ++k) {
        if (adiff > q.eps[k]) curve |= 1u << q.perm[k];
        band = band || near(adiff, q.eps[k]);
    }
    if (band) {
        const PgExact e = pg_exact(lt, lo, ls, A, q);
        clip = e.clip;
        dual = e.dual;
        tis_trunc = e.tis_trunc;
        ice_lo = e.ice_lo;
        ice_hi = e.ice_hi;
        curve = e.curve;
    }
    // branch choices follow the exact decisions above: the clipped branch has no
    // gradient, the dual-clip cap has none either
    const float loss_ppo = dual ? l3 : lc;
    const float g_c = clip ? 0.f : -A * r;
    const float rho = fminf(rho_raw, q.tis);
    out_lp = loss_ppo;
    out_ld = rho * lc;
    out_gp = dual ? 0.f : g_c;
    out_gd = rho * g_c;
    acc.sum[0] += loss_ppo;
    acc.sum[1] += rho * lc;
    acc.sum[2] += lo - lt;
    acc.sum[3] += ls - lo;
    acc.sum[4] += rho_raw - d - 1.f;
    acc.sum[5] += rho;
    acc.cnt[0] += 1;
    acc.cnt[1] += clip ? 1 : 0;
    acc.cnt[2] += dual ? 1 : 0;
    acc.cnt[3] += ice_lo ? 1 : 0;
    acc.cnt[4] += ice_hi ? 1 : 0;
    acc.cnt[5] += tis_trunc ? 1 : 0;
#pragma unroll
    for (int k = 0; k < RL_PG_MAX_CURVE; ++k) acc.cnt[6 + k] += (curve >> k) & 1u;
}

// Every token of [tid, T) with stride nthreads on the exact path (scalar loads, any
// alignment and length); outputs written.
RL_DEVINL void pg_exact_pass(const PgArgs& a, int64_t tid, int64_t nthreads, PgAcc& acc) {
    for (int64_t i = tid; i < a.T; i += nthreads) {
        float lp, ld, gp, gd;
        pg_token(a.lt[i], a.lo[i], a.ls[i], a.adv[i], a.mask[i] != 0, a.q, lp, ld, gp, gd, acc);
        if (a.loss_ppo) a.loss_ppo[i] = lp;
        if (a.loss_dec) a.loss_dec[i] = ld;
        if (a.grad_ppo) a.grad_ppo[i] = gp;
        if (a.grad_dec) a.grad_dec[i] = gd;
    }
}

// ----------------------------------------------------------------------------------
// Reductions
// ----------------------------------------------------------------------------------
// Fixed-order block reduction of the per-thread accumulators (any block size up to 1024):
// warp trees (fp32 sums, exact int32 counts), then one thread per field adds the warps in
// order (no fp64: it is a slow pipe on this part).  Results in sums[] / cnts[] (shared).
RL_DEVINL void pg_block_reduce(const PgAcc& acc, float* sums, int* cnts) {
    __shared__ float shs[32][kPgSums];
    __shared__ int shc[32][kPgCounts];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int k = 0; k < kPgSums; ++k) {
        const float v = warp_sum(acc.sum[k]);
        if (lane == 0) shs[warp][k] = v;
    }
#pragma unroll
    for (int k = 0; k < kPgCounts; ++k) {
        const int v = __reduce_add_sync(0xffffffffu, acc.cnt[k]);
        if (lane == 0) shc[warp][k] = v;
    }
    __syncthreads();
    const int k = threadIdx.x;
    if (k < kPgSums) {
        float v = 0.f;
        for (int w = 0; w < nw; ++w) v += shs[w][k];
        sums[k] = v;
    } else if (k < kPgFields) {
        int v = 0;
        for (int w = 0; w < nw; ++w) v += shc[w][k - kPgSums];
        cnts[k - kPgSums] = v;
    }
    __syncthreads();
}

RL_DEVINL void pg_write_metric(int k, double s, rl_pg_metrics* out) {
    switch (k) {
        case 0: out->loss_ppo = s; break;
        case 1: out->loss_dec = s; break;
        case 2: out->ppo_kl = s; break;
        case 3: out->mis_kl = s; break;
        case 4: out->k3 = s; break;
        case 5: out->tis_sum = s; break;
        case 6: out->n_valid = static_cast<int64_t>(s); break;
        case 7: out->n_clip = static_cast<int64_t>(s); break;
        case 8: out->n_clip_lower = static_cast<int64_t>(s); break;
        case 9: out->icepop_low = static_cast<int64_t>(s); break;
        case 10: out->icepop_high = static_cast<int64_t>(s); break;
        case 11: out->n_tis_trunc = static_cast<int64_t>(s); break;
        default: out->ipo_curve[k - 12] = static_cast<int64_t>(s); break;
    }
}

// Exact-path tokens list[0, n), kPgBandRows at a time (thread i < kPgBandRows takes one
// and fills its shared-memory row: sums in 2^-16 fixed point, counts), then thread
// k < kPgFields adds column k into fix[k] (shared).  Integer sums are exact, so the order
// of the list does not matter.  Outputs of the listed tokens are rewritten.  Called by
// every thread of the block.
__device__ __noinline__ void pg_band_tokens(const PgArgs& a, const int* list, int n, long long* fix) {
    __shared__ long long rows[kPgBandRows][kPgFields];
    for (int c0 = 0; c0 < n; c0 += kPgBandRows) {
        if (threadIdx.x < kPgBandRows) {
            long long* row = rows[threadIdx.x];
            const int e = c0 + threadIdx.x;
            if (e < n) {
                const int64_t t = list[e];
                PgAcc one;
                pg_zero(one);
                float lp, ld, gp, gd;
                pg_token(a.lt[t], a.lo[t], a.ls[t], a.adv[t], true, a.q, lp, ld, gp, gd, one);
                if (a.loss_ppo) a.loss_ppo[t] = lp;
                if (a.loss_dec) a.loss_dec[t] = ld;
                if (a.grad_ppo) a.grad_ppo[t] = gp;
                if (a.grad_dec) a.grad_dec[t] = gd;
                for (int f = 0; f < kPgSums; ++f) row[f] = __float2ll_rn(one.sum[f] * kPgFix);
                for (int f = 0; f < kPgCounts; ++f) row[kPgSums + f] = one.cnt[f];
            } else {
                for (int f = 0; f < kPgFields; ++f) row[f] = 0;
            }
        }
        __syncthreads();
        if (threadIdx.x < kPgFields) {
            long long v = 0;
            for (int r = 0; r < kPgBandRows; ++r) v += rows[r][threadIdx.x];
            fix[threadIdx.x] += v;
        }
        __syncthreads();
    }
}

// ----------------------------------------------------------------------------------
// Slow pass
// ----------------------------------------------------------------------------------
__global__ void __launch_bounds__(kPgThreads, kPgSlowPerSm) policy_slow_kernel(PgArgs a) {
    PgAcc acc;
    pg_zero(acc);
    pg_exact_pass(a, static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x,
                  static_cast<int64_t>(gridDim.x) * blockDim.x, acc);
    __shared__ float sums[kPgSums];
    __shared__ int cnts[kPgCounts];
    pg_block_reduce(acc, sums, cnts);
    const int k = threadIdx.x;
    if (k < kPgSums)
        a.psum[k * a.nb + blockIdx.x] = sums[k];
    else if (k < kPgFields)
        a.pcnt[(k - kPgSums) * a.nb + blockIdx.x] = cnts[k - kPgSums];
}

// ----------------------------------------------------------------------------------
// Fast pass
// ----------------------------------------------------------------------------------
struct PgTok {
    float lp, ld, gp, gd;          // outputs
    float s[kPgSums];              // metric sum terms
    int clip, dual, ice_lo, ice_hi, tis;
    int j;                         // number of sorted eps below |p_old - p_samp|
    bool band;                     // some value lies inside a threshold's band
};

// One token, fp32 decisions, no branches (the tokens of a round interleave freely).
// |p_old - p_samp| = p_samp |rho - 1| with rho = e^(lp_old - lp_samp) (one EX2 less).
RL_DEVINL PgTok pg_fast(float lt, float lo, float ls, float A, const PgPrep& q) {
    PgTok o;
    const float r = exp_fast(lt - lo);
    const float l1 = -A * r;
    const float l2 = -A * fminf(fmaxf(r, q.lo_b), q.hi_b);
    const float lc = fmaxf(l1, l2);
    const float l3 = -A * q.cc;
    const float d = lo - ls;
    const float rho_raw = exp_fast(d);
    const float adiff = exp_fast(ls) * fabsf(rho_raw - 1.f);
    int j = 0;
#pragma unroll
    for (int step = 8; step >= 1; step >>= 1)
        j = (j + step <= q.n && q.eps[j + step - 1] < adiff) ? j + step : j;
    const int jl = j > 0 ? j - 1 : 0, jh = j < q.n ? j : 0;
    o.band = ((A < 0.f) & ((fabsf(r - q.lo_b) <= q.w_lo_b) | (fabsf(r - q.cc) <= q.w_cc))) |
             ((A > 0.f) & (fabsf(r - q.hi_b) <= q.w_hi_b)) |
             (fabsf(rho_raw - q.tis) <= q.w_tis) | (fabsf(rho_raw - q.ice_lo) <= q.w_ice_lo) |
             (fabsf(rho_raw - q.ice_hi) <= q.w_ice_hi) | ((j > 0) & (fabsf(adiff - q.eps[jl]) <= q.weps[jl])) |
             ((j < q.n) & (fabsf(adiff - q.eps[jh]) <= q.weps[jh]));
    const bool dual = (A < 0.f) & (r > q.cc);   // on the ratio, as in pg_token
    const bool clip = ((A > 0.f) & (r > q.hi_b)) | ((A < 0.f) & (r < q.lo_b));
    const float loss_ppo = dual ? l3 : lc;
    const float g_c = clip ? 0.f : -A * r;
    const float rho = fminf(rho_raw, q.tis);
    o.lp = loss_ppo;
    o.ld = rho * lc;
    o.gp = dual ? 0.f : g_c;
    o.gd = rho * g_c;
    o.s[0] = loss_ppo;
    o.s[1] = rho * lc;
    o.s[2] = lo - lt;
    o.s[3] = ls - lo;
    o.s[4] = rho_raw - d - 1.f;
    o.s[5] = rho;
    o.clip = clip;
    o.dual = dual;
    o.ice_lo = rho_raw < q.ice_lo;
    o.ice_hi = rho_raw > q.ice_hi;
    o.tis = rho_raw > q.tis;
    o.j = j;
    return o;
}

struct PgFastAcc {
    float sum[kPgSums];
    int cnt[6];
};

// Take one token's values unless it is masked out or in a band (then outputs are 0 here;
// a band token goes to the list).
RL_DEVINL void pg_take(const PgTok& t, bool valid, int* hist, PgFastAcc& acc, float& lp, float& ld, float& gp,
                       float& gd) {
    const bool use = valid & !t.band;
    const float f = use ? 1.f : 0.f;
    lp = use ? t.lp : 0.f;
    ld = use ? t.ld : 0.f;
    gp = use ? t.gp : 0.f;
    gd = use ? t.gd : 0.f;
#pragma unroll
    for (int k = 0; k < kPgSums; ++k) acc.sum[k] = fmaf(f, t.s[k], acc.sum[k]);
    const int u = use;
    acc.cnt[0] += u;
    acc.cnt[1] += u & t.clip;
    acc.cnt[2] += u & t.dual;
    acc.cnt[3] += u & t.ice_lo;
    acc.cnt[4] += u & t.ice_hi;
    acc.cnt[5] += u & t.tis;
    hist[t.j * kPgThreads] += u;
}

RL_DEVINL void pg_append(const PgArgs& a, int64_t t) {
    const int s = atomicAdd(a.count, 1);
    if (s < a.cap) a.list[s] = static_cast<int>(t);
}

// Two tokens per thread and round; rounds of nthreads pairs with a warp-aligned rotation
// (rot_step) so a thread does not meet the same position of a padded sequence layout in
// every round (a grid stride that is a multiple of the padding period would give some
// threads only valid tokens and others only padding).  The next round's inputs are
// loaded before this round's math.
__global__ void __launch_bounds__(kPgThreads, kPgFastPerSm) policy_fast_kernel(PgArgs a) {
    __shared__ int hist_s[kPgBins * kPgThreads];   // bin-major: thread t's bin b at b * 256 + t
    __shared__ int blist[kPgBlockBand];            // this block's band tokens
    __shared__ int bcount;
    __shared__ long long bfix[kPgFields];
    for (int b = 0; b <= a.q.n; ++b) hist_s[b * kPgThreads + threadIdx.x] = 0;
    if (threadIdx.x == 0) bcount = 0;
    if (threadIdx.x < kPgFields) bfix[threadIdx.x] = 0;
    __syncthreads();
    int* hist = hist_s + threadIdx.x;
    auto band = [&](int64_t t) {
        const int s = atomicAdd(&bcount, 1);
        if (s < kPgBlockBand)
            blist[s] = static_cast<int>(t);
        else
            pg_append(a, t);   // spill to the global list (the last block takes it)
    };
    PgFastAcc acc;
#pragma unroll
    for (int k = 0; k < kPgSums; ++k) acc.sum[k] = 0.f;
#pragma unroll
    for (int k = 0; k < 6; ++k) acc.cnt[k] = 0;
    const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t n2 = a.T / 2;
    int64_t rot = 0;
    auto next = [&](int64_t base) -> int64_t {
        int64_t idx = tid + rot;
        if (idx >= nthreads) idx -= nthreads;
        rot += a.rot_step;
        if (rot >= nthreads) rot -= nthreads;
        return base + idx;
    };
    float2 lt = make_float2(0.f, 0.f), lo = lt, ls = lt, A = lt;
    uchar2 m = make_uchar2(0, 0);
    auto load = [&](int64_t k) {
        if (k < n2) {
            lt = __ldcs(reinterpret_cast<const float2*>(a.lt) + k);
            lo = __ldcs(reinterpret_cast<const float2*>(a.lo) + k);
            ls = __ldcs(reinterpret_cast<const float2*>(a.ls) + k);
            A = __ldcs(reinterpret_cast<const float2*>(a.adv) + k);
            m = __ldcs(reinterpret_cast<const uchar2*>(a.mask) + k);
        }
    };
    int64_t i = next(0);
    load(i);
    for (int64_t base = 0; base < n2; base += nthreads) {
        const float2 clt = lt, clo = lo, cls = ls, cA = A;
        const uchar2 cm = m;
        const int64_t ci = i;
        i = next(base + nthreads);
        load(i);
        if (ci >= n2) continue;
        float2 lp = make_float2(0.f, 0.f), ld = lp, gp = lp, gd = lp;
        if ((cm.x | cm.y) != 0) {
            const PgTok tx = pg_fast(clt.x, clo.x, cls.x, cA.x, a.q);
            const PgTok ty = pg_fast(clt.y, clo.y, cls.y, cA.y, a.q);
            pg_take(tx, cm.x != 0, hist, acc, lp.x, ld.x, gp.x, gd.x);
            pg_take(ty, cm.y != 0, hist, acc, lp.y, ld.y, gp.y, gd.y);
            if ((cm.x != 0) & tx.band) band(2 * ci);
            if ((cm.y != 0) & ty.band) band(2 * ci + 1);
        }
        if (a.loss_ppo) __stcs(reinterpret_cast<float2*>(a.loss_ppo) + ci, lp);
        if (a.loss_dec) __stcs(reinterpret_cast<float2*>(a.loss_dec) + ci, ld);
        if (a.grad_ppo) __stcs(reinterpret_cast<float2*>(a.grad_ppo) + ci, gp);
        if (a.grad_dec) __stcs(reinterpret_cast<float2*>(a.grad_dec) + ci, gd);
    }
    // this block's band tokens on the exact path (few: fp32 float-float work, spread over
    // all blocks), into bfix
    __syncthreads();
    const int nband = bcount < kPgBlockBand ? bcount : kPgBlockBand;
    if (nband > 0) pg_band_tokens(a, blist, nband, bfix);
    // block partial: warp trees (fp32 sums, exact int32 counts), then the 8 warps in order
    // plus the band tokens' terms; the curve counts from the histogram, cnt_k = #(j > k),
    // back in the caller's order
    __shared__ float shs[kPgThreads / 32][kPgSums];
    __shared__ int shc[kPgThreads / 32][6];
    __shared__ int bins[kPgBins];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int k = 0; k < kPgSums; ++k) {
        const float v = warp_sum(acc.sum[k]);
        if (lane == 0) shs[warp][k] = v;
    }
#pragma unroll
    for (int k = 0; k < 6; ++k) {
        const int v = __reduce_add_sync(0xffffffffu, acc.cnt[k]);
        if (lane == 0) shc[warp][k] = v;
    }
    __syncthreads();
    for (int b = warp; b <= a.q.n; b += kPgThreads / 32) {
        int v = 0;
        for (int t = lane; t < kPgThreads; t += 32) v += hist_s[b * kPgThreads + t];
        v = __reduce_add_sync(0xffffffffu, v);
        if (lane == 0) bins[b] = v;
    }
    __syncthreads();
    const int k = threadIdx.x;
    if (k < kPgSums) {
        float v = 0.f;
        for (int w = 0; w < kPgThreads / 32; ++w) v += shs[w][k];
        a.psum[k * a.nb + blockIdx.x] = v + static_cast<float>(bfix[k]) / kPgFix;
    } else if (k < kPgSums + 6) {
        int v = 0;
        for (int w = 0; w < kPgThreads / 32; ++w) v += shc[w][k - kPgSums];
        a.pcnt[(k - kPgSums) * a.nb + blockIdx.x] = v + static_cast<int>(bfix[k]);
    } else if (k < kPgFields) {
        const int c = k - kPgSums - 6;        // caller's curve index
        int v = 0;
        if (c < a.q.n) {
            int js = 0;                        // its sorted position
            while (a.q.perm[js] != c) ++js;
            for (int b = js + 1; b <= a.q.n; ++b) v += bins[b];
        }
        a.pcnt[(k - kPgSums) * a.nb + blockIdx.x] = v + static_cast<int>(bfix[k]);
    }
}

// ----------------------------------------------------------------------------------
// Final reduction
// ----------------------------------------------------------------------------------
__global__ void __launch_bounds__(kPgFinalThreads) policy_final_kernel(PgArgs a) {
    const int cnt = *a.count;
    if (cnt > a.cap) {   // the spill list overflowed: every token again, exact decisions
        PgAcc acc;
        pg_zero(acc);
        pg_exact_pass(a, threadIdx.x, blockDim.x, acc);
        __shared__ float sums[kPgSums];
        __shared__ int cnts[kPgCounts];
        pg_block_reduce(acc, sums, cnts);
        if (a.metrics && threadIdx.x < kPgFields) {
            const int k = threadIdx.x;
            pg_write_metric(k, k < kPgSums ? static_cast<double>(sums[k]) : static_cast<double>(cnts[k - kPgSums]),
                            a.metrics);
        }
        return;
    }
    __shared__ long long fix[kPgFields];
    if (threadIdx.x < kPgFields) fix[threadIdx.x] = 0;
    __syncthreads();
    if (cnt > 0) pg_band_tokens(a, a.list, cnt, fix);
    if (!a.metrics) return;
    // warp k: field k over the partials, lane l adding b = l, l + 32, ... in order
    const int k = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (k >= kPgFields) return;
    double s;
    if (k < kPgSums) {
        float v = 0.f;
        for (int b = lane; b < a.nb; b += 32) v += a.psum[k * a.nb + b];
        s = static_cast<double>(warp_sum(v)) + static_cast<double>(fix[k]) / static_cast<double>(kPgFix);
    } else {
        long long v = 0;
        for (int b = lane; b < a.nb; b += 32) v += a.pcnt[(k - kPgSums) * a.nb + b];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        s = static_cast<double>(v + fix[k]);
    }
    if (lane == 0) pg_write_metric(k, s, a.metrics);
}

// ----------------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------------
// Workspace: a 256-byte header (spill-list length), the block partials (field-major),
// then the spill list in whatever room is left.
struct PgWs {
    int* count;
    float* psum;
    int* pcnt;
    int* list;
    int cap;
};
constexpr size_t kPgHeader = 256;

static int fast_blocks(int sms) { return sms * kPgFastPerSm; }
static int slow_blocks(int sms) { return sms * kPgSlowPerSm; }
static int max_blocks(int sms) { return fast_blocks(sms) > slow_blocks(sms) ? fast_blocks(sms) : slow_blocks(sms); }

static size_t fixed_bytes(int sms) {
    return kPgHeader + align_up(static_cast<size_t>(max_blocks(sms)) * kPgFields * 4, 256);
}

static PgWs pg_ws(void* ws, size_t ws_bytes, int sms) {
    PgWs w;
    uint8_t* b = static_cast<uint8_t*>(ws);
    w.count = reinterpret_cast<int*>(b);
    w.psum = reinterpret_cast<float*>(b + kPgHeader);
    w.pcnt = reinterpret_cast<int*>(w.psum + static_cast<size_t>(max_blocks(sms)) * kPgSums);
    const size_t fixed = fixed_bytes(sms);
    w.list = reinterpret_cast<int*>(b + fixed);
    const size_t room = ws_bytes > fixed ? (ws_bytes - fixed) / sizeof(int) : 0;
    w.cap = room > static_cast<size_t>(INT32_MAX) ? INT32_MAX : static_cast<int>(room);
    return w;
}

size_t policy_ws_need(int64_t T) {
    (void)T;
    return fixed_bytes(num_sms());
}

size_t policy_ws_bytes(int64_t T) {
    // any device up to 256 SMs, and a band list of max(4096, T / 16) entries (the expected
    // share of band tokens is well under 1e-3; an overflow only costs the slow fallback)
    const int64_t list = T / 16 > 4096 ? T / 16 : 4096;
    return align_up(fixed_bytes(256) + static_cast<size_t>(list) * sizeof(int), 256);
}

// ln t as a float-float pair (hi = the float nearest ln t, lo = the float nearest the rest)
static FF ln_ff(double t) {
    if (!(t > 0.0)) return {-INFINITY, 0.f};
    const double l = std::log(t);
    const float hi = static_cast<float>(l);
    return {hi, static_cast<float>(l - static_cast<double>(hi))};
}

static PgPrep prepare(const rl_pg_params& p) {
    PgPrep q{};
    auto band = [](float t) { return 1e-5f * fmaxf(1.f, fabsf(t)); };
    q.lo_b = 1.f - p.clip_ratio_low;
    q.hi_b = 1.f + p.clip_ratio_high;
    q.cc = p.clip_ratio_c;
    q.tis = p.tis_upper;
    q.ice_lo = p.icepop_low;
    q.ice_hi = p.icepop_high;
    q.w_lo_b = band(q.lo_b);
    q.w_hi_b = band(q.hi_b);
    q.w_cc = band(q.cc);
    q.w_tis = band(q.tis);
    q.w_ice_lo = band(q.ice_lo);
    q.w_ice_hi = band(q.ice_hi);
    // the exact thresholds as the definition forms them from the fp32 knobs (1 - low and
    // 1 + high in double, not the fp32 sums the fp32 comparisons use)
    q.ln_lo_b = ln_ff(1.0 - static_cast<double>(p.clip_ratio_low));
    q.ln_hi_b = ln_ff(1.0 + static_cast<double>(p.clip_ratio_high));
    q.ln_cc = ln_ff(static_cast<double>(p.clip_ratio_c));
    q.ln_tis = ln_ff(static_cast<double>(p.tis_upper));
    q.ln_ice_lo = ln_ff(static_cast<double>(p.icepop_low));
    q.ln_ice_hi = ln_ff(static_cast<double>(p.icepop_high));
    q.n = p.n_curve;
    for (int k = 0; k < q.n; ++k) q.perm[k] = k;
    for (int x = 1; x < q.n; ++x)   // stable insertion sort of the indices by eps
        for (int y = x; y > 0 && p.curve_eps[q.perm[y - 1]] > p.curve_eps[q.perm[y]]; --y) {
            const int t = q.perm[y];
            q.perm[y] = q.perm[y - 1];
            q.perm[y - 1] = t;
        }
    for (int k = 0; k < q.n; ++k) {
        q.eps[k] = p.curve_eps[q.perm[k]];
        q.weps[k] = band(q.eps[k]);
    }
    return q;
}

// Warp-aligned rotation per round: about 0.618 of the warps with an odd residue near
// 0.6 x 32 modulo 32 warps, so successive rounds spread over the phases of any
// power-of-two padding period instead of creeping by one warp.
static int64_t rotation(int nb) {
    const int64_t nwarps = static_cast<int64_t>(nb) * (kPgThreads / 32);
    int64_t kw = (nwarps * 618 / 1000) / 32 * 32 + 19;
    while (kw >= nwarps && kw > 0) kw -= 32;
    return (kw < 0 ? 0 : kw) * 32;
}

int policy_impl(const float* lt, const float* lo, const float* ls, const float* adv,
                const uint8_t* mask, int64_t T, const rl_pg_params* p, float* loss_ppo,
                float* loss_dec, float* grad_ppo, float* grad_dec, rl_pg_metrics* metrics,
                void* ws, size_t ws_bytes, cudaStream_t stream) {
    const int sms = num_sms();
    if (ws_bytes < fixed_bytes(sms)) return RL_ERR_WORKSPACE;
    const PgWs w = pg_ws(ws, ws_bytes, sms);
    auto al = [](const void* ptr, uintptr_t n) { return (reinterpret_cast<uintptr_t>(ptr) & (n - 1)) == 0; };
    const bool fast = T % 2 == 0 && T < (int64_t(1) << 31) && al(lt, 8) && al(lo, 8) && al(ls, 8) && al(adv, 8) &&
                      al(mask, 2) && al(loss_ppo, 8) && al(loss_dec, 8) && al(grad_ppo, 8) && al(grad_dec, 8);
    PgArgs a{};
    a.lt = lt;
    a.lo = lo;
    a.ls = ls;
    a.adv = adv;
    a.mask = mask;
    a.T = T;
    a.p = *p;
    a.q = prepare(*p);
    a.loss_ppo = loss_ppo;
    a.loss_dec = loss_dec;
    a.grad_ppo = grad_ppo;
    a.grad_dec = grad_dec;
    a.count = w.count;
    a.list = w.list;
    a.cap = w.cap;
    a.psum = w.psum;
    a.pcnt = w.pcnt;
    a.metrics = metrics;
    ProfScope ps(RL_PROF_POLICY, stream);
    if (cudaMemsetAsync(ws, 0, sizeof(int), stream) != cudaSuccess) return RL_ERR_CUDA;   // spill count
    if (fast) {
        a.nb = fast_blocks(sms);
        a.rot_step = rotation(a.nb);
        policy_fast_kernel<<<a.nb, kPgThreads, 0, stream>>>(a);
    } else {
        a.nb = slow_blocks(sms);
        policy_slow_kernel<<<a.nb, kPgThreads, 0, stream>>>(a);
    }
    policy_final_kernel<<<1, kPgFinalThreads, 0, stream>>>(a);
    count_launch(2);
    return cudaPeekAtLastError() == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}

}  // namespace rl
