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
//  1. policy_fast_kernel   one streaming pass: stages of 512 slots dealt round-robin to
//                          the blocks, each block's through a ring of shared-memory stages
//                          that a producer warp fills with bulk copies (cp.async.bulk,
//                          mbarriers); branch-free fp32 math, thresholds and their bands
//                          prepared on the host, the IPO curve as a per-thread histogram
//                          over the sorted eps (binary search; only the two neighbouring
//                          eps are band-checked).  A token inside a band is re-decided
//                          exactly by the thread that met it.
//  1'. policy_packed_kernel the same pass for packed input (no mask): 1024-token stages,
//                          the first few dealt round-robin and the rest claimed by the
//                          blocks as they free a ring slot (so blocks on faster SMs take
//                          more), four tokens per thread, no selects, the curve bin from
//                          a bucket table.
//  2. policy_slow_kernel   the whole pass with exact decisions in the bands, for inputs the
//                          fast passes do not take (unaligned, T >= 2^31).
//  With no mask (packed input: every slot a valid token) the mask is neither read nor
//  copied: 16 bytes in per token instead of 17.
//  Each block adds its partial (fp32 sums in a fixed order within the block, then in 2^-24
//  fixed point; counts) to the batch accumulators with integer atomics, whose total does
//  not depend on the order of arrival.  In the packed pass a thread's fp32 sum over its
//  four tokens of a stage goes into 2^-24 fixed point at once, so the totals do not depend
//  on which block took the stage either.  The last block to arrive (an arrival counter)
//  writes the metrics and sets every accumulator and the counter back to zero, so a
//  workspace zeroed once before its first use needs no clearing before later calls and a
//  call is one kernel launch.  The last block's code is kept short: it runs once, on one
//  SM, with every instruction fetched cold.  If a block's sum was too large for the fixed
//  point, that block redoes the whole batch's metrics with exact decisions (slow, correct).
//
// Results are bitwise reproducible for a given device and T.
#include <atomic>
#include <cmath>
#include <climits>
#include <cstddef>

#include "common.cuh"
#include "ff.cuh"
#include "internal.h"

namespace rl {

constexpr int kPgThreads = 256;
constexpr int kPgSums = 6;
constexpr int kPgCounts = 6 + RL_PG_MAX_CURVE;
constexpr int kPgFields = kPgSums + kPgCounts;
constexpr int kPgBins = RL_PG_MAX_CURVE + 1;
constexpr int kPgFastPerSm = 2;   // resident blocks per SM of the fast pass
constexpr int kPgStageSlots = 2 * kPgThreads;   // token slots per stage of the fast pass
constexpr int kPgDepth = 6;       // stages in its ring
constexpr int kPgSlowPerSm = 2;

// ----------------------------------------------------------------------------------
// Parameters
// ----------------------------------------------------------------------------------
// Thresholds and band half-widths prepared on the host; ln of each ratio threshold as a
// float-float pair (-inf for a threshold <= 0); the curve eps sorted ascending with perm
// mapping sorted position -> caller's index.
constexpr int kPkLut = 256;                    // buckets of |p_old - p_samp| over [0, 1]
struct PgPrep {
    float lo_b, hi_b, cc, tis, ice_lo, ice_hi;
    float w_lo_b, w_hi_b, w_cc, w_tis, w_ice_lo, w_ice_hi;
    FF ln_lo_b, ln_hi_b, ln_cc, ln_tis, ln_ice_lo, ln_ice_hi;
    int n;
    float eps[RL_PG_MAX_CURVE];
    float weps[RL_PG_MAX_CURVE];
    int perm[RL_PG_MAX_CURVE];
    int pos[RL_PG_MAX_CURVE];   // inverse of perm: caller's index -> sorted position
    // the packed pass's bucket table: entry b = (eps below bucket b) | (1 + the one eps
    // inside it, sorted index; 0: none) << 8 | (1: take the exact path) << 16; eps_s / weps_s
    // are eps / weps shifted up by one, entry 0 a sentinel no value is above or near
    int lut[kPkLut];
    float eps_s[RL_PG_MAX_CURVE + 1];
    float weps_s[RL_PG_MAX_CURVE + 1];
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
    long long* acc;               // the batch's sums (2^-24 fixed point) and counts, kPgAccStride apart
    int* range;                   // set when a sum term is too large for the fixed point
    float range_lim;              // |term| bound that keeps every accumulator inside int64
    int32_t* status;              // RL_STATUS_* bits of this call's waits
    unsigned int* arrive;         // blocks of this launch that have added their partial (0 between calls)
    unsigned int* claim;          // stages claimed past the round-robin ones (packed pass; 0 between calls)
    int nb;                       // blocks of the pass
    int curve_bins;               // curve accumulators hold sorted-eps bins 1..n (streaming passes),
                                  // else the curve counts in the caller's order
    uint64_t wait_ns;             // limit of the streaming loop's waits (RL_OPT_WAIT_LIMIT_US)
    rl_pg_metrics* metrics;       // or nullptr
};

constexpr float kPgFix = 16777216.f;   // 2^24: fixed-point scale of the metric sums
constexpr int kPgMaxBlocks = 512;
constexpr int kPgAccStride = 16;       // one 128-byte line per accumulator: the blocks' atomics spread over L2

// The metrics struct read as 8-byte words: the sums (fp64) in field order, then the counts.
static_assert(offsetof(rl_pg_metrics, n_valid) == 8 * kPgSums && offsetof(rl_pg_metrics, ipo_curve) == 8 * 12 &&
                  offsetof(rl_pg_metrics, status) == 8 * kPgFields,
              "rl_pg_metrics layout");

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
    int j;            // how many of the sorted eps lie below |p_old - p_samp|
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
    e.j = 0;
    for (int k = 0; k < q.n; ++k)
        if (ff_gt(diff, {q.eps[k], 0.f})) {
            e.curve |= 1u << q.perm[k];
            ++e.j;
        }
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
        pg_token(a.lt[i], a.lo[i], a.ls[i], a.adv[i], a.mask == nullptr || a.mask[i] != 0, a.q, lp, ld, gp, gd, acc);
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


// ----------------------------------------------------------------------------------
// Batch totals
// ----------------------------------------------------------------------------------
// A sum term in 2^-24 fixed point, or 0 with the range flag raised when |v| is at or past
// the bound that keeps the batch's accumulators inside int64 (or v is not finite).
RL_DEVINL long long pg_fix(const PgArgs& a, float v) {
    if (fabsf(v) < a.range_lim) return __float2ll_rn(v * kPgFix);
    atomicOr(a.range, 1);
    return 0;
}

// The same value as pg_fix, through a 32-bit conversion whenever v 2^24 fits in an int32
// (then |v| < 128, inside the range bound for any T < 2^31, and both conversions round to
// nearest even): the 64-bit conversion is a slow instruction and most terms never need it.
RL_DEVINL long long pg_fix_fast(const PgArgs& a, float v) {
    const float x = v * kPgFix;
    if (fabsf(x) < 2147483648.f) return static_cast<long long>(__float2int_rn(x));
    return pg_fix(a, v);
}

// A block's partial goes into the batch accumulators with integer atomics (sums in 2^-24
// fixed point, counts as they are): integer addition does not depend on the order the
// blocks arrive in, so the totals are reproducible.
RL_DEVINL void pg_add_partial(const PgArgs& a, int k, float sum, long long count) {
    const long long x = k < kPgSums ? pg_fix(a, sum) + count : count;
    if (x != 0)
        atomicAdd(reinterpret_cast<unsigned long long*>(a.acc + k * kPgAccStride), static_cast<unsigned long long>(x));
}

// The last block of the pass to finish: the accumulators into the metrics (a streaming
// pass's curve bins turned into the curve counts, cnt_c = the tokens in the bins above
// eps_c's sorted position), then every accumulator, the flags and the counters back to
// zero.  If a sum term was too large for the fixed point, the whole batch again with exact
// decisions and fp32 sums instead (one block: slow, correct).  Called by every thread of
// the block.
RL_DEVINL void pg_final(const PgArgs& a) {
    const int k = threadIdx.x;
    __shared__ long long tot[kPgFields];
    // the accumulators, the range flag and the status together (one round trip)
    const long long mine =
        k < kPgFields ? static_cast<long long>(__ldcg(reinterpret_cast<const unsigned long long*>(a.acc + k * kPgAccStride)))
                      : 0;
    const bool range = __ldcg(a.range) != 0;
    const int32_t st = __ldcg(a.status);
    long long* out = reinterpret_cast<long long*>(a.metrics);   // see the layout assertion
    if (range) {
        PgAcc acc;
        pg_zero(acc);
        pg_exact_pass(a, threadIdx.x, blockDim.x, acc);
        __shared__ float sums[kPgSums];
        __shared__ int cnts[kPgCounts];
        pg_block_reduce(acc, sums, cnts);
        if (out && k < kPgFields)
            out[k] = k < kPgSums ? __double_as_longlong(static_cast<double>(sums[k])) : cnts[k - kPgSums];
    } else {
        if (k < kPgFields) tot[k] = mine;
        __syncthreads();
        long long v = k < kPgFields ? tot[k] : 0;
        if (k < kPgSums) {
            v = __double_as_longlong(static_cast<double>(v) * (1.0 / kPgFix));
        } else if (k >= kPgSums + 6 && k < kPgFields && a.curve_bins) {
            const int c = k - kPgSums - 6;   // caller's curve index
            v = 0;
            if (c < a.q.n)
                for (int b = a.q.pos[c] + 1; b <= a.q.n; ++b) v += tot[kPgSums + 5 + b];
        }
        if (out && k < kPgFields) out[k] = v;
    }
    if (k == 0 && out) out[kPgFields] = st;
    __syncthreads();   // every read of the accumulators is done
    if (k < kPgFields) a.acc[k * kPgAccStride] = 0;
    if (k == 0) {
        *a.range = 0;
        *a.status = 0;
        *a.claim = 0u;
        *a.arrive = 0u;
    }
}

// Every block calls this after adding its partial; the last one to arrive finishes.  One
// thread counts the block in with an acquire-release atomic after the block's barrier:
// the release makes the block's atomics (ordered before it by the barrier) visible
// before the count, and the acquire, passed on by the second barrier, makes every other
// block's visible to the last block's reads.
RL_DEVINL void pg_finish(const PgArgs& a) {
    __shared__ int last;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned int old;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(a.arrive) : "memory");
        last = old == static_cast<unsigned int>(a.nb - 1);
    }
    __syncthreads();
    if (!last) return;
    pg_final(a);
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
        pg_add_partial(a, k, sums[k], 0);
    else if (k < kPgFields)
        pg_add_partial(a, k, 0.f, cnts[k - kPgSums]);
    pg_finish(a);
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

// One token, fp32 decisions, no branches (the tokens of a thread interleave freely).
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

// A token inside a band, re-decided exactly (float-float) by the thread that met it: the
// decisions, then the outputs and the sum term that depend on them (loss_ppo and the two
// gradients); the values no decision touches stay as pg_fast formed them.
RL_DEVINL void pg_resolve(PgTok& o, float lt, float lo, float ls, float A, const PgPrep& q) {
    const PgExact e = pg_exact(lt, lo, ls, A, q);
    const float r = exp_fast(lt - lo);
    const float lc = fmaxf(-A * r, -A * fminf(fmaxf(r, q.lo_b), q.hi_b));
    const float rho = fminf(exp_fast(lo - ls), q.tis);
    const float loss_ppo = e.dual ? -A * q.cc : lc;
    const float g_c = e.clip ? 0.f : -A * r;
    o.lp = loss_ppo;
    o.gp = e.dual ? 0.f : g_c;
    o.gd = rho * g_c;
    o.s[0] = loss_ppo;
    o.clip = e.clip;
    o.dual = e.dual;
    o.ice_lo = e.ice_lo;
    o.ice_hi = e.ice_hi;
    o.tis = e.tis_trunc;
    o.j = e.j;
    o.band = false;
}

struct PgFastAcc {
    float sum[kPgSums];
    int cnt[6];
};

// Take one token's values unless it is masked out (band tokens are resolved first).
RL_DEVINL void pg_take(const PgTok& t, bool valid, int* hist, PgFastAcc& acc, float& lp, float& ld, float& gp,
                       float& gd) {
    const bool use = valid & !t.band;
    lp = use ? t.lp : 0.f;
    ld = use ? t.ld : 0.f;
    gp = use ? t.gp : 0.f;
    gd = use ? t.gd : 0.f;
#pragma unroll
    for (int k = 0; k < kPgSums; ++k) acc.sum[k] += use ? t.s[k] : 0.f;   // a select: a masked NaN stays out
    const int u = use;
    acc.cnt[0] += u;
    acc.cnt[1] += u & t.clip;
    acc.cnt[2] += u & t.dual;
    acc.cnt[3] += u & t.ice_lo;
    acc.cnt[4] += u & t.ice_hi;
    acc.cnt[5] += u & t.tis;
    hist[t.j * kPgThreads] += u;
}


// One stage of the ring: kPgStageSlots consecutive token slots of the five inputs.
struct alignas(16) PgStage {
    float lt[kPgStageSlots], lo[kPgStageSlots], ls[kPgStageSlots], A[kPgStageSlots];
    uint8_t m[kPgStageSlots];
};
constexpr int kPgStageBytes = static_cast<int>(sizeof(PgStage));
constexpr int kPgStreamSmem = kPgDepth * kPgStageBytes;

// The block's partial into the batch accumulators: warp trees (fp32 sums, exact int32
// counts), then the eight consumer warps in order; the curve bins 1..n from the histogram
// (the last block turns them into the curve counts).  Called by every thread of a
// streaming block (288).
RL_DEVINL void pg_block_partial(const PgArgs& a, const PgFastAcc& acc, const int* hist_s, const int32_t* blk_status) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool consumer = threadIdx.x < kPgThreads;
    __shared__ float shs[kPgThreads / 32][kPgSums];
    __shared__ int shc[kPgThreads / 32][6];
    __shared__ int bins[kPgBins];
    __syncthreads();
#pragma unroll
    for (int f = 0; f < kPgSums; ++f) {
        const float v = warp_sum(acc.sum[f]);
        if (lane == 0 && consumer) shs[warp][f] = v;
    }
#pragma unroll
    for (int f = 0; f < 6; ++f) {
        const int v = __reduce_add_sync(0xffffffffu, acc.cnt[f]);
        if (lane == 0 && consumer) shc[warp][f] = v;
    }
    __syncthreads();
    if (consumer)
        for (int b = warp; b <= a.q.n; b += kPgThreads / 32) {
            int v = 0;
            for (int t = lane; t < kPgThreads; t += 32) v += hist_s[b * kPgThreads + t];
            v = __reduce_add_sync(0xffffffffu, v);
            if (lane == 0) bins[b] = v;
        }
    __syncthreads();
    const int f = threadIdx.x;
    if (f < kPgSums) {
        float v = 0.f;
        for (int w = 0; w < kPgThreads / 32; ++w) v += shs[w][f];
        pg_add_partial(a, f, v, 0);
    } else if (f < kPgSums + 6) {
        int v = 0;
        for (int w = 0; w < kPgThreads / 32; ++w) v += shc[w][f - kPgSums];
        pg_add_partial(a, f, 0.f, v);
    } else if (f < kPgFields) {
        const int b = f - kPgSums - 5;        // sorted bin 1..16
        pg_add_partial(a, f, 0.f, b <= a.q.n ? bins[b] : 0);
    } else if (f == kPgFields && *blk_status != 0) {
        atomicOr(a.status, *blk_status);
    }
}


// Stages of kPgStageSlots slots are dealt round-robin to the blocks (block b takes stages
// b, b + nb, b + 2 nb, ... with nb odd, so a block's stages walk through every phase of a
// power-of-two padding period and the valid tokens, where the arithmetic is, spread
// evenly).  Warp-specialised, 288 threads:
//   * warps 0-7 (consumers) take 2 consecutive slots each per stage (vector shared-memory
//     reads, streaming stores) and release the stage on its "empty" mbarrier (one
//     arrival per warp), so no consumer waits for another; a token inside a band is
//     re-decided exactly on the spot by the thread that met it (rare: the warp waits
//     for that lane, the other warps go on);
//   * warp 8 (producer): lane 0 fills a ring of kPgDepth shared-memory stages with bulk
//     copies, five per stage, one "full" mbarrier per stage.
// A thread's tokens and their order are fixed by the stage assignment, so its fp32 sums,
// and with them the block partial, are reproducible.  The last T mod 16 slots go to the
// last block with scalar loads.  Every wait is bounded: on a timeout the block records
// RL_STATUS_TIMEOUT, stops, and waits (bounded) for the copies it still has in flight.
__global__ void __launch_bounds__(kPgThreads + 32, kPgFastPerSm) policy_fast_kernel(PgArgs a) {
    extern __shared__ __align__(128) uint8_t pg_smem[];
    PgStage* ring = reinterpret_cast<PgStage*>(pg_smem);
    __shared__ __align__(8) uint64_t full[kPgDepth];
    __shared__ __align__(8) uint64_t empty[kPgDepth];
    __shared__ int hist_s[kPgBins * kPgThreads];   // bin-major: thread t's bin b at b * 256 + t
    __shared__ int abort_flag;
    __shared__ int32_t blk_status;                  // RL_STATUS_* bits of this block's waits

    const int64_t n16 = a.T >> 4;
    const int64_t nstages = (n16 * 16 + kPgStageSlots - 1) / kPgStageSlots;
    const int64_t mine = blockIdx.x < nstages ? (nstages - blockIdx.x + a.nb - 1) / a.nb : 0;
    const int nst = static_cast<int>(mine);
    const bool consumer = threadIdx.x < kPgThreads;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == kPgThreads) {
        for (int s = 0; s < kPgDepth; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, kPgThreads / 32);
        }
        fence_mbar_init();
    }
    if (threadIdx.x == 0) {
        abort_flag = 0;
        blk_status = 0;
    }
    if (consumer)
        for (int b = 0; b <= a.q.n; ++b) hist_s[b * kPgThreads + threadIdx.x] = 0;
    __syncthreads();

    PgFastAcc acc;
#pragma unroll
    for (int k = 0; k < kPgSums; ++k) acc.sum[k] = 0.f;
#pragma unroll
    for (int k = 0; k < 6; ++k) acc.cnt[k] = 0;
    auto stage_start = [&](int i) { return (static_cast<int64_t>(i) * a.nb + blockIdx.x) * kPgStageSlots; };
    volatile int* vflag = &abort_flag;

    if (!consumer) {
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < nst; ++i) {
                const int slot = i % kPgDepth;
                if (i >= kPgDepth &&
                    !mbar_wait(empty + slot, static_cast<uint32_t>((i / kPgDepth - 1) & 1), &blk_status, a.wait_ns)) {
                    atomicExch(&abort_flag, 1);
                    break;
                }
                if (*vflag) break;
                const int64_t g = stage_start(i);
                const int64_t left = n16 * 16 - g;
                const uint32_t L = static_cast<uint32_t>(left < kPgStageSlots ? left : kPgStageSlots);
                PgStage& st = ring[slot];
                mbar_arrive_expect_tx(full + slot, (a.mask ? 17u : 16u) * L);
                bulk_load(st.lt, a.lt + g, 4u * L, full + slot);
                bulk_load(st.lo, a.lo + g, 4u * L, full + slot);
                bulk_load(st.ls, a.ls + g, 4u * L, full + slot);
                bulk_load(st.A, a.adv + g, 4u * L, full + slot);
                if (a.mask) bulk_load(st.m, a.mask + g, L, full + slot);
                issued = i + 1;
            }
            if (*vflag) {
                // the last kPgDepth stages issued may still be in flight: wait for them
                // (bounded by the fixed kWaitLimitNs, whatever the work loop's limit)
                // before the block's shared memory goes away
                for (int i = issued > kPgDepth ? issued - kPgDepth : 0; i < issued; ++i)
                    mbar_wait(full + i % kPgDepth, static_cast<uint32_t>((i / kPgDepth) & 1), &blk_status);
            }
        }
    } else {
        int* hist = hist_s + threadIdx.x;
        const int j = 2 * threadIdx.x;
        for (int i = 0; i < nst; ++i) {
            const int slot = i % kPgDepth;
            if (!mbar_wait(full + slot, static_cast<uint32_t>((i / kPgDepth) & 1), &blk_status, a.wait_ns)) {
                atomicExch(&abort_flag, 1);
                break;
            }
            if (*vflag) break;
            const int64_t g = stage_start(i);
            if (g + j < n16 * 16) {
                const PgStage& st = ring[slot];
                const float2 lt = *reinterpret_cast<const float2*>(st.lt + j);
                const float2 lo = *reinterpret_cast<const float2*>(st.lo + j);
                const float2 ls = *reinterpret_cast<const float2*>(st.ls + j);
                const float2 A = *reinterpret_cast<const float2*>(st.A + j);
                // packed input (no mask): every slot is a valid token
                const uint32_t mw = a.mask ? *reinterpret_cast<const uint16_t*>(st.m + j) : 0x0101u;
                float2 lp = make_float2(0.f, 0.f), ld = lp, gp = lp, gd = lp;
                if (mw != 0u) {
                    const bool v0 = (mw & 0xffu) != 0u, v1 = (mw & 0xff00u) != 0u;
                    PgTok t0 = pg_fast(lt.x, lo.x, ls.x, A.x, a.q);
                    PgTok t1 = pg_fast(lt.y, lo.y, ls.y, A.y, a.q);
                    if (v0 & t0.band) pg_resolve(t0, lt.x, lo.x, ls.x, A.x, a.q);
                    if (v1 & t1.band) pg_resolve(t1, lt.y, lo.y, ls.y, A.y, a.q);
                    pg_take(t0, v0, hist, acc, lp.x, ld.x, gp.x, gd.x);
                    pg_take(t1, v1, hist, acc, lp.y, ld.y, gp.y, gd.y);
                }
                if (a.loss_ppo) __stcs(reinterpret_cast<float2*>(a.loss_ppo + g + j), lp);
                if (a.loss_dec) __stcs(reinterpret_cast<float2*>(a.loss_dec + g + j), ld);
                if (a.grad_ppo) __stcs(reinterpret_cast<float2*>(a.grad_ppo + g + j), gp);
                if (a.grad_dec) __stcs(reinterpret_cast<float2*>(a.grad_dec + g + j), gd);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + slot);
        }
        // the last T mod 16 slots, scalar loads
        if (blockIdx.x == a.nb - 1) {
            const int64_t t = n16 * 16 + threadIdx.x;
            if (t < a.T) {
                float lp = 0.f, ld = 0.f, gp = 0.f, gd = 0.f;
                if (a.mask == nullptr || a.mask[t] != 0) {
                    const float xt = a.lt[t], xo = a.lo[t], xs = a.ls[t], xa = a.adv[t];
                    PgTok tk = pg_fast(xt, xo, xs, xa, a.q);
                    if (tk.band) pg_resolve(tk, xt, xo, xs, xa, a.q);
                    pg_take(tk, true, hist, acc, lp, ld, gp, gd);
                }
                if (a.loss_ppo) a.loss_ppo[t] = lp;
                if (a.loss_dec) a.loss_dec[t] = ld;
                if (a.grad_ppo) a.grad_ppo[t] = gp;
                if (a.grad_dec) a.grad_dec[t] = gd;
            }
        }
    }
    pg_block_partial(a, acc, hist_s, &blk_status);
    pg_finish(a);
}

// ----------------------------------------------------------------------------------
// Packed pass (no mask: every slot a valid token)
// ----------------------------------------------------------------------------------
// The tokens (the whole groups of four) are cut into 1024-token stages.  Block b's producer
// warp fills a ring of kPkDepth shared-memory stages with bulk copies (four per stage):
// first stages b, b + nb, ..., then, each time a slot frees, the next stage from a claim
// counter, until none is left (it then marks the slot "end").  Blocks that get more of the
// memory system's bandwidth so take more stages, and all of them finish together.  Each
// consumer thread takes four consecutive tokens of a stage (16-byte shared loads, 16-byte
// streaming stores), and its fp32 sums over those four go into its 2^-24 fixed-point
// accumulators at once: a stage's contribution is the same whichever block took it.
// Every token's values enter the sums and counts without a select (there is no padding
// to keep out); a token inside a band is re-decided exactly first.  The IPO-curve bin comes from a 1024-bucket table of |p_old - p_samp|
// built in shared memory at block start: a bucket records how many curve eps lie below
// it, the one eps inside it (compared exactly), or that the token needs the full search
// (two eps inside, or an eps whose band reaches into the bucket).
constexpr int kPkStage = 1024;                 // tokens per stage
constexpr int kPkDepth = 3;                    // stages in the ring (more measured no faster)
struct alignas(16) PkStage {
    float lt[kPkStage], lo[kPkStage], ls[kPkStage], A[kPkStage];
};
constexpr int kPkSmem = kPkDepth * static_cast<int>(sizeof(PkStage));
static_assert(kPkSmem >= (kPgSums * 8 + 6 * 4) * kPgThreads, "the ring holds the block's values at the end");

// One bucket of |p_old - p_samp| in shared memory: its code (eps below it | the eps inside
// it << 8 | needs the exact path << 16) with that eps and its band half-width beside it,
// so a token reads its bucket with one 16-byte load.
struct __align__(16) PkBucket {
    int code;
    float eps, weps;
    int pad;
};

// Curve bin of one |p_old - p_samp| value from the bucket table, and whether it lies in
// the band of a curve eps (or its bucket needs the exact path: two eps inside it, or an
// eps whose band reaches into it).  Branch-free.
RL_DEVINL void pk_curve(float adiff, const PkBucket* lut, int& j, bool& band) {
    int b = static_cast<int>(adiff * static_cast<float>(kPkLut));   // exact scaling: bucket edges are exact
    b = b < 0 ? 0 : (b > kPkLut - 1 ? kPkLut - 1 : b);
    const PkBucket e = lut[b];
    j = (e.code & 31) + (adiff > e.eps ? 1 : 0);
    band = band | (fabsf(adiff - e.eps) <= e.weps) | ((e.code >> 16) != 0);
}

RL_DEVINL PgTok pg_fast_packed(float lt, float lo, float ls, float A, const PgPrep& q, const PkBucket* lut) {
    PgTok o;
    const float r = exp_fast(lt - lo);
    const float l1 = -A * r;
    const float l2 = -A * fminf(fmaxf(r, q.lo_b), q.hi_b);
    const float lc = fmaxf(l1, l2);
    const float l3 = -A * q.cc;
    const float d = lo - ls;
    const float rho_raw = exp_fast(d);
    const float adiff = exp_fast(ls) * fabsf(rho_raw - 1.f);
    bool band = ((A < 0.f) & ((fabsf(r - q.lo_b) <= q.w_lo_b) | (fabsf(r - q.cc) <= q.w_cc))) |
                ((A > 0.f) & (fabsf(r - q.hi_b) <= q.w_hi_b)) | (fabsf(rho_raw - q.tis) <= q.w_tis) |
                (fabsf(rho_raw - q.ice_lo) <= q.w_ice_lo) | (fabsf(rho_raw - q.ice_hi) <= q.w_ice_hi);
    int j;
    pk_curve(adiff, lut, j, band);
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
    o.band = band;
    return o;
}

// The packed pass's per-thread accumulators: sums in 2^-24 fixed point, counts.
struct PkAcc {
    long long fx[kPgSums];
    int cnt[6];
};

// The packed block's partial into the batch accumulators.  The ring is idle once every
// consumer is past its last stage, so it holds the threads' values field-major; then warp
// w < 6 sums fixed-point field w (eight values a lane, then a shuffle tree), warps 6 and 7
// the counts, and every warp some of the curve bins 1..n from the histogram, each adding
// its total with one atomic (integers: any order gives the same total).  Called by every
// thread of the block (288).
RL_DEVINL void pk_block_partial(const PgArgs& a, const PkAcc& acc, const int* hist_s, const int32_t* blk_status,
                                uint8_t* scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    long long* vx = reinterpret_cast<long long*>(scratch);                  // [kPgSums][256]
    int* vc = reinterpret_cast<int*>(scratch + kPgSums * kPgThreads * 8);    // [6][256]
    __syncthreads();   // the ring is free
    if (threadIdx.x < kPgThreads) {
#pragma unroll
        for (int f = 0; f < kPgSums; ++f) vx[f * kPgThreads + threadIdx.x] = acc.fx[f];
#pragma unroll
        for (int f = 0; f < 6; ++f) vc[f * kPgThreads + threadIdx.x] = acc.cnt[f];
    }
    __syncthreads();
    auto add = [&](int k, long long x) {
        if (x != 0)
            atomicAdd(reinterpret_cast<unsigned long long*>(a.acc + k * kPgAccStride), static_cast<unsigned long long>(x));
    };
    if (warp < kPgSums) {
        long long v = 0;
#pragma unroll
        for (int i = 0; i < kPgThreads / 32; ++i) v += vx[warp * kPgThreads + lane + 32 * i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) add(warp, v);
    } else if (warp < kPgThreads / 32) {
        for (int f = (warp - kPgSums) * 3; f < (warp - kPgSums) * 3 + 3; ++f) {
            int v = 0;
#pragma unroll
            for (int i = 0; i < kPgThreads / 32; ++i) v += vc[f * kPgThreads + lane + 32 * i];
            v = __reduce_add_sync(0xffffffffu, v);
            if (lane == 0) add(kPgSums + f, v);
        }
    } else if (lane == 0 && *blk_status != 0) {
        atomicOr(a.status, *blk_status);
    }
    if (warp < kPgThreads / 32)
        for (int b = 1 + warp; b <= a.q.n; b += kPgThreads / 32) {
            int v = 0;
#pragma unroll
            for (int i = 0; i < kPgThreads / 32; ++i) v += hist_s[b * kPgThreads + lane + 32 * i];
            v = __reduce_add_sync(0xffffffffu, v);
            if (lane == 0) add(kPgSums + 5 + b, v);
        }
}

__global__ void __launch_bounds__(kPgThreads + 32, kPgFastPerSm) policy_packed_kernel(PgArgs a) {
    extern __shared__ __align__(128) uint8_t pk_smem[];
    PkStage* ring = reinterpret_cast<PkStage*>(pk_smem);
    __shared__ __align__(8) uint64_t full[kPkDepth];
    __shared__ __align__(8) uint64_t empty[kPkDepth];
    __shared__ int stage_of[kPkDepth];             // the stage in each ring slot, -1: no more
    __shared__ int hist_s[kPgBins * kPgThreads];   // bin-major: thread t's bin b at b * 256 + t
    __shared__ PkBucket lut[kPkLut];
    __shared__ int abort_flag;
    __shared__ int32_t blk_status;

    const PgPrep& q = a.q;
    const int64_t n4 = a.T >> 2;                   // groups of four tokens
    const int64_t ntok = 4 * n4;                   // tokens the stages cover
    const int nst = static_cast<int>((ntok + kPkStage - 1) / kPkStage);
    const bool consumer = threadIdx.x < kPgThreads;
    const int lane = threadIdx.x & 31;
    volatile int* vflag = &abort_flag;
    // The producer lane fills the ring: entry i goes to slot i mod kPkDepth, stage
    // blockIdx + i nb for the first kPkDepth entries, then claimed ones (the claim's round
    // trip overlaps the wait for the slot).  Returns false once it has placed the end mark
    // (no stage left) or the block aborts.
    int issued = 0;
    auto fill = [&](int i) -> bool {
        const int slot = i % kPkDepth;
        const int s = i < kPkDepth ? static_cast<int>(blockIdx.x) + i * a.nb
                                   : kPkDepth * a.nb + static_cast<int>(atomicAdd(a.claim, 1u));
        if (i >= kPkDepth &&
            !mbar_wait(empty + slot, static_cast<uint32_t>((i / kPkDepth - 1) & 1), &blk_status, a.wait_ns)) {
            atomicExch(&abort_flag, 1);
            return false;
        }
        if (*vflag) return false;
        if (s >= nst) {   // none left: the consumers stop at this slot
            stage_of[slot] = -1;
            mbar_arrive(full + slot);
            return false;
        }
        stage_of[slot] = s;
        const int64_t g = static_cast<int64_t>(s) * kPkStage;
        const int64_t left = ntok - g;
        const uint32_t L = static_cast<uint32_t>(left < kPkStage ? left : kPkStage);
        PkStage& st = ring[slot];
        mbar_arrive_expect_tx(full + slot, 16u * L);
        bulk_load(st.lt, a.lt + g, 4u * L, full + slot);
        bulk_load(st.lo, a.lo + g, 4u * L, full + slot);
        bulk_load(st.ls, a.ls + g, 4u * L, full + slot);
        bulk_load(st.A, a.adv + g, 4u * L, full + slot);
        issued = i + 1;
        return true;
    };
    int pi = 0;
    if (threadIdx.x == kPgThreads) {
        for (int s = 0; s < kPkDepth; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, kPgThreads / 32);
        }
        fence_mbar_init();
        abort_flag = 0;
        blk_status = 0;
        // the first ring entries at once: their copies overlap the block's table setup
        while (pi < kPkDepth && fill(pi)) ++pi;
    }
    if (consumer) {
        for (int b = 0; b <= q.n; ++b) hist_s[b * kPgThreads + threadIdx.x] = 0;
        for (int i = threadIdx.x; i < kPkLut; i += kPgThreads) {
            const int e = q.lut[i];
            const int kin = (e >> 8) & 31;
            lut[i] = PkBucket{e, q.eps_s[kin], q.weps_s[kin], 0};
        }
    }
    __syncthreads();

    PkAcc acc;
#pragma unroll
    for (int k = 0; k < kPgSums; ++k) acc.fx[k] = 0;
#pragma unroll
    for (int k = 0; k < 6; ++k) acc.cnt[k] = 0;

    if (!consumer) {
        if (lane == 0) {
            // after the first entries (pi < kPkDepth here only if the stages ran out)
            if (pi == kPkDepth)
                while (fill(pi)) ++pi;
            if (*vflag) {
                // the last stages issued may still be in flight: wait for them (bounded by
                // the fixed kWaitLimitNs) before the block's shared memory goes away
                for (int i = issued > kPkDepth ? issued - kPkDepth : 0; i < issued; ++i)
                    mbar_wait(full + i % kPkDepth, static_cast<uint32_t>((i / kPkDepth) & 1), &blk_status);
            }
        }
    } else {
        int* hist = hist_s + threadIdx.x;
        const int j4 = 4 * threadIdx.x;
        for (int i = 0;; ++i) {
            const int slot = i % kPkDepth;
            if (!mbar_wait(full + slot, static_cast<uint32_t>((i / kPkDepth) & 1), &blk_status, a.wait_ns)) {
                atomicExch(&abort_flag, 1);
                break;
            }
            if (*vflag) break;
            const int s = stage_of[slot];
            if (s < 0) break;
            const int64_t g = static_cast<int64_t>(s) * kPkStage;
            if (g + j4 < ntok) {
                const PkStage& st = ring[slot];
                const float4 lt4 = *reinterpret_cast<const float4*>(st.lt + j4);
                const float4 lo4 = *reinterpret_cast<const float4*>(st.lo + j4);
                const float4 ls4 = *reinterpret_cast<const float4*>(st.ls + j4);
                const float4 A4 = *reinterpret_cast<const float4*>(st.A + j4);
                const float vt[4] = {lt4.x, lt4.y, lt4.z, lt4.w}, vo[4] = {lo4.x, lo4.y, lo4.z, lo4.w};
                const float vs[4] = {ls4.x, ls4.y, ls4.z, ls4.w}, vA[4] = {A4.x, A4.y, A4.z, A4.w};
                float lp[4], ld[4], gp[4], gd[4];
                float sum4[kPgSums];
#pragma unroll
                for (int k = 0; k < kPgSums; ++k) sum4[k] = 0.f;
#pragma unroll
                for (int u = 0; u < 4; u += 2) {   // two tokens at a time: two independent chains, no branch
                    PgTok t[2] = {pg_fast_packed(vt[u], vo[u], vs[u], vA[u], q, lut),
                                  pg_fast_packed(vt[u + 1], vo[u + 1], vs[u + 1], vA[u + 1], q, lut)};
                    if (t[0].band | t[1].band) {   // rare: re-decide exactly
                        if (t[0].band) pg_resolve(t[0], vt[u], vo[u], vs[u], vA[u], q);
                        if (t[1].band) pg_resolve(t[1], vt[u + 1], vo[u + 1], vs[u + 1], vA[u + 1], q);
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        lp[u + h] = t[h].lp;
                        ld[u + h] = t[h].ld;
                        gp[u + h] = t[h].gp;
                        gd[u + h] = t[h].gd;
#pragma unroll
                        for (int k = 0; k < kPgSums; ++k) sum4[k] += t[h].s[k];
                        acc.cnt[1] += t[h].clip;
                        acc.cnt[2] += t[h].dual;
                        acc.cnt[3] += t[h].ice_lo;
                        acc.cnt[4] += t[h].ice_hi;
                        acc.cnt[5] += t[h].tis;
                        atomicAdd(hist + t[h].j * kPgThreads, 1);   // the thread's own column: no contention
                    }
                }
#pragma unroll
                for (int k = 0; k < kPgSums; ++k) acc.fx[k] += pg_fix_fast(a, sum4[k]);
                acc.cnt[0] += 4;
                if (a.loss_ppo) __stcs(reinterpret_cast<float4*>(a.loss_ppo + g + j4), make_float4(lp[0], lp[1], lp[2], lp[3]));
                if (a.loss_dec) __stcs(reinterpret_cast<float4*>(a.loss_dec + g + j4), make_float4(ld[0], ld[1], ld[2], ld[3]));
                if (a.grad_ppo) __stcs(reinterpret_cast<float4*>(a.grad_ppo + g + j4), make_float4(gp[0], gp[1], gp[2], gp[3]));
                if (a.grad_dec) __stcs(reinterpret_cast<float4*>(a.grad_dec + g + j4), make_float4(gd[0], gd[1], gd[2], gd[3]));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + slot);
        }
        // the last T mod 4 tokens, scalar loads
        if (blockIdx.x == a.nb - 1) {
            const int64_t t = ntok + threadIdx.x;
            if (t < a.T) {
                float lp, ld, gp, gd;
                const float xt = a.lt[t], xo = a.lo[t], xs = a.ls[t], xa = a.adv[t];
                PgTok tk = pg_fast_packed(xt, xo, xs, xa, q, lut);
                if (tk.band) pg_resolve(tk, xt, xo, xs, xa, q);
                PgFastAcc one;
#pragma unroll
                for (int k = 0; k < kPgSums; ++k) one.sum[k] = 0.f;
#pragma unroll
                for (int k = 0; k < 6; ++k) one.cnt[k] = 0;
                pg_take(tk, true, hist, one, lp, ld, gp, gd);
#pragma unroll
                for (int k = 0; k < kPgSums; ++k) acc.fx[k] += pg_fix(a, one.sum[k]);
#pragma unroll
                for (int k = 0; k < 6; ++k) acc.cnt[k] += one.cnt[k];
                if (a.loss_ppo) a.loss_ppo[t] = lp;
                if (a.loss_dec) a.loss_dec[t] = ld;
                if (a.grad_ppo) a.grad_ppo[t] = gp;
                if (a.grad_dec) a.grad_dec[t] = gd;
            }
        }
    }
    pk_block_partial(a, acc, hist_s, &blk_status, pk_smem);
    pg_finish(a);
}

// ----------------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------------
// Workspace (kPolicyWorkspaceBytes): the first 128-byte line holds the arrival counter
// (byte 0), the status word (4), the range flag (8) and the claim counter (12); the
// kPgFields accumulators follow, one 128-byte line each.  All of it is zero before the
// first call, and the last block of every call leaves it zero again.  At most
// kPgMaxBlocks blocks run, so the workspace size does not depend on the device.
constexpr size_t kPgAccBase = 128;
static_assert(kPgAccBase + kPgFields * kPgAccStride * 8 <= kPolicyWorkspaceBytes, "workspace layout");

static int fast_blocks(int sms) {   // odd: see policy_fast_kernel
    const int n = sms * kPgFastPerSm - 1;
    return n < kPgMaxBlocks ? n : kPgMaxBlocks - 1;
}
static int slow_blocks(int sms) {
    const int n = sms * kPgSlowPerSm;
    return n < kPgMaxBlocks ? n : kPgMaxBlocks;
}

size_t policy_ws_bytes(int64_t T) {
    (void)T;
    return kPolicyWorkspaceBytes;
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
    for (int k = 0; k < q.n; ++k) q.pos[q.perm[k]] = k;
    for (int k = 0; k < q.n; ++k) {
        q.eps[k] = p.curve_eps[q.perm[k]];
        q.weps[k] = band(q.eps[k]);
    }
    // the packed pass's bucket table over |p_old - p_samp| in [0, 1]: bucket b holds
    // [b / kPkLut, (b + 1) / kPkLut) (the last one up to 1 inclusive)
    q.eps_s[0] = INFINITY;
    q.weps_s[0] = -1.f;
    for (int k = 0; k < q.n; ++k) {
        q.eps_s[k + 1] = q.eps[k];
        q.weps_s[k + 1] = q.weps[k];
    }
    for (int b = 0; b < kPkLut; ++b) {
        const float blo = static_cast<float>(b) / static_cast<float>(kPkLut);
        const float bhi = static_cast<float>(b + 1) / static_cast<float>(kPkLut);
        int below = 0, inside = 0, kin = 0, slow = 0;
        for (int k = 0; k < q.n; ++k) {
            const float e = q.eps[k];
            if (e < blo) {
                ++below;
                slow |= blo - e <= q.weps[k];
            } else if (e < bhi || b == kPkLut - 1) {
                ++inside;
                kin = k + 1;
            } else {
                slow |= e - bhi <= q.weps[k];
            }
        }
        slow |= inside > 1;
        q.lut[b] = below | (kin << 8) | (slow << 16);
    }
    return q;
}

int policy_impl(const float* lt, const float* lo, const float* ls, const float* adv,
                const uint8_t* mask, int64_t T, const rl_pg_params* p, float* loss_ppo,
                float* loss_dec, float* grad_ppo, float* grad_dec, rl_pg_metrics* metrics,
                void* ws, size_t ws_bytes, cudaStream_t stream) {
    const int sms = num_sms();
    if (ws_bytes < policy_ws_bytes(T)) return RL_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 7u) != 0) {   // int64 accumulators
        set_last_error("workspace not 8-byte aligned");
        return RL_ERR_ARG;
    }
    auto al = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
    const bool fast = T < (int64_t(1) << 31) && al(lt) && al(lo) && al(ls) && al(adv) && al(mask) &&
                      al(loss_ppo) && al(loss_dec) && al(grad_ppo) && al(grad_dec);
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
    uint8_t* hb = static_cast<uint8_t*>(ws);
    a.arrive = reinterpret_cast<unsigned int*>(hb);
    a.status = reinterpret_cast<int32_t*>(hb + 4);
    a.range = reinterpret_cast<int*>(hb + 8);
    a.claim = reinterpret_cast<unsigned int*>(hb + 12);
    a.acc = reinterpret_cast<long long*>(hb + kPgAccBase);
    a.metrics = metrics;
    a.wait_ns = wait_limit_ns();
    // per device: the fast pass's shared-memory opt-in (set once; concurrent first calls
    // from several host threads at worst set the same attribute twice)
    static std::atomic<int> smem_set[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return RL_ERR_CUDA;
    if (fast && !smem_set[dev].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(policy_fast_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPgStreamSmem) !=
                cudaSuccess ||
            cudaFuncSetAttribute(policy_packed_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPkSmem) !=
                cudaSuccess)
            return RL_ERR_CUDA;
        smem_set[dev].store(1, std::memory_order_release);
    }
    ProfScope ps(RL_PROF_POLICY, stream);   // the kernel launch
    a.nb = fast ? fast_blocks(sms) : slow_blocks(sms);
    a.curve_bins = fast;
    // a term below 2^38 / (terms per accumulator) keeps each accumulator's total below 2^62
    // in 2^-24 units: one term per block, or in the packed pass one per thread and stage
    // (a group of four tokens) and one per tail token
    const double terms = fast && mask == nullptr ? static_cast<double>(T / 4 + 3) : static_cast<double>(a.nb);
    a.range_lim = static_cast<float>(ldexp(1.0, 38) / terms);
    if (fast && mask == nullptr) {
        policy_packed_kernel<<<a.nb, kPgThreads + 32, kPkSmem, stream>>>(a);
    } else if (fast) {
        policy_fast_kernel<<<a.nb, kPgThreads + 32, kPgStreamSmem, stream>>>(a);
    } else {
        policy_slow_kernel<<<a.nb, kPgThreads, 0, stream>>>(a);
    }
    count_launch(1);
    return cudaPeekAtLastError() == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}

}  // namespace rl
