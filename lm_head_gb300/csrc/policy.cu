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
//  1'. policy_packed_kernel the same pass for packed input (no mask): an equal contiguous
//                          range per block, four tokens per thread, no selects, the curve
//                          bin from a bucket table.
//  2. policy_slow_kernel   the whole pass with exact decisions in the bands, for inputs the
//                          fast passes do not take (unaligned, T >= 2^31).
//  With no mask (packed input: every slot a valid token) the mask is neither read nor
//  copied: 16 bytes in per token instead of 17.
//  Each block writes its partial (fp32 sums in a fixed order within the block, counts, the
//  status bits of its waits) to its own record in the workspace; the last block to arrive
//  (an arrival counter) sums the records in block order (fp64 sums, int64 counts), writes
//  the metrics and sets the counter back to zero.  So a workspace zeroed once before its
//  first use needs no clearing before later calls, and a call is one kernel launch.
//
// Results are bitwise reproducible for a given device and T.
#include <atomic>
#include <cmath>
#include <climits>

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
    struct PgRecords* rec;        // the blocks' partials
    unsigned int* arrive;         // blocks of this launch that have written their record (0 between calls)
    int nb;                       // blocks of the pass
    uint64_t wait_ns;             // limit of the streaming loop's waits (RL_OPT_WAIT_LIMIT_US)
    rl_pg_metrics* metrics;       // or nullptr
};

// A block's partial, one 128-byte record per block (the last block loads them 16 bytes at
// a time): fp32 sums in the block's fixed order, counts (the curve in the caller's order),
// the RL_STATUS_* bits the block's waits raised.
constexpr int kPgRecFields = kPgSums + 6 + RL_PG_MAX_CURVE + 1;   // + status
constexpr int kPgMaxBlocks = 512;
struct alignas(16) PgRecord {
    float sum[kPgSums];
    int cnt[6 + RL_PG_MAX_CURVE];
    int status;
    int pad[3];
};
static_assert(sizeof(PgRecord) == 128, "one record per 128 bytes");
struct PgRecords {
    PgRecord r[kPgMaxBlocks];
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

// ----------------------------------------------------------------------------------
// Batch totals
// ----------------------------------------------------------------------------------
// The last block.  The records come into shared memory (`scratch`, the block's stage ring,
// idle by now; cap_bytes of it) 16 bytes per load, all loads of a chunk in flight at once;
// then thread (f, g), f < 29, g < 9 (8 in a 256-thread block), adds field f of the staged
// records g, g + 9, g + 18, ... (the sums as float-float pairs, about 44 significant bits, the counts as integers,
// the status bits OR-ed), and thread f adds its field's nine group totals in order.  With
// no scratch (the slow pass) the records are read from global memory directly.  Fixed
// order throughout, whatever order the blocks arrived in.
RL_DEVINL void pg_final(const PgArgs& a, uint8_t* scratch, int cap_bytes) {
    constexpr int kGMax = 9;
    __shared__ FF part_s[kPgSums][kGMax];
    __shared__ int part_c[kPgRecFields - kPgSums][kGMax];
    // groups per field: 9 with 288 threads (the streaming passes), 8 with 256 (the slow pass)
    const int kG = static_cast<int>(blockDim.x) / kPgRecFields < kGMax ? static_cast<int>(blockDim.x) / kPgRecFields
                                                                       : kGMax;
    const int tid = threadIdx.x;
    FF vs = {0.f, 0.f};
    int vc = 0;
    const int chunk = scratch ? cap_bytes / static_cast<int>(sizeof(PgRecord)) : a.nb;
    for (int c0 = 0; c0 < a.nb; c0 += chunk) {
        const int n = a.nb - c0 < chunk ? a.nb - c0 : chunk;
        const PgRecord* src = a.rec->r + c0;
        if (scratch) {
            // nine loads of each thread in flight before its first store: one L2 round trip
            // per 9 x blockDim 16-byte pieces (303 records of 128 bytes: one round), not one
            // per load
            const uint4* g4 = reinterpret_cast<const uint4*>(src);
            uint4* s4 = reinterpret_cast<uint4*>(scratch);
            constexpr int kPer = 9;
            const int step = kPer * static_cast<int>(blockDim.x);
            for (int base = 0; base < n * 8; base += step) {
                uint4 v[kPer];
#pragma unroll
                for (int k = 0; k < kPer; ++k) {
                    const int i = base + tid + k * static_cast<int>(blockDim.x);
                    if (i < n * 8) v[k] = __ldcg(g4 + i);
                }
#pragma unroll
                for (int k = 0; k < kPer; ++k) {
                    const int i = base + tid + k * static_cast<int>(blockDim.x);
                    if (i < n * 8) s4[i] = v[k];
                }
            }
            __syncthreads();
            src = reinterpret_cast<const PgRecord*>(scratch);
        }
        if (tid < kPgRecFields * kG) {
            const int f = tid / kG, g = tid - (tid / kG) * kG;
            if (f < kPgSums) {
                for (int b = g; b < n; b += kG) vs = ff_add(vs, {scratch ? src[b].sum[f] : __ldcg(&src[b].sum[f]), 0.f});
            } else if (f < kPgRecFields - 1) {
                for (int b = g; b < n; b += kG) vc += scratch ? src[b].cnt[f - kPgSums] : __ldcg(&src[b].cnt[f - kPgSums]);
            } else {
                for (int b = g; b < n; b += kG) vc |= scratch ? src[b].status : __ldcg(&src[b].status);
            }
        }
        __syncthreads();   // the chunk is read before the next one overwrites it
    }
    if (tid < kPgRecFields * kG) {
        const int f = tid / kG, g = tid - (tid / kG) * kG;
        if (f < kPgSums)
            part_s[f][g] = vs;
        else
            part_c[f - kPgSums][g] = vc;
    }
    __syncthreads();
    if (tid == 0) *a.arrive = 0u;   // every block has arrived: ready for the next call
    if (!a.metrics || tid >= kPgRecFields) return;
    if (tid < kPgSums) {
        FF v = part_s[tid][0];
        for (int g = 1; g < kG; ++g) v = ff_add(v, part_s[tid][g]);
        pg_write_metric(tid, static_cast<double>(v.hi) + static_cast<double>(v.lo), a.metrics);
    } else if (tid < kPgRecFields - 1) {
        int v = 0;
        for (int g = 0; g < kG; ++g) v += part_c[tid - kPgSums][g];
        pg_write_metric(tid, static_cast<double>(v), a.metrics);   // counts are exact integers
    } else {
        int v = 0;
        for (int g = 0; g < kG; ++g) v |= part_c[tid - kPgSums][g];
        a.metrics->status = v;
    }
}

// Every thread of every block calls this after the block's record is written; the last
// block to arrive finishes.
RL_DEVINL void pg_finish(const PgArgs& a, uint8_t* scratch, int cap_bytes) {
    __shared__ int last;
    __threadfence();   // this block's record (and outputs) before its arrival
    __syncthreads();
    if (threadIdx.x == 0) last = atomicAdd(a.arrive, 1u) == static_cast<unsigned int>(a.nb - 1);
    __syncthreads();
    if (!last) return;
    __threadfence();
    pg_final(a, scratch, cap_bytes);
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
    PgRecord& rec = a.rec->r[blockIdx.x];
    if (k < kPgSums)
        rec.sum[k] = sums[k];
    else if (k < kPgFields)
        rec.cnt[k - kPgSums] = cnts[k - kPgSums];
    else if (k == kPgFields)
        rec.status = 0;
    pg_finish(a, nullptr, 0);
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

// One bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16),
// completion counted on an mbarrier of this CTA.
RL_DEVINL void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// The block's partial into its record: warp trees (fp32 sums, exact int32 counts), then the
// eight consumer warps in order; the curve counts from the histogram, cnt_k = #(j > k),
// back in the caller's order.  Called by every thread of a streaming block (288).
RL_DEVINL void pg_block_record(const PgArgs& a, const PgFastAcc& acc, const int* hist_s, const int32_t* blk_status) {
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
    PgRecord& rec = a.rec->r[blockIdx.x];
    if (f < kPgSums) {
        float v = 0.f;
        for (int w = 0; w < kPgThreads / 32; ++w) v += shs[w][f];
        rec.sum[f] = v;
    } else if (f < kPgSums + 6) {
        int v = 0;
        for (int w = 0; w < kPgThreads / 32; ++w) v += shc[w][f - kPgSums];
        rec.cnt[f - kPgSums] = v;
    } else if (f < kPgFields) {
        const int c = f - kPgSums - 6;        // caller's curve index
        int v = 0;
        if (c < a.q.n) {
            int js = 0;                        // its sorted position
            while (a.q.perm[js] != c) ++js;
            for (int k = js + 1; k <= a.q.n; ++k) v += bins[k];
        }
        rec.cnt[6 + c] = v;
    } else if (f == kPgFields) {
        rec.status = *blk_status;
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
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
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
    pg_block_record(a, acc, hist_s, &blk_status);
    pg_finish(a, pg_smem, kPgStreamSmem);   // the ring is idle now: scratch for the last block
}

// ----------------------------------------------------------------------------------
// Packed pass (no mask: every slot a valid token)
// ----------------------------------------------------------------------------------
// Each block takes one contiguous range of the tokens (an equal share, in groups of four),
// streamed through a ring of 1024-token stages by a producer warp (four bulk copies per
// stage); each consumer thread takes four consecutive tokens of a stage (16-byte shared
// loads, 16-byte streaming stores).  Every token's values enter the sums and counts
// without a select (there is no padding to keep out); a token inside a band is re-decided
// exactly first.  The IPO-curve bin comes from a 1024-bucket table of |p_old - p_samp|
// built in shared memory at block start: a bucket records how many curve eps lie below
// it, the one eps inside it (compared exactly), or that the token needs the full search
// (two eps inside, or an eps whose band reaches into the bucket).
constexpr int kPkStage = 1024;                 // tokens per stage
constexpr int kPkDepth = 5;                    // stages in the ring
struct alignas(16) PkStage {
    float lt[kPkStage], lo[kPkStage], ls[kPkStage], A[kPkStage];
};
constexpr int kPkSmem = kPkDepth * static_cast<int>(sizeof(PkStage));

// Curve bin of one |p_old - p_samp| value from the bucket table (in shared memory), and
// whether it lies in the band of a curve eps (or its bucket needs the exact path: two eps
// inside it, or an eps whose band reaches into it).  Branch-free.
RL_DEVINL void pk_curve(float adiff, const int* lut, const float* eps_s, const float* weps_s, int& j, bool& band) {
    int b = static_cast<int>(adiff * static_cast<float>(kPkLut));   // exact scaling: bucket edges are exact
    b = b < 0 ? 0 : (b > kPkLut - 1 ? kPkLut - 1 : b);
    const int e = lut[b];
    const int kin = (e >> 8) & 31;
    j = (e & 31) + (adiff > eps_s[kin] ? 1 : 0);
    band = band | (fabsf(adiff - eps_s[kin]) <= weps_s[kin]) | ((e >> 16) != 0);
}

RL_DEVINL PgTok pg_fast_packed(float lt, float lo, float ls, float A, const PgPrep& q, const int* lut,
                               const float* eps_s, const float* weps_s) {
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
    pk_curve(adiff, lut, eps_s, weps_s, j, band);
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

__global__ void __launch_bounds__(kPgThreads + 32, kPgFastPerSm) policy_packed_kernel(PgArgs a) {
    extern __shared__ __align__(128) uint8_t pk_smem[];
    PkStage* ring = reinterpret_cast<PkStage*>(pk_smem);
    __shared__ __align__(8) uint64_t full[kPkDepth];
    __shared__ __align__(8) uint64_t empty[kPkDepth];
    __shared__ int hist_s[kPgBins * kPgThreads];   // bin-major: thread t's bin b at b * 256 + t
    __shared__ int lut[kPkLut];
    __shared__ float s_eps[RL_PG_MAX_CURVE + 1], s_weps[RL_PG_MAX_CURVE + 1];
    __shared__ int abort_flag;
    __shared__ int32_t blk_status;

    const PgPrep& q = a.q;
    const int64_t n4 = a.T >> 2;                   // groups of four tokens
    const int64_t g0 = static_cast<int64_t>(blockIdx.x) * n4 / a.nb;
    const int64_t g1 = static_cast<int64_t>(blockIdx.x + 1) * n4 / a.nb;
    const int64_t t0 = 4 * g0, ntok = 4 * (g1 - g0);
    const int nst = static_cast<int>((ntok + kPkStage - 1) / kPkStage);
    const bool consumer = threadIdx.x < kPgThreads;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == kPgThreads) {
        for (int s = 0; s < kPkDepth; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, kPgThreads / 32);
        }
        fence_mbar_init();
    }
    if (threadIdx.x == 0) {
        abort_flag = 0;
        blk_status = 0;
    }
    if (consumer) {
        for (int b = 0; b <= q.n; ++b) hist_s[b * kPgThreads + threadIdx.x] = 0;
        if (threadIdx.x <= RL_PG_MAX_CURVE) {
            s_eps[threadIdx.x] = q.eps_s[threadIdx.x];
            s_weps[threadIdx.x] = q.weps_s[threadIdx.x];
        }
        for (int i = threadIdx.x; i < kPkLut; i += kPgThreads) lut[i] = q.lut[i];
    }
    __syncthreads();

    PgFastAcc acc;
#pragma unroll
    for (int k = 0; k < kPgSums; ++k) acc.sum[k] = 0.f;
#pragma unroll
    for (int k = 0; k < 6; ++k) acc.cnt[k] = 0;
    volatile int* vflag = &abort_flag;

    if (!consumer) {
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < nst; ++i) {
                const int slot = i % kPkDepth;
                if (i >= kPkDepth &&
                    !mbar_wait(empty + slot, static_cast<uint32_t>((i / kPkDepth - 1) & 1), &blk_status, a.wait_ns)) {
                    atomicExch(&abort_flag, 1);
                    break;
                }
                if (*vflag) break;
                const int64_t g = t0 + static_cast<int64_t>(i) * kPkStage;
                const int64_t left = t0 + ntok - g;
                const uint32_t L = static_cast<uint32_t>(left < kPkStage ? left : kPkStage);
                PkStage& st = ring[slot];
                mbar_arrive_expect_tx(full + slot, 16u * L);
                bulk_load(st.lt, a.lt + g, 4u * L, full + slot);
                bulk_load(st.lo, a.lo + g, 4u * L, full + slot);
                bulk_load(st.ls, a.ls + g, 4u * L, full + slot);
                bulk_load(st.A, a.adv + g, 4u * L, full + slot);
                issued = i + 1;
            }
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
        for (int i = 0; i < nst; ++i) {
            const int slot = i % kPkDepth;
            if (!mbar_wait(full + slot, static_cast<uint32_t>((i / kPkDepth) & 1), &blk_status, a.wait_ns)) {
                atomicExch(&abort_flag, 1);
                break;
            }
            if (*vflag) break;
            const int64_t g = t0 + static_cast<int64_t>(i) * kPkStage;
            if (g + j4 < t0 + ntok) {
                const PkStage& st = ring[slot];
                const float4 lt4 = *reinterpret_cast<const float4*>(st.lt + j4);
                const float4 lo4 = *reinterpret_cast<const float4*>(st.lo + j4);
                const float4 ls4 = *reinterpret_cast<const float4*>(st.ls + j4);
                const float4 A4 = *reinterpret_cast<const float4*>(st.A + j4);
                const float vt[4] = {lt4.x, lt4.y, lt4.z, lt4.w}, vo[4] = {lo4.x, lo4.y, lo4.z, lo4.w};
                const float vs[4] = {ls4.x, ls4.y, ls4.z, ls4.w}, vA[4] = {A4.x, A4.y, A4.z, A4.w};
                float lp[4], ld[4], gp[4], gd[4];
#pragma unroll
                for (int u = 0; u < 4; u += 2) {   // two tokens at a time: two independent chains, no branch
                    PgTok t[2] = {pg_fast_packed(vt[u], vo[u], vs[u], vA[u], q, lut, s_eps, s_weps),
                                  pg_fast_packed(vt[u + 1], vo[u + 1], vs[u + 1], vA[u + 1], q, lut, s_eps, s_weps)};
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
                        for (int k = 0; k < kPgSums; ++k) acc.sum[k] += t[h].s[k];
                        acc.cnt[1] += t[h].clip;
                        acc.cnt[2] += t[h].dual;
                        acc.cnt[3] += t[h].ice_lo;
                        acc.cnt[4] += t[h].ice_hi;
                        acc.cnt[5] += t[h].tis;
                        hist[t[h].j * kPgThreads] += 1;
                    }
                }
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
            const int64_t t = 4 * n4 + threadIdx.x;
            if (t < a.T) {
                float lp, ld, gp, gd;
                const float xt = a.lt[t], xo = a.lo[t], xs = a.ls[t], xa = a.adv[t];
                PgTok tk = pg_fast_packed(xt, xo, xs, xa, q, lut, s_eps, s_weps);
                if (tk.band) pg_resolve(tk, xt, xo, xs, xa, q);
                pg_take(tk, true, hist, acc, lp, ld, gp, gd);
                if (a.loss_ppo) a.loss_ppo[t] = lp;
                if (a.loss_dec) a.loss_dec[t] = ld;
                if (a.grad_ppo) a.grad_ppo[t] = gp;
                if (a.grad_dec) a.grad_dec[t] = gd;
            }
        }
    }
    pg_block_record(a, acc, hist_s, &blk_status);
    pg_finish(a, pk_smem, kPkSmem);   // the ring is idle now: scratch for the last block
}

// ----------------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------------
// Workspace: a 256-byte header (the arrival counter at byte 0: zero before the first call,
// and the last block of every call leaves it zero), then the blocks' partial records
// (PgRecords, one 128-byte record per block).  At most kPgMaxBlocks blocks run (fewer than two per SM on a part with
// more than 256 SMs), so the workspace size does not depend on the device.
constexpr size_t kPgHeader = 256;
static_assert(kPgHeader + sizeof(PgRecords) <= kPolicyWorkspaceBytes, "workspace layout");

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
    if ((reinterpret_cast<uintptr_t>(ws) & 15u) != 0) {
        set_last_error("workspace not 16-byte aligned");
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
    a.arrive = static_cast<unsigned int*>(ws);
    a.rec = reinterpret_cast<PgRecords*>(static_cast<uint8_t*>(ws) + kPgHeader);   // 16-byte aligned
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
