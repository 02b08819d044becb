// Rollout correction over a batch of sequences ("Rollout Correction Methods": "Config
// keys", "Importance Sampling", "Rejection Sampling" with the veto, "Mismatch Metrics"):
// per-token importance weights at token, sequence or geometric level, bounded by
// truncate / clip / mask, rejection sampling at any level, the veto, batch
// normalisation, and the IS / RS and mismatch-monitoring sums.
//
// Every decision (a bound, a rejection, the veto) is the exact predicate on the fp32
// inputs: a token's log-ratio d = lp_train - lp_rollout is formed exactly as a
// float-float pair, a sequence's sum of log-ratios (and, for sequence-level rejection,
// its sum of token weights) is carried in float-float, and each comparison is taken
// against a threshold's logarithm (or n times it) prepared on the host as a float-float
// pair.  Weight values are fp32.
//
//  1. rc_seq_kernel     one block per sequence: the sequence staged in shared memory (whole,
//                       by bulk copies, up to 4096 tokens; longer ones chunk by chunk), a
//                       pass over its tokens for the sequence sums, the sequence's
//                       decisions by one thread, a second pass writing weights and keep
//                       flags; one record of partial sums per sequence.  The last block of
//                       each group of 32 sequences to finish sums the group's records in
//                       sequence order, and the last group to finish sums the group records
//                       in group order: a fixed order, so the totals are reproducible.  That
//                       block writes the metrics and the batch-normalisation factor.
//  2. rc_scale_kernel   with batch normalisation: weights *= factor.
//  The counters the blocks meet at are set back to zero by the blocks that finish with
//  them, so a workspace zeroed once before its first use needs no clearing between calls.
#include <cmath>
#include <climits>

#include "common.cuh"
#include "ff.cuh"
#include "internal.h"

namespace rl {

constexpr int kRcThreads = 128;
// per-sequence record: double sums, int64 counts, then the kept weights' min and max
enum {
    RD_W_BEFORE, RD_W_AFTER, RD_KEPT_W, RD_MIS_KL, RD_K3, RD_ABS, RD_CHI2T, RD_TRAIN_LPPL, RD_ROLL_LPPL,
    RD_LPPL_DIFF, RD_LPPL_ABS, RD_PPL_RATIO, RD_CHI2S, kRcD
};
enum { RC_VALID, RC_SEQ, RC_KEPT, RC_TIS_LO, RC_TIS_HI, RC_RS_LO, RC_RS_HI, RC_CAT_TOK, RC_CAT_SEQ, kRcC };
constexpr int kRcFields = kRcD + kRcC + 2;   // + min, max

struct RcPrep {
    int use_tis, mode, level, norm, use_rs, rs_level, veto;
    float L, U, rsL, rsU;
    FF lnL, lnU, lnRsL, lnRsU, lnVeto;
};

struct RcArgs {
    const float* lt;
    const float* lr;
    const uint8_t* mask;
    const int64_t* off;
    int64_t B, T;
    RcPrep q;
    float* w;
    uint8_t* keep;
    double* pd;          // [kRcD][B]
    long long* pc;       // [kRcC][B]
    float* pmin;         // [B]
    float* pmax;         // [B]
    double* gd;          // [kRcD][G] the group records
    long long* gc;       // [kRcC][G]
    float* gmin;         // [G]
    float* gmax;         // [G]
    int64_t G;           // groups of kRcGroup sequences
    unsigned int* gcnt;  // [G] sequences of the group done (0 between calls)
    unsigned int* tcnt;  // groups done (0 between calls)
    int32_t* status;     // RL_STATUS_* bits of this call (0 between calls)
    float* factor;       // the batch-normalisation factor applied
    uint64_t wait_ns;    // limit of the staging wait
    rl_rc_metrics* metrics;
};
constexpr int kRcGroup = 32;   // sequences per first-level group of the reduction

// Fixed-order reductions: a butterfly within each warp (every lane ends with the same
// value, the same operands in the same order on both lanes of an exchange), then the
// warps in order by one thread.
RL_DEVINL float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
RL_DEVINL int warp_sum_i(int v) { return __reduce_add_sync(0xffffffffu, v); }
RL_DEVINL FF warp_sum_ff(FF v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const FF u = {__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
        v = (lane & o) ? ff_add(u, v) : ff_add(v, u);
    }
    return v;
}
// e^(hi + lo) for a float-float exponent: e^hi (float-float) times 1 + lo (|lo| tiny).
RL_DEVINL FF exp_ff2(FF d) { return ff_mul(exp_ff(d.hi), two_sum(1.f, d.lo)); }

struct RcSeq {   // one sequence's decisions (thread 0 -> block)
    int n, tis_lo, tis_hi, rs_lo, rs_hi, veto;
    float wseq;
};

// The factor and the metrics from the reduced fields (one thread).
RL_DEVINL void rc_write_metrics(const RcArgs& a, const double* t) {
    const double kept_w = t[RD_KEPT_W], n_kept = t[kRcD + RC_KEPT];
    const double factor = a.q.use_tis && a.q.norm && n_kept > 0 && kept_w > 0 ? n_kept / kept_w : 1.0;
    *a.factor = static_cast<float>(factor);
    rl_rc_metrics* m = a.metrics;
    if (!m) return;
    m->w_before_sum = t[RD_W_BEFORE];
    m->w_after_sum = t[RD_W_AFTER];
    m->kept_w_sum = kept_w;
    m->batch_norm_factor = factor;
    m->final_sum = kept_w * factor;
    m->final_min = n_kept > 0 ? t[kRcD + kRcC] * factor : 0.0;
    m->final_max = n_kept > 0 ? t[kRcD + kRcC + 1] * factor : 0.0;
    m->mis_kl_sum = t[RD_MIS_KL];
    m->k3_sum = t[RD_K3];
    m->abs_diff_sum = t[RD_ABS];
    m->chi2_token_sum = t[RD_CHI2T];
    m->train_lppl_sum = t[RD_TRAIN_LPPL];
    m->rollout_lppl_sum = t[RD_ROLL_LPPL];
    m->lppl_diff_sum = t[RD_LPPL_DIFF];
    m->lppl_abs_diff_sum = t[RD_LPPL_ABS];
    m->ppl_ratio_sum = t[RD_PPL_RATIO];
    m->chi2_seq_sum = t[RD_CHI2S];
    m->n_valid = static_cast<int64_t>(t[kRcD + RC_VALID]);
    m->n_seq = static_cast<int64_t>(t[kRcD + RC_SEQ]);
    m->n_kept = static_cast<int64_t>(n_kept);
    m->n_tis_low = static_cast<int64_t>(t[kRcD + RC_TIS_LO]);
    m->n_tis_high = static_cast<int64_t>(t[kRcD + RC_TIS_HI]);
    m->n_rs_low = static_cast<int64_t>(t[kRcD + RC_RS_LO]);
    m->n_rs_high = static_cast<int64_t>(t[kRcD + RC_RS_HI]);
    m->n_cat_tokens = static_cast<int64_t>(t[kRcD + RC_CAT_TOK]);
    m->n_cat_seqs = static_cast<int64_t>(t[kRcD + RC_CAT_SEQ]);
    m->status = *a.status;
}

// A sequence of up to kRcChunk tokens is staged in shared memory whole, by bulk copies
// when the arrays are 16-byte aligned (the aligned body; the few tokens past its last
// 16-byte boundary by plain loads), and read from there by both passes.  A longer one is
// staged kRcChunk tokens at a time with plain coalesced loads, chunk by chunk in each pass
// (pass 2 starts from the chunk still staged).  A bulk copy must start on a 16-byte
// boundary: it starts at the boundary at or before the sequence's first token and the
// sequence sits at a small offset in the buffer (0..3 floats, 0..15 mask bytes).  128
// threads and 37 KB of shared memory keep six blocks on an SM.  Loops stay rolled: the
// code is fetched cold by every block, so its size is part of the latency.
constexpr int kRcChunk = 4096;
constexpr int kRcW = kRcThreads / 32;

// The sums of up to 32 records (a group of sequence records, or the group records), as a
// fixed-shape warp tree: lane l takes record r0 + l (a lane past r1 contributes the
// identity), then a butterfly of five levels in which both lanes of an exchange add the
// same operands in the same order, so the result does not depend on scheduling.  A warp
// takes fields f = warp, warp + 4, ... (fp64 sums, int64 counts, min, max): five dependent
// fp64 additions per field rather than one per record (fp64 is a slow pipe on this part).
// Lane 0's results go to dsum / csum / mn / mx (shared, indexed by field).
// Record fields that need the fp64 range (a sequence-level weight e^S n, chi^2 e^(2 S));
// the others are sums of fp32 values and are carried as float-float pairs in their 8 bytes.
RL_DEVINL constexpr bool rc_wide(int f) { return f == RD_W_BEFORE || f == RD_CHI2S; }

struct RcRecs {
    const double* d;
    const long long* c;
    const float* mn;
    const float* mx;
    int64_t ld;
};
RL_DEVINL void rc_sum_records(const RcRecs& r, int64_t r0, int64_t r1, double* dsum, long long* csum, float* mnmx) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t i = r0 + lane;
    const bool in = i < r1;
    constexpr int kPer = (kRcFields + kRcW - 1) / kRcW;
    // every load of the warp's fields first (one round trip to L2 rather than one per field)
    unsigned long long raw[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int f = warp + kRcW * k;
        raw[k] = 0ull;
        if (in && f < kRcFields) {
            if (f < kRcD)
                raw[k] = __ldcg(reinterpret_cast<const unsigned long long*>(r.d) + f * r.ld + i);
            else if (f < kRcD + kRcC)
                raw[k] = __ldcg(reinterpret_cast<const unsigned long long*>(r.c) + (f - kRcD) * r.ld + i);
            else
                raw[k] = __float_as_uint(__ldcg((f == kRcD + kRcC ? r.mn : r.mx) + i));
        }
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int f = warp + kRcW * k;
        if (f >= kRcFields) continue;
        if (f < kRcD && rc_wide(f)) {
            double v = __longlong_as_double(static_cast<long long>(raw[k]));
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double u = __shfl_xor_sync(0xffffffffu, v, o);
                v = (lane & o) ? u + v : v + u;
            }
            if (lane == 0) dsum[f] = v;
        } else if (f < kRcD) {
            FF v = {__uint_as_float(static_cast<unsigned>(raw[k])), __uint_as_float(static_cast<unsigned>(raw[k] >> 32))};
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const FF u = {__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
                v = (lane & o) ? ff_add(u, v) : ff_add(v, u);
            }
            if (lane == 0)
                dsum[f] = __longlong_as_double(static_cast<long long>(__float_as_uint(v.hi)) |
                                               (static_cast<long long>(__float_as_uint(v.lo)) << 32));
        } else if (f < kRcD + kRcC) {
            long long v = static_cast<long long>(raw[k]);
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) csum[f - kRcD] = v;
        } else {
            const bool is_min = f == kRcD + kRcC;
            float v = in ? __uint_as_float(static_cast<unsigned>(raw[k])) : (is_min ? INFINITY : -INFINITY);
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float u = __shfl_xor_sync(0xffffffffu, v, o);
                v = is_min ? fminf(v, u) : fmaxf(v, u);
            }
            if (lane == 0) mnmx[f - kRcD - kRcC] = v;
        }
    }
}

__global__ void __launch_bounds__(kRcThreads, 6) rc_seq_kernel(RcArgs a) {
    __shared__ __align__(16) float s_lt[kRcChunk + 4];
    __shared__ __align__(16) float s_lr[kRcChunk + 4];
    __shared__ __align__(16) uint8_t s_m[kRcChunk + 16];
    __shared__ __align__(8) uint64_t bar;
    __shared__ FF shff[kRcW][4];
    __shared__ float shf[kRcW][5];
    __shared__ int shi[kRcW][6];
    __shared__ RcSeq sq;
    __shared__ int role;
    const RcPrep& q = a.q;
    const int64_t b = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t o0 = a.off[b], o1 = a.off[b + 1];
    const bool bad = o0 < 0 || o1 < o0 || o1 > a.T || (b == 0 && o0 != 0) || (b == a.B - 1 && o1 != a.T);
    if (bad) {
        if (threadIdx.x == 0) set_status(a.status, RL_STATUS_OFFSETS);
        o0 = o0 < 0 ? 0 : (o0 > a.T ? a.T : o0);
        o1 = o1 < o0 ? o0 : (o1 > a.T ? a.T : o1);
    }
    const bool rs_seq = q.use_rs && q.rs_level == RL_LEVEL_SEQUENCE;
    const int64_t len = o1 - o0;
    const int nchunks = static_cast<int>((len + kRcChunk - 1) / kRcChunk);
    // token i of the staged chunk is s_lt[fo + i], s_lr[fo + i], s_m[mo + i]
    int fo = 0, mo = 0;
    const bool whole = nchunks == 1 &&
                       ((reinterpret_cast<uintptr_t>(a.lt) | reinterpret_cast<uintptr_t>(a.lr) |
                         reinterpret_cast<uintptr_t>(a.mask)) & 15) == 0;
    if (whole) {
        // the bodies from the 16-byte boundary at or before o0 to the last one at or before
        // o1 by bulk copies, the rest of the sequence by plain loads
        const int64_t f0 = o0 & ~int64_t(3), f1 = o1 & ~int64_t(3);
        const int64_t m0 = o0 & ~int64_t(15), m1 = o1 & ~int64_t(15);
        fo = static_cast<int>(o0 - f0);
        mo = static_cast<int>(o0 - m0);
        const uint32_t fb = static_cast<uint32_t>(4 * (f1 - f0)), mb = static_cast<uint32_t>(m1 - m0);
        if (threadIdx.x == 0) {
            mbar_init(&bar, 1);
            fence_mbar_init();
            mbar_arrive_expect_tx(&bar, 2 * fb + mb);
            if (fb > 0) {
                bulk_load(s_lt, a.lt + f0, fb, &bar);
                bulk_load(s_lr, a.lr + f0, fb, &bar);
            }
            if (mb > 0) bulk_load(s_m, a.mask + m0, mb, &bar);
        }
        for (int64_t t = (f1 > o0 ? f1 : o0) + threadIdx.x; t < o1; t += kRcThreads) {
            s_lt[fo + (t - o0)] = a.lt[t];
            s_lr[fo + (t - o0)] = a.lr[t];
        }
        for (int64_t t = (m1 > o0 ? m1 : o0) + threadIdx.x; t < o1; t += kRcThreads) s_m[mo + (t - o0)] = a.mask[t];
        __syncthreads();   // the barrier's initialisation is visible
        if (!mbar_wait(&bar, 0, a.status, a.wait_ns)) {
            // a copy that never completed: the block's results are incomplete (the status
            // says so); wait once more, bounded, for the copies before leaving
            if (threadIdx.x == 0) mbar_wait(&bar, 0, a.status);
        }
        __syncthreads();
    }
    auto stage = [&](int c) {   // chunk c into shared memory (plain loads); returns its length
        const int64_t c0 = o0 + static_cast<int64_t>(c) * kRcChunk;
        const int n = static_cast<int>(o1 - c0 < kRcChunk ? o1 - c0 : kRcChunk);
        const float* lt = a.lt + c0;
        const float* lr = a.lr + c0;
        const uint8_t* mk = a.mask + c0;
        int i0 = 0;
        if ((((reinterpret_cast<uintptr_t>(lt) | reinterpret_cast<uintptr_t>(lr)) & 15) |
             (reinterpret_cast<uintptr_t>(mk) & 3)) == 0) {
            // 16-byte loads (4-byte for the mask)
            const int n4 = n >> 2;
#pragma unroll 4
            for (int i = threadIdx.x; i < n4; i += kRcThreads) {
                const float4 x = reinterpret_cast<const float4*>(lt)[i];
                const float4 y = reinterpret_cast<const float4*>(lr)[i];
                const uchar4 m = reinterpret_cast<const uchar4*>(mk)[i];
                reinterpret_cast<float4*>(s_lt)[i] = x;
                reinterpret_cast<float4*>(s_lr)[i] = y;
                reinterpret_cast<uchar4*>(s_m)[i] = m;
            }
            i0 = 4 * n4;
        }
#pragma unroll 4
        for (int i = i0 + threadIdx.x; i < n; i += kRcThreads) {
            s_lt[i] = lt[i];
            s_lr[i] = lr[i];
            s_m[i] = mk[i];
        }
        __syncthreads();
        return n;
    };

    // pass 1: the sequence's sums.  Two accumulator sets per thread (tokens i and
    // i + 128 of each step), added in that order at the end: two independent float-float
    // chains in flight instead of one.
    int n = 0, cat = 0;
    FF S = {0.f, 0.f}, E = {0.f, 0.f};   // the decisions' sums, float-float
    FF S2 = {0.f, 0.f}, E2 = {0.f, 0.f};
    float st = 0.f, sr = 0.f;            // metric sums: fp32 per thread
    float mis = 0.f, k3 = 0.f, ad = 0.f, c2 = 0.f;
    auto take = [&](int i, FF& Sx, FF& Ex) {
        if (s_m[mo + i] == 0) return;
        const float x = s_lt[fo + i], y = s_lr[fo + i];
        const FF d = two_sum(x, -y);
        ++n;
        Sx = ff_add(Sx, d);
        st += x;
        sr += y;
        if (rs_seq) Ex = ff_add(Ex, exp_ff2(d));
        if (q.veto) cat += ff_lt(d, q.lnVeto) ? 1 : 0;
        const float df = d.hi;
        const float ed = expf(df);
        mis -= df;
        k3 += ed - df - 1.f;
        ad += fabsf(df);
        c2 += ed * ed;
    };
    int staged = whole ? 0 : -1;
    for (int c = 0; c < nchunks; ++c) {
        int cn;
        if (c == staged) {
            cn = static_cast<int>(len);
        } else {
            if (c > 0) __syncthreads();   // the previous chunk's readers are done
            cn = stage(c);
            staged = c;
        }
#pragma unroll 1
        for (int i = threadIdx.x; i < cn; i += 2 * kRcThreads) {
            take(i, S, E);
            if (i + kRcThreads < cn) take(i + kRcThreads, S2, E2);
        }
    }
    S = ff_add(S, S2);
    E = ff_add(E, E2);
    {
        const FF w4[4] = {warp_sum_ff(S), rs_seq ? warp_sum_ff(E) : FF{0.f, 0.f}, {warp_sum_f(st), 0.f},
                          {warp_sum_f(sr), 0.f}};
        const float f4[4] = {warp_sum_f(mis), warp_sum_f(k3), warp_sum_f(ad), warp_sum_f(c2)};
        const int i2[2] = {warp_sum_i(n), warp_sum_i(cat)};
        if (lane == 0) {
            for (int f = 0; f < 4; ++f) shff[warp][f] = w4[f];
            for (int f = 0; f < 4; ++f) shf[warp][f] = f4[f];
            for (int f = 0; f < 2; ++f) shi[warp][f] = i2[f];
        }
    }
    __syncthreads();
    double seqd[2] = {0, 0};                   // w_before (sequence levels), chi2_seq: fp64 range
    float seqf[5] = {0.f, 0.f, 0.f, 0.f, 0.f};   // the log-perplexity terms
    float tok1[4] = {0.f, 0.f, 0.f, 0.f};      // mis, k3, |d|, e^2d
    int nt = 0, catt = 0;
    if (threadIdx.x == 0) {
        FF R[4] = {shff[0][0], shff[0][1], shff[0][2], shff[0][3]};
        for (int f = 0; f < 4; ++f) tok1[f] = shf[0][f];
        nt = shi[0][0];
        catt = shi[0][1];
        for (int w = 1; w < kRcW; ++w) {
            for (int f = 0; f < 4; ++f) R[f] = ff_add(R[f], shff[w][f]);
            for (int f = 0; f < 4; ++f) tok1[f] += shf[w][f];
            nt += shi[w][0];
            catt += shi[w][1];
        }
        const FF Sb = R[0], Eb = R[1], Stb = R[2], Srb = R[3];
        RcSeq s{};
        s.n = nt;
        if (nt > 0) {
            // fp32 and float-float here: fp64 is a slow pipe on this part and this thread
            // is on the block's critical path
            const FF nf = {static_cast<float>(nt), 0.f};   // exact below 2^24 tokens per sequence
            const float rn = 1.f / static_cast<float>(nt);
            if (q.level == RL_LEVEL_SEQUENCE) {
                s.tis_lo = ff_lt(Sb, q.lnL);
                s.tis_hi = ff_gt(Sb, q.lnU);
                s.wseq = expf(Sb.hi) * (1.f + Sb.lo);
                seqd[0] = Sb.hi < 88.f ? static_cast<double>(s.wseq) * nt : exp(static_cast<double>(Sb.hi)) * nt;
            } else if (q.level == RL_LEVEL_GEOMETRIC) {
                s.tis_lo = ff_lt(Sb, ff_mul(nf, q.lnL));
                s.tis_hi = ff_gt(Sb, ff_mul(nf, q.lnU));
                s.wseq = expf((Sb.hi + Sb.lo) * rn);
                seqd[0] = static_cast<double>(s.wseq) * nt;
            }
            if (q.use_rs && q.rs_level == RL_LEVEL_SEQUENCE) {   // mean token weight vs the bounds
                s.rs_lo = ff_lt(Eb, two_prod(static_cast<float>(nt), q.rsL));
                s.rs_hi = !s.rs_lo && ff_gt(Eb, two_prod(static_cast<float>(nt), q.rsU));
            } else if (q.use_rs && q.rs_level == RL_LEVEL_GEOMETRIC) {
                s.rs_lo = ff_lt(Sb, ff_mul(nf, q.lnRsL));
                s.rs_hi = !s.rs_lo && ff_gt(Sb, ff_mul(nf, q.lnRsU));
            }
            s.veto = catt > 0;
            const float tr = -(Stb.hi + Stb.lo) * rn;
            const float ro = -(Srb.hi + Srb.lo) * rn;
            const float df = -(Sb.hi + Sb.lo) * rn;   // tr - ro = -S / n, from the exact sum of d
            seqf[0] = tr;
            seqf[1] = ro;
            seqf[2] = df;
            seqf[3] = fabsf(df);
            seqf[4] = expf(df);
            // e^(2 S): fp32 while it fits, fp64 (one call) past the fp32 range
            seqd[1] = Sb.hi < 44.f ? static_cast<double>(expf(2.f * Sb.hi) * (1.f + 2.f * Sb.lo))
                                   : exp(2.0 * (static_cast<double>(Sb.hi) + static_cast<double>(Sb.lo)));
        }
        sq = s;
    }
    __syncthreads();
    const RcSeq s = sq;

    // pass 2: weights and keep flags (the staged chunk is reused when it is the only one)
    float wb_sum = 0.f, kept_sum = 0.f, wraw_sum = 0.f, mn = INFINITY, mx = -INFINITY;
    int kept = 0, tlo = 0, thi = 0, rlo = 0, rhi = 0;
    // the last chunk of pass 1 is still staged: take the chunks from the last one down
    for (int c = nchunks - 1; c >= 0; --c) {
        int cn;
        if (c == staged) {
            const int64_t rest = len - static_cast<int64_t>(c) * kRcChunk;
            cn = static_cast<int>(rest < kRcChunk ? rest : kRcChunk);
        } else {
            __syncthreads();
            cn = stage(c);
            staged = c;
        }
        const int64_t c0 = o0 + static_cast<int64_t>(c) * kRcChunk;
#pragma unroll 1
        for (int i = threadIdx.x; i < cn; i += kRcThreads) {
            float wout = 0.f;
            uint8_t kp8 = 0;
            if (s_m[mo + i] != 0) {
                const bool tok = q.level == RL_LEVEL_TOKEN || (q.use_rs && q.rs_level == RL_LEVEL_TOKEN);
                const FF d = tok ? two_sum(s_lt[fo + i], -s_lr[fo + i]) : FF{0.f, 0.f};
                float w;
                bool lo, hi;
                if (q.level == RL_LEVEL_TOKEN) {
                    w = expf(d.hi) * (1.f + d.lo);
                    lo = ff_lt(d, q.lnL);
                    hi = ff_gt(d, q.lnU);
                    wraw_sum += w;
                } else {
                    w = s.wseq;
                    lo = s.tis_lo;
                    hi = s.tis_hi;
                }
                float wb;
                if (!q.use_tis)
                    wb = 1.f;
                else if (q.mode == RL_TIS_TRUNCATE)
                    wb = hi ? q.U : w;
                else if (q.mode == RL_TIS_CLIP)
                    wb = lo ? q.L : (hi ? q.U : w);
                else
                    wb = (lo || hi) ? 0.f : w;
                bool r_lo = false, r_hi = false;
                if (q.use_rs && q.rs_level == RL_LEVEL_TOKEN) {
                    r_lo = ff_lt(d, q.lnRsL);
                    r_hi = !r_lo && ff_gt(d, q.lnRsU);
                } else if (q.use_rs) {
                    r_lo = s.rs_lo;
                    r_hi = s.rs_hi;
                }
                tlo += lo;
                thi += hi;
                rlo += r_lo;
                rhi += r_hi;
                wb_sum += wb;
                if (!r_lo && !r_hi && !s.veto) {
                    kp8 = 1;
                    wout = wb;
                    ++kept;
                    kept_sum += wb;
                    mn = fminf(mn, wb);
                    mx = fmaxf(mx, wb);
                }
            }
            if (a.w) a.w[c0 + i] = wout;
            if (a.keep) a.keep[c0 + i] = kp8;
        }
    }
    {
        float f5[5] = {warp_sum_f(wb_sum), warp_sum_f(kept_sum), warp_sum_f(wraw_sum), mn, mx};
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            f5[3] = fminf(f5[3], __shfl_xor_sync(0xffffffffu, f5[3], o));
            f5[4] = fmaxf(f5[4], __shfl_xor_sync(0xffffffffu, f5[4], o));
        }
        const int i5[5] = {warp_sum_i(kept), warp_sum_i(tlo), warp_sum_i(thi), warp_sum_i(rlo), warp_sum_i(rhi)};
        __syncthreads();   // the shared rows of pass 1 are read
        if (lane == 0) {
            for (int f = 0; f < 5; ++f) shf[warp][f] = f5[f];
            for (int f = 0; f < 5; ++f) shi[warp][f] = i5[f];
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float F[5];
        int I[5];
        for (int f = 0; f < 5; ++f) F[f] = shf[0][f];
        for (int f = 0; f < 5; ++f) I[f] = shi[0][f];
        for (int w = 1; w < kRcW; ++w) {
            for (int f = 0; f < 3; ++f) F[f] += shf[w][f];
            F[3] = fminf(F[3], shf[w][3]);
            F[4] = fmaxf(F[4], shf[w][4]);
            for (int f = 0; f < 5; ++f) I[f] += shi[w][f];
        }
        const int64_t B = a.B;
        // the two fp64-range fields as doubles, the others as float-float pairs (lo = 0)
        a.pd[RD_W_BEFORE * B + b] = q.level == RL_LEVEL_TOKEN ? static_cast<double>(F[2]) : seqd[0];
        a.pd[RD_CHI2S * B + b] = seqd[1];
        const float nf[kRcD] = {0.f, F[0], F[1], tok1[0], tok1[1], tok1[2], tok1[3],
                                seqf[0], seqf[1], seqf[2], seqf[3], seqf[4], 0.f};
        for (int f = 0; f < kRcD; ++f)
            if (!rc_wide(f)) reinterpret_cast<float2*>(a.pd)[f * B + b] = make_float2(nf[f], 0.f);
        const long long c[kRcC] = {nt, nt > 0 ? 1 : 0, I[0], I[1], I[2], I[3], I[4], catt, catt > 0 ? 1 : 0};
        for (int f = 0; f < kRcC; ++f) a.pc[f * B + b] = c[f];
        a.pmin[b] = F[3];
        a.pmax[b] = F[4];
        // count the sequence in with its group: release (the record) and acquire (if this is
        // the group's last, the other blocks' records)
        const int64_t g = b / kRcGroup;
        const int64_t gsize = a.B - g * kRcGroup < kRcGroup ? a.B - g * kRcGroup : kRcGroup;
        unsigned int old;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(a.gcnt + g) : "memory");
        role = old == static_cast<unsigned int>(gsize - 1);
    }
    __syncthreads();
    // the scaling kernel may be scheduled from here on (it waits for this grid to end)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (!role) return;
    // the group's last block: its records into group record g
    __shared__ double dsum[kRcD];
    __shared__ long long csum[kRcC];
    __shared__ float mnmx[2];
    {
        const int64_t g = b / kRcGroup;
        const int64_t r0 = g * kRcGroup, r1 = r0 + kRcGroup < a.B ? r0 + kRcGroup : a.B;
        rc_sum_records(RcRecs{a.pd, a.pc, a.pmin, a.pmax, a.B}, r0, r1, dsum, csum, mnmx);
        __syncthreads();
        const int f = threadIdx.x;
        if (f < kRcD) a.gd[f * a.G + g] = dsum[f];
        else if (f < kRcD + kRcC) a.gc[(f - kRcD) * a.G + g] = csum[f - kRcD];
        else if (f == kRcD + kRcC) a.gmin[g] = mnmx[0];
        else if (f == kRcD + kRcC + 1) a.gmax[g] = mnmx[1];
        __syncthreads();
        if (threadIdx.x == 0) {
            a.gcnt[g] = 0u;   // for the next call
            unsigned int old;
            asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(a.tcnt) : "memory");
            role = old == static_cast<unsigned int>(a.G - 1);
        }
        __syncthreads();
        if (!role) return;
    }
    // the last group: the group records (32 at a time, the partial totals added in group
    // order), then the factor and the metrics
    {
        __shared__ double tot[kRcFields];
        for (int64_t g0 = 0; g0 < a.G; g0 += 32) {
            rc_sum_records(RcRecs{a.gd, a.gc, a.gmin, a.gmax, a.G}, g0, g0 + 32 < a.G ? g0 + 32 : a.G, dsum, csum, mnmx);
            __syncthreads();
            const int f = threadIdx.x;
            if (f < kRcFields) {
                double x;
                if (f < kRcD && !rc_wide(f)) {   // a float-float pair in the slot's bits
                    const long long bits = __double_as_longlong(dsum[f]);
                    x = static_cast<double>(__uint_as_float(static_cast<unsigned>(bits))) +
                        static_cast<double>(__uint_as_float(static_cast<unsigned>(bits >> 32)));
                } else {
                    x = f < kRcD ? dsum[f] : (f < kRcD + kRcC ? static_cast<double>(csum[f - kRcD]) : mnmx[f - kRcD - kRcC]);
                }
                if (g0 == 0) tot[f] = x;
                else if (f < kRcD + kRcC) tot[f] += x;
                else if (f == kRcD + kRcC) tot[f] = fmin(tot[f], x);
                else tot[f] = fmax(tot[f], x);
            }
            __syncthreads();
        }
        if (threadIdx.x == 0) {
            rc_write_metrics(a, tot);
            *a.status = 0;     // for the next call
            *a.tcnt = 0u;
        }
    }
}



// No sequence: zero sums, factor 1 (one thread).
__global__ void rc_empty_kernel(RcArgs a) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    double t[kRcFields];
    for (int f = 0; f < kRcFields; ++f) t[f] = 0.0;
    rc_write_metrics(a, t);
    *a.status = 0;
}

// Batch normalisation: w *= factor, float4 over the 16-byte-aligned body (four loads in
// flight per thread) and scalars at the two ends.
constexpr int kRcScaleThreads = 256;
__global__ void __launch_bounds__(kRcScaleThreads) rc_scale_kernel(RcArgs a) {
    // launched as a programmatic dependent of the sequence kernel: it may be resident
    // before that kernel ends, and waits here (in hardware) until it has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const float f = *a.factor;
    float* w = a.w;
    const int64_t T = a.T;
    const int64_t head = ((16 - (reinterpret_cast<uintptr_t>(w) & 15)) & 15) / 4;
    const int64_t h = head < T ? head : T;
    const int64_t n4 = (T - h) / 4;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nth = static_cast<int64_t>(gridDim.x) * blockDim.x;
    float4* w4 = reinterpret_cast<float4*>(w + h);
#pragma unroll 4
    for (int64_t i = tid; i < n4; i += nth) {
        float4 v = w4[i];
        v.x *= f;
        v.y *= f;
        v.z *= f;
        v.w *= f;
        w4[i] = v;
    }
    if (tid < h) w[tid] *= f;
    const int64_t t0 = h + 4 * n4;
    if (tid < T - t0) w[t0 + tid] *= f;
}

// ----------------------------------------------------------------------------------
// Named metrics ("Mismatch Metrics" tables) from the sums and counts
// ----------------------------------------------------------------------------------
struct RcEmit {
    int use_tis, mode, use_rs, veto;
};

// Mean of a sum over a count; an empty set gives 0.
RL_DEVINL double rc_mean(double sum, int64_t n) { return n > 0 ? sum / static_cast<double>(n) : 0.0; }

__global__ void rc_named_kernel(const rl_rc_metrics* m, RcEmit e, rl_rc_named* o) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    const double nan = __longlong_as_double(0x7ff8000000000000ll);
    const int64_t nv = m->n_valid, ns = m->n_seq, nk = m->n_kept;
    // per-sequence log-perplexities averaged over sequences, perplexity = exp(average)
    const double tr = rc_mean(m->train_lppl_sum, ns), ro = rc_mean(m->rollout_lppl_sum, ns);
    o->training_log_ppl = tr;
    o->training_ppl = exp(tr);
    o->rollout_log_ppl = ro;
    o->rollout_ppl = exp(ro);
    o->kl = rc_mean(m->mis_kl_sum, nv);
    o->k3_kl = rc_mean(m->k3_sum, nv);
    o->log_ppl_diff = rc_mean(m->lppl_diff_sum, ns);
    o->log_ppl_abs_diff = rc_mean(m->lppl_abs_diff_sum, ns);
    o->ppl_ratio = rc_mean(m->ppl_ratio_sum, ns);
    // chi^2 under the rollout policy: E[w^2] - 1 (nothing to average over: 0)
    o->chi2_token = nv > 0 ? m->chi2_token_sum / static_cast<double>(nv) - 1.0 : 0.0;
    o->chi2_seq = ns > 0 ? m->chi2_seq_sum / static_cast<double>(ns) - 1.0 : 0.0;
    o->train_rollout_logprob_abs_diff = rc_mean(m->abs_diff_sum, nv);
    const double lo = rc_mean(static_cast<double>(m->n_tis_low), nv);
    const double hi = rc_mean(static_cast<double>(m->n_tis_high), nv);
    o->tis_weight_before_bound = e.use_tis ? rc_mean(m->w_before_sum, nv) : nan;
    o->tis_weight_after_bound = e.use_tis ? rc_mean(m->w_after_sum, nv) : nan;
    o->tis_truncate_fraction = e.use_tis && e.mode == RL_TIS_TRUNCATE ? hi : nan;
    o->tis_clip_fraction_low = e.use_tis && e.mode == RL_TIS_CLIP ? lo : nan;
    o->tis_clip_fraction_high = e.use_tis && e.mode == RL_TIS_CLIP ? hi : nan;
    o->tis_mask_fraction_low = e.use_tis && e.mode == RL_TIS_MASK ? lo : nan;
    o->tis_mask_fraction_high = e.use_tis && e.mode == RL_TIS_MASK ? hi : nan;
    o->rs_mask_fraction_low = e.use_rs ? rc_mean(static_cast<double>(m->n_rs_low), nv) : nan;
    o->rs_mask_fraction_high = e.use_rs ? rc_mean(static_cast<double>(m->n_rs_high), nv) : nan;
    o->rs_catastrophic_token_fraction = e.veto ? rc_mean(static_cast<double>(m->n_cat_tokens), nv) : nan;
    o->rs_catastrophic_seq_fraction = e.veto ? rc_mean(static_cast<double>(m->n_cat_seqs), ns) : nan;
    o->is_ratio_mean_after_tis_rs = e.use_tis ? rc_mean(m->kept_w_sum, nk) : nan;
    o->batch_norm_factor = e.use_tis ? m->batch_norm_factor : nan;
    o->is_ratio_mean_final = e.use_tis ? rc_mean(m->final_sum, nk) : nan;
    o->is_ratio_min_final = e.use_tis ? m->final_min : nan;
    o->is_ratio_max_final = e.use_tis ? m->final_max : nan;
}

int rollout_named_impl(const rl_rc_metrics* m, const rl_rc_params* p, rl_rc_named* named, cudaStream_t stream) {
    RcEmit e;
    e.use_tis = p->use_tis != 0;
    e.mode = p->tis_mode;
    e.use_rs = p->use_rs != 0;
    e.veto = p->rs_veto_threshold > 0.f;   // NaN compares false: no veto, as rl_rollout_correction
    {
        ProfScope ps(RL_PROF_ROLLOUT, stream);
        rc_named_kernel<<<1, 32, 0, stream>>>(m, e, named);
    }
    count_launch();
    return cudaPeekAtLastError() == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}

// ----------------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------------
// Workspace: a 256-byte header (the group counter at byte 0, the status word at 4, the
// factor at 8), the per-sequence records, the group records and the per-group counters.
// Zero before the first call; every call leaves the counters and the status word at zero.
constexpr size_t kRcHeader = 256;

static size_t rc_record_bytes(int64_t n) {   // n records of kRcD fp64, kRcC int64, min, max
    return align_up(static_cast<size_t>(n) * (kRcD * 8 + kRcC * 8 + 2 * 4) + 64, 256);
}
static int64_t rc_groups(int64_t B) { return (B + kRcGroup - 1) / kRcGroup; }

size_t rollout_ws_bytes(int64_t B) {
    const int64_t b = B < 1 ? 1 : B, G = rc_groups(b);
    return kRcHeader + rc_record_bytes(b) + rc_record_bytes(G) + align_up(static_cast<size_t>(G) * 4, 256);
}

int rollout_impl(const float* lt, const float* lr, const uint8_t* mask, const int64_t* off, int64_t B, int64_t T,
                 const rl_rc_params* p, float* w, uint8_t* keep, rl_rc_metrics* metrics, void* ws,
                 size_t ws_bytes, cudaStream_t stream) {
    if (ws_bytes < rollout_ws_bytes(B)) return RL_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 7u) != 0) {
        set_last_error("rollout-correction workspace not 8-byte aligned");
        return RL_ERR_ARG;
    }
    RcArgs a{};
    a.lt = lt;
    a.lr = lr;
    a.mask = mask;
    a.off = off;
    a.B = B;
    a.T = T;
    RcPrep& q = a.q;
    q.use_tis = p->use_tis != 0;
    q.mode = p->tis_mode;
    q.level = p->tis_level;
    q.norm = p->tis_batch_normalize != 0;
    q.use_rs = p->use_rs != 0;
    q.rs_level = p->rs_level;
    q.L = p->tis_lower_bound;
    q.U = p->tis_upper_bound;
    q.rsL = std::isnan(p->rs_lower_bound) ? q.L : p->rs_lower_bound;
    q.rsU = std::isnan(p->rs_upper_bound) ? q.U : p->rs_upper_bound;
    q.veto = p->rs_veto_threshold > 0.f;   // NaN compares false: no veto
    q.lnL = ln_ff(q.L);
    q.lnU = ln_ff(q.U);
    q.lnRsL = ln_ff(q.rsL);
    q.lnRsU = ln_ff(q.rsU);
    q.lnVeto = ln_ff(q.veto ? p->rs_veto_threshold : 0.0);
    a.w = w;
    a.keep = keep;
    uint8_t* base = static_cast<uint8_t*>(ws);
    a.tcnt = reinterpret_cast<unsigned int*>(base);
    a.status = reinterpret_cast<int32_t*>(base + 4);
    a.factor = reinterpret_cast<float*>(base + 8);
    const int64_t b1 = B < 1 ? 1 : B;
    a.G = rc_groups(b1);
    uint8_t* rec = base + kRcHeader;
    a.pd = reinterpret_cast<double*>(rec);
    a.pc = reinterpret_cast<long long*>(a.pd + kRcD * b1);
    a.pmin = reinterpret_cast<float*>(a.pc + kRcC * b1);
    a.pmax = a.pmin + b1;
    uint8_t* grec = rec + rc_record_bytes(b1);
    a.gd = reinterpret_cast<double*>(grec);
    a.gc = reinterpret_cast<long long*>(a.gd + kRcD * a.G);
    a.gmin = reinterpret_cast<float*>(a.gc + kRcC * a.G);
    a.gmax = a.gmin + a.G;
    a.gcnt = reinterpret_cast<unsigned int*>(grec + rc_record_bytes(a.G));
    a.wait_ns = wait_limit_ns();
    a.metrics = metrics;
    ProfScope ps(RL_PROF_ROLLOUT, stream);   // the kernel launches
    int launches = 1;
    if (B > 0)
        rc_seq_kernel<<<static_cast<unsigned>(B), kRcThreads, 0, stream>>>(a);
    else
        rc_empty_kernel<<<1, 32, 0, stream>>>(a);
    if (q.use_tis && q.norm && w != nullptr && T > 0) {
        const int64_t blocks = (T / 4 + kRcScaleThreads - 1) / kRcScaleThreads + 1;
        const int64_t cap = 4L * num_sms();
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(blocks < cap ? blocks : cap), 1, 1);
        cfg.blockDim = dim3(kRcScaleThreads, 1, 1);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = B > 0 ? 1 : 0;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, rc_scale_kernel, a) != cudaSuccess) return RL_ERR_CUDA;
        ++launches;
    }
    count_launch(launches);
    return cudaPeekAtLastError() == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}

}  // namespace rl
