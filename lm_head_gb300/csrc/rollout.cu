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
//  1. rc_seq_kernel     one block per sequence: a pass over its tokens for the sequence
//                       sums, the sequence's decisions by one thread, a second pass (the
//                       tokens are now in L2) writing weights and keep flags; one record
//                       of partial sums per sequence.
//  2. rc_reduce_kernel  one block, one warp per field: the records summed in sequence
//                       order (fixed tree), so results are reproducible; then the
//                       metrics.  Without batch normalisation only.
//  2'. rc_scale_kernel  with batch normalisation, instead: every block forms the factor
//                       from the records in the same order (block 0 also all fields and
//                       the metrics), then weights *= factor.
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
    int32_t* status;
    float* factor;       // the batch-normalisation factor applied
    // batch normalisation: kept tokens and their weight sum over all sequences, exact
    // integer totals (the weight in 2^-24 fixed point); kept_range set if a sequence's sum
    // was too large for that (the factor then comes from the ordered record reduction)
    long long* kept_n;
    long long* kept_wfix;
    int* kept_range;
    float kept_lim;
    rl_rc_metrics* metrics;
};

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
template <typename T, typename Op>
RL_DEVINL T rc_block_reduce(T v, T* sh, Op op) {   // sh: one slot per warp
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if (lane == 0) sh[warp] = v;
    __syncthreads();
    T r = sh[0];
    for (int i = 1; i < nw; ++i) r = op(r, sh[i]);
    return r;
}

// e^(hi + lo) for a float-float exponent: e^hi (float-float) times 1 + lo (|lo| tiny).
RL_DEVINL FF exp_ff2(FF d) { return ff_mul(exp_ff(d.hi), two_sum(1.f, d.lo)); }

struct RcSeq {   // one sequence's decisions (thread 0 -> block)
    int n, tis_lo, tis_hi, rs_lo, rs_hi, veto;
    float wseq;
};

// A sequence is staged in shared memory kRcChunk tokens at a time (coalesced loads, 16
// bytes wide where the chunk is aligned, scalar otherwise); a sequence of at most kRcChunk tokens is read from memory once
// for both passes, a longer one chunk by chunk in each pass (pass 2 starts from the chunk
// still staged; the earlier ones come back from L2).  128 threads and 2048-token chunks
// keep eight blocks on an SM, so a batch of up to 8 x SMs sequences is resident at once
// (256 threads with 4096-token chunks, four per SM: 4 % slower on 879 sequences of 4096
// slots).  Loops stay rolled: the code is fetched cold by every block, so its size is
// part of the latency.
constexpr int kRcChunk = 2048;
constexpr int kRcW = kRcThreads / 32;

__global__ void __launch_bounds__(kRcThreads, 8) rc_seq_kernel(RcArgs a) {
    __shared__ __align__(16) float s_lt[kRcChunk];
    __shared__ __align__(16) float s_lr[kRcChunk];
    __shared__ __align__(16) uint8_t s_m[kRcChunk];
    __shared__ FF shff[kRcW][4];
    __shared__ float shf[kRcW][5];
    __shared__ int shi[kRcW][6];
    __shared__ RcSeq sq;
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
    auto stage = [&](int c) {   // chunk c into shared memory; returns its length
        const int64_t c0 = o0 + static_cast<int64_t>(c) * kRcChunk;
        const int n = static_cast<int>(o1 - c0 < kRcChunk ? o1 - c0 : kRcChunk);
        const float* lt = a.lt + c0;
        const float* lr = a.lr + c0;
        const uint8_t* mk = a.mask + c0;
        int i0 = 0;
        if ((((reinterpret_cast<uintptr_t>(lt) | reinterpret_cast<uintptr_t>(lr)) & 15) |
             (reinterpret_cast<uintptr_t>(mk) & 3)) == 0) {
            // 16-byte loads (4-byte for the mask), all of a thread's loads in flight at once
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

    // pass 1: the sequence's sums
    int n = 0, cat = 0;
    FF S = {0.f, 0.f}, E = {0.f, 0.f};   // the decisions' sums, float-float
    float st = 0.f, sr = 0.f;            // metric sums: fp32 per thread
    float mis = 0.f, k3 = 0.f, ad = 0.f, c2 = 0.f;
    int staged = -1;
    for (int c = 0; c < nchunks; ++c) {
        if (c > 0) __syncthreads();   // the previous chunk's readers are done
        const int cn = stage(c);
        staged = c;
#pragma unroll 1
        for (int i = threadIdx.x; i < cn; i += kRcThreads) {
            if (s_m[i] == 0) continue;
            const float x = s_lt[i], y = s_lr[i];
            const FF d = two_sum(x, -y);
            ++n;
            S = ff_add(S, d);
            st += x;
            sr += y;
            if (rs_seq) E = ff_add(E, exp_ff2(d));
            if (q.veto) cat += ff_lt(d, q.lnVeto) ? 1 : 0;
            const float df = d.hi;
            const float ed = expf(df);
            mis -= df;
            k3 += ed - df - 1.f;
            ad += fabsf(df);
            c2 += ed * ed;
        }
    }
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
    double seqd[7] = {0, 0, 0, 0, 0, 0, 0};   // w_before (sequence levels), lppl terms, chi2_seq
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
            seqd[1] = tr;
            seqd[2] = ro;
            seqd[3] = df;
            seqd[4] = fabsf(df);
            seqd[5] = expf(df);
            // e^(2 S): fp32 while it fits, fp64 (one call) past the fp32 range
            seqd[6] = Sb.hi < 44.f ? static_cast<double>(expf(2.f * Sb.hi) * (1.f + 2.f * Sb.lo))
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
            if (s_m[i] != 0) {
                const bool tok = q.level == RL_LEVEL_TOKEN || (q.use_rs && q.rs_level == RL_LEVEL_TOKEN);
                const FF d = tok ? two_sum(s_lt[i], -s_lr[i]) : FF{0.f, 0.f};
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
        const double d[kRcD] = {q.level == RL_LEVEL_TOKEN ? static_cast<double>(F[2]) : seqd[0],
                                F[0], F[1], tok1[0], tok1[1], tok1[2], tok1[3],
                                seqd[1], seqd[2], seqd[3], seqd[4], seqd[5], seqd[6]};
        for (int f = 0; f < kRcD; ++f) a.pd[f * B + b] = d[f];
        const long long c[kRcC] = {nt, nt > 0 ? 1 : 0, I[0], I[1], I[2], I[3], I[4], catt, catt > 0 ? 1 : 0};
        for (int f = 0; f < kRcC; ++f) a.pc[f * B + b] = c[f];
        a.pmin[b] = F[3];
        a.pmax[b] = F[4];
        if (q.use_tis && q.norm) {   // the factor's two totals, in any order of arrival
            if (I[0] != 0) atomicAdd(reinterpret_cast<unsigned long long*>(a.kept_n), static_cast<unsigned long long>(I[0]));
            if (fabsf(F[1]) < a.kept_lim) {
                const long long x = __float2ll_rn(F[1] * 16777216.f);
                if (x != 0) atomicAdd(reinterpret_cast<unsigned long long*>(a.kept_wfix), static_cast<unsigned long long>(x));
            } else {
                atomicExch(a.kept_range, 1);
            }
        }
    }
}

// Warp f sums field f of the records over the sequences in order (lane l takes
// b = l, l + 32, ..., sixteen loads in flight ahead of their adds, then a butterfly) into
// tot[f].  With only_factor, just the two fields the batch-normalisation factor needs.
// Every block that calls it computes the same bits.
constexpr int kRcReduceThreads = 32 * kRcFields;
RL_DEVINL void rc_reduce_fields(const RcArgs& a, double* tot, bool only_factor) {
    const int f = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t B = a.B;
    if (f >= kRcFields) return;
    if (only_factor && f != RD_KEPT_W && f != kRcD + RC_KEPT) return;
    if (f < kRcD) {
        const double* src = a.pd + f * B;
        double v = 0.0;
        for (int64_t b0 = lane; b0 < B; b0 += 32 * 16) {
            double x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = b0 + 32 * i < B ? src[b0 + 32 * i] : 0.0;
#pragma unroll
            for (int i = 0; i < 16; ++i) v += x[i];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) tot[f] = v;
    } else if (f < kRcD + kRcC) {
        const long long* src = a.pc + (f - kRcD) * B;
        long long v = 0;
        for (int64_t b0 = lane; b0 < B; b0 += 32 * 16) {
            long long x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = b0 + 32 * i < B ? src[b0 + 32 * i] : 0;
#pragma unroll
            for (int i = 0; i < 16; ++i) v += x[i];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) tot[f] = static_cast<double>(v);
    } else {
        const bool is_min = f == kRcD + kRcC;
        const float* src = is_min ? a.pmin : a.pmax;
        float v = is_min ? INFINITY : -INFINITY;
        for (int64_t b0 = lane; b0 < B; b0 += 32 * 16) {
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = b0 + 32 * i < B ? src[b0 + 32 * i] : v;
#pragma unroll
            for (int i = 0; i < 16; ++i) v = is_min ? fminf(v, x[i]) : fmaxf(v, x[i]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float u = __shfl_xor_sync(0xffffffffu, v, o);
            v = is_min ? fminf(v, u) : fmaxf(v, u);
        }
        if (lane == 0) tot[f] = v;
    }
}

// The batch-normalisation factor n_kept / sum of kept weights: from the integer totals the
// sequence blocks accumulated (t may then be null), else from the reduced fields t.
RL_DEVINL bool rc_factor_fixed(const RcArgs& a) { return a.q.use_tis && a.q.norm && *a.kept_range == 0; }
RL_DEVINL double rc_factor(const RcArgs& a, const double* t) {
    if (!(a.q.use_tis && a.q.norm)) return 1.0;
    double kept_w, n_kept;
    if (rc_factor_fixed(a)) {
        n_kept = static_cast<double>(*a.kept_n);
        kept_w = static_cast<double>(*a.kept_wfix) * (1.0 / 16777216.0);
    } else {
        kept_w = t[RD_KEPT_W];
        n_kept = t[kRcD + RC_KEPT];
    }
    return (n_kept > 0 && kept_w > 0) ? n_kept / kept_w : 1.0;
}

// The factor and the metrics from the reduced fields (one thread).
RL_DEVINL void rc_write_metrics(const RcArgs& a, const double* t) {
    const double kept_w = t[RD_KEPT_W], n_kept = t[kRcD + RC_KEPT];
    const double factor = rc_factor(a, t);
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


// One block of kRcFields warps: the fields in sequence order, then the factor and the
// metrics (used when no batch normalisation follows).
__global__ void __launch_bounds__(kRcReduceThreads) rc_reduce_kernel(RcArgs a) {
    __shared__ double tot[kRcFields];
    rc_reduce_fields(a, tot, false);
    __syncthreads();
    if (threadIdx.x == 0) rc_write_metrics(a, tot);
}

// Batch normalisation: every block forms the factor (from the integer totals, or, when a
// sequence's sum was out of their range, from the two fields it needs in the order
// rc_reduce_kernel uses, so every block has the same bits), block 0 also reduces all the
// fields and writes the metrics while the other blocks scale: w *= factor, float4 over the
// 16-byte-aligned body (four loads in flight per thread) and scalars at the two ends.  One
// launch where a reduce and a scale kernel would take two.
__global__ void __launch_bounds__(kRcReduceThreads) rc_scale_kernel(RcArgs a) {
    __shared__ double tot[kRcFields];
    __shared__ float fac;
    if (blockIdx.x == 0 || !rc_factor_fixed(a)) rc_reduce_fields(a, tot, blockIdx.x != 0);
    __syncthreads();
    if (threadIdx.x == 0) {
        fac = static_cast<float>(rc_factor(a, tot));
        if (blockIdx.x == 0) rc_write_metrics(a, tot);
    }
    __syncthreads();
    // block 0 (the metrics) takes no share of the scaling when there are other blocks
    if (gridDim.x > 1 && blockIdx.x == 0) return;
    const int64_t sb = gridDim.x > 1 ? blockIdx.x - 1 : 0, nsb = gridDim.x > 1 ? gridDim.x - 1 : 1;
    const float f = fac;
    float* w = a.w;
    const int64_t T = a.T;
    const int64_t head = ((16 - (reinterpret_cast<uintptr_t>(w) & 15)) & 15) / 4;
    const int64_t h = head < T ? head : T;
    const int64_t n4 = (T - h) / 4;
    const int64_t tid = sb * blockDim.x + threadIdx.x;
    const int64_t nth = nsb * blockDim.x;
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
// Workspace: a 256-byte header (status, factor, the factor's range flag and integer
// totals), then the per-sequence records.
constexpr size_t kRcHeader = 256;

static size_t rc_record_bytes(int64_t B) {
    return align_up(static_cast<size_t>(B) * (kRcD * 8 + kRcC * 8 + 2 * 4) + 64, 256);
}

size_t rollout_ws_bytes(int64_t B) { return kRcHeader + rc_record_bytes(B < 1 ? 1 : B); }

int rollout_impl(const float* lt, const float* lr, const uint8_t* mask, const int64_t* off, int64_t B, int64_t T,
                 const rl_rc_params* p, float* w, uint8_t* keep, rl_rc_metrics* metrics, void* ws,
                 size_t ws_bytes, cudaStream_t stream) {
    if (ws_bytes < rollout_ws_bytes(B)) return RL_ERR_WORKSPACE;
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
    a.status = reinterpret_cast<int32_t*>(base + 4);
    a.factor = reinterpret_cast<float*>(base + 8);
    a.kept_range = reinterpret_cast<int*>(base + 12);
    a.kept_n = reinterpret_cast<long long*>(base + 16);
    a.kept_wfix = reinterpret_cast<long long*>(base + 24);
    // a sequence's kept-weight sum below 2^38 / B keeps the total below 2^62 in 2^-24 units
    a.kept_lim = static_cast<float>(ldexp(1.0, 38) / static_cast<double>(B > 0 ? B : 1));
    uint8_t* rec = base + kRcHeader;
    a.pd = reinterpret_cast<double*>(rec);
    a.pc = reinterpret_cast<long long*>(a.pd + kRcD * B);
    a.pmin = reinterpret_cast<float*>(a.pc + kRcC * B);
    a.pmax = a.pmin + B;
    a.metrics = metrics;
    {
        ProfScope pm(RL_PROF_MEMSET, stream);
        if (cudaMemsetAsync(ws, 0, 32, stream) != cudaSuccess) return RL_ERR_CUDA;   // status .. kept_wfix
    }
    ProfScope ps(RL_PROF_ROLLOUT, stream);   // the kernel launches alone
    int launches = 0;
    if (B > 0) {
        rc_seq_kernel<<<static_cast<unsigned>(B), kRcThreads, 0, stream>>>(a);
        ++launches;
    }
    if (q.use_tis && q.norm && w != nullptr && T > 0) {
        // the reduction rides along with the scaling (every block forms the factor)
        const int64_t blocks = (T / 4 + kRcReduceThreads - 1) / kRcReduceThreads + 1;
        const int64_t cap = 2L * num_sms();
        rc_scale_kernel<<<static_cast<unsigned>(blocks < cap ? blocks : cap), kRcReduceThreads, 0, stream>>>(a);
    } else {
        rc_reduce_kernel<<<1, kRcReduceThreads, 0, stream>>>(a);
    }
    ++launches;
    count_launch(launches);
    return cudaPeekAtLastError() == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}

}  // namespace rl
