// Elementwise PPO / dual-clip / decoupled-TIS losses and mismatch statistics on per-token
// log-probabilities ("Rollout Correction Methods": standard, bypass and decoupled
// 3-policy PPO, "Mismatch Metrics"; "10-KL-clip-entropy" section 2: clip, dual clip,
// pg_clipfrac / ppo_kl / pg_clipfrac_lower; "IPO (INTELLECT Policy Optimization)",
// "Choosing eps": masked fraction vs eps against the IcePop ratio band).
//
// One streaming pass: 16-byte vector loads of the four fp32 inputs and 4-byte loads of
// the mask, per-thread fp32 sums / int32 counts, then a fixed-order fp64 block tree and
// a single-block final sum (bitwise reproducible for a given device).  Count predicates
// are decided in fp32 and re-decided in fp64 inside a 1e-5 band around each threshold,
// so they equal the fp64 predicates on the same fp32 inputs.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace rl {

constexpr int kPgThreads = 256;
constexpr int kPgSums = 6;
constexpr int kPgCounts = 6 + RL_PG_MAX_CURVE;
constexpr int kPgFields = kPgSums + kPgCounts;

struct PgArgs {
    const float* lt;
    const float* lo;
    const float* ls;
    const float* adv;
    const uint8_t* mask;
    int64_t T;
    rl_pg_params p;
    float* loss_ppo;
    float* loss_dec;
    float* grad_ppo;
    float* grad_dec;
    double* part;
    int64_t rot_step;   // per-round rotation of the thread -> group map (threads, warp-aligned)
};

struct PgAcc {
    float sum[kPgSums];
    int cnt[kPgCounts];
};

// fp64 restatement used inside the guard bands (same expressions as the definition).
// Not inlined: fp64 is slow on this part, and an inlined copy of a pure function may be
// hoisted or if-converted so that it runs for every token, not just inside the bands.
struct PgExact {
    bool clip, dual, tis_trunc, ice_lo, ice_hi;
};
__device__ __noinline__ double exact_pdiff(float lo, float ls) {
    return exp(static_cast<double>(lo)) - exp(static_cast<double>(ls));
}
__device__ __noinline__ PgExact pg_exact(float lt, float lo, float ls, float A, const rl_pg_params& p) {
    const double r = exp(static_cast<double>(lt) - static_cast<double>(lo));
    const double Ad = A;
    const double l1 = -Ad * r;
    const double lo_b = 1.0 - static_cast<double>(p.clip_ratio_low);
    const double hi_b = 1.0 + static_cast<double>(p.clip_ratio_high);
    const double rc = r < lo_b ? lo_b : (r > hi_b ? hi_b : r);
    const double l2 = -Ad * rc;
    const double lc = l1 > l2 ? l1 : l2;
    const double l3 = -Ad * static_cast<double>(p.clip_ratio_c);
    const double rho = exp(static_cast<double>(lo) - static_cast<double>(ls));
    PgExact e;
    e.clip = l2 > l1;
    e.dual = (Ad < 0.0) && (l3 < lc);
    e.tis_trunc = rho > static_cast<double>(p.tis_upper);
    e.ice_lo = rho < static_cast<double>(p.icepop_low);
    e.ice_hi = rho > static_cast<double>(p.icepop_high);
    return e;
}

RL_DEVINL bool near(float x, float thr) { return fabsf(x - thr) <= 1e-5f * fmaxf(1.f, fabsf(thr)); }

// e^x as 2^(x log2 e) on the hardware EX2 unit: relative error about 2^-22 plus the rounding
// of x log2 e (|x| < 25 here: under 2e-6), well inside the 1e-5 bands around thresholds.
RL_DEVINL float exp_fast(float x) { return exp2_approx(x * kLog2e); }

// The IPO curve's decisions 1(|p_old - p_samp| > eps_k) taken in fp64 for one token, as a
// bit mask (used only when the fp32 difference lies within 1e-5 of some eps_k).
__device__ __noinline__ unsigned curve_bits_exact(float lo, float ls, const rl_pg_params& p) {
    const double dd = fabs(exact_pdiff(lo, ls));
    unsigned bits = 0u;
    for (int k = 0; k < p.n_curve; ++k)
        if (dd > static_cast<double>(p.curve_eps[k])) bits |= 1u << k;
    return bits;
}

// One token.  An invalid (masked-out) token writes zeros and adds nothing; the caller
// skips it before any arithmetic when the whole group of four is invalid.
RL_DEVINL void pg_token(float lt, float lo, float ls, float A, bool valid, const rl_pg_params& p,
                        float& out_lp, float& out_ld, float& out_gp, float& out_gd, PgAcc& acc) {
    if (!valid) {
        out_lp = out_ld = out_gp = out_gd = 0.f;
        return;
    }
    const float r = exp_fast(lt - lo);
    const float l1 = -A * r;
    const float lo_b = 1.f - p.clip_ratio_low, hi_b = 1.f + p.clip_ratio_high;
    const float l2 = -A * fminf(fmaxf(r, lo_b), hi_b);
    const float lc = fmaxf(l1, l2);
    const float l3 = -A * p.clip_ratio_c;
    bool dual = (A < 0.f) && (l3 < lc);
    bool clip = l2 > l1;
    const float d = lo - ls;
    const float rho_raw = exp_fast(d);
    bool tis_trunc = rho_raw > p.tis_upper;
    bool ice_lo = rho_raw < p.icepop_low;
    bool ice_hi = rho_raw > p.icepop_high;
    if (near(r, lo_b) || near(r, hi_b) || (A < 0.f && near(lc, l3)) || near(rho_raw, p.tis_upper) ||
        near(rho_raw, p.icepop_low) || near(rho_raw, p.icepop_high)) {
        const PgExact e = pg_exact(lt, lo, ls, A, p);
        clip = e.clip;
        dual = e.dual;
        tis_trunc = e.tis_trunc;
        ice_lo = e.ice_lo;
        ice_hi = e.ice_hi;
    }
    // branch choices follow the (fp64-exact) decisions above: the clipped branch has no
    // gradient, the dual-clip cap has none either
    const float loss_ppo = dual ? l3 : lc;
    const float g_c = clip ? 0.f : -A * r;
    const float rho = fminf(rho_raw, p.tis_upper);
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
    const float adiff = fabsf(exp_fast(lo) - exp_fast(ls));
    // fp32 decisions, and the distance to the nearest eps in units of its 1e-5 band; only
    // a token inside some band re-takes the decisions in fp64 (full unroll with a guard
    // keeps every counter in a register)
    float close = INFINITY;
#pragma unroll
    for (int k = 0; k < RL_PG_MAX_CURVE; ++k) {
        if (k < p.n_curve) {
            const float eps = p.curve_eps[k];
            acc.cnt[6 + k] += adiff > eps ? 1 : 0;
            close = fminf(close, fabsf(adiff - eps) - 1e-5f * fmaxf(1.f, eps));
        }
    }
    if (close <= 0.f) {
        const unsigned bits = curve_bits_exact(lo, ls, p);
#pragma unroll
        for (int k = 0; k < RL_PG_MAX_CURVE; ++k)
            if (k < p.n_curve)
                acc.cnt[6 + k] += static_cast<int>((bits >> k) & 1u) - (adiff > p.curve_eps[k] ? 1 : 0);
    }
}

__global__ void __launch_bounds__(kPgThreads, 2) policy_kernel(PgArgs a) {
    PgAcc acc;
#pragma unroll
    for (int k = 0; k < kPgSums; ++k) acc.sum[k] = 0.f;
#pragma unroll
    for (int k = 0; k < kPgCounts; ++k) acc.cnt[k] = 0;
    const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const bool vec = (a.T % 4 == 0) &&
                     (((reinterpret_cast<uintptr_t>(a.lt) | reinterpret_cast<uintptr_t>(a.lo) |
                        reinterpret_cast<uintptr_t>(a.ls) | reinterpret_cast<uintptr_t>(a.adv)) &
                       15) == 0) &&
                     ((reinterpret_cast<uintptr_t>(a.mask) & 3) == 0) &&
                     ((reinterpret_cast<uintptr_t>(a.loss_ppo) | reinterpret_cast<uintptr_t>(a.loss_dec) |
                       reinterpret_cast<uintptr_t>(a.grad_ppo) | reinterpret_cast<uintptr_t>(a.grad_dec)) &
                      15) == 0;
    if (vec) {
        // Rounds of nthreads groups of four tokens.  Within round j the thread takes group
        // base + (tid + j S) mod nthreads, a warp-aligned rotation (S from rot_step), so a
        // thread does not meet the same position of a padded sequence layout in every
        // round (a plain grid stride that is a multiple of the padding period gives some
        // threads only valid tokens and others only padding).
        const int64_t n4 = a.T / 4;
        int64_t rot = 0;
        for (int64_t base = 0; base < n4; base += nthreads) {
            int64_t idx = tid + rot;
            if (idx >= nthreads) idx -= nthreads;
            rot += a.rot_step;
            if (rot >= nthreads) rot -= nthreads;
            const int64_t i = base + idx;
            if (i >= n4) continue;
            const float4 lt = __ldcs(reinterpret_cast<const float4*>(a.lt) + i);
            const float4 lo = __ldcs(reinterpret_cast<const float4*>(a.lo) + i);
            const float4 ls = __ldcs(reinterpret_cast<const float4*>(a.ls) + i);
            const float4 A = __ldcs(reinterpret_cast<const float4*>(a.adv) + i);
            const uchar4 m = __ldcs(reinterpret_cast<const uchar4*>(a.mask) + i);
            float4 lp = make_float4(0.f, 0.f, 0.f, 0.f), ld = lp, gp = lp, gd = lp;
            if ((m.x | m.y | m.z | m.w) != 0) {
            pg_token(lt.x, lo.x, ls.x, A.x, m.x != 0, a.p, lp.x, ld.x, gp.x, gd.x, acc);
            pg_token(lt.y, lo.y, ls.y, A.y, m.y != 0, a.p, lp.y, ld.y, gp.y, gd.y, acc);
            pg_token(lt.z, lo.z, ls.z, A.z, m.z != 0, a.p, lp.z, ld.z, gp.z, gd.z, acc);
            pg_token(lt.w, lo.w, ls.w, A.w, m.w != 0, a.p, lp.w, ld.w, gp.w, gd.w, acc);
            }
            if (a.loss_ppo) __stcs(reinterpret_cast<float4*>(a.loss_ppo) + i, lp);
            if (a.loss_dec) __stcs(reinterpret_cast<float4*>(a.loss_dec) + i, ld);
            if (a.grad_ppo) __stcs(reinterpret_cast<float4*>(a.grad_ppo) + i, gp);
            if (a.grad_dec) __stcs(reinterpret_cast<float4*>(a.grad_dec) + i, gd);
        }
    } else {
        for (int64_t i = tid; i < a.T; i += nthreads) {
            float lp, ld, gp, gd;
            pg_token(a.lt[i], a.lo[i], a.ls[i], a.adv[i], a.mask[i] != 0, a.p, lp, ld, gp, gd, acc);
            if (a.loss_ppo) a.loss_ppo[i] = lp;
            if (a.loss_dec) a.loss_dec[i] = ld;
            if (a.grad_ppo) a.grad_ppo[i] = gp;
            if (a.grad_dec) a.grad_dec[i] = gd;
        }
    }
    // fixed-order block reduction: warp trees (fp32 sums, exact int32 counts; fp64 is a
    // slow pipe on this part), then one thread per field adds the 8 warps in fp64
    __shared__ double sh[kPgThreads / 32][kPgFields];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int k = 0; k < kPgSums; ++k) {
        const float v = warp_sum(acc.sum[k]);
        if (lane == 0) sh[warp][k] = static_cast<double>(v);
    }
#pragma unroll
    for (int k = 0; k < kPgCounts; ++k) {
        const int v = __reduce_add_sync(0xffffffffu, acc.cnt[k]);
        if (lane == 0) sh[warp][kPgSums + k] = static_cast<double>(v);
    }
    __syncthreads();
    if (threadIdx.x < kPgFields) {
        double v = 0.0;
        for (int w = 0; w < kPgThreads / 32; ++w) v += sh[w][threadIdx.x];
        a.part[static_cast<int64_t>(blockIdx.x) * kPgFields + threadIdx.x] = v;
    }
}

// One warp per field: lane l sums the block partials b = l, l + 32, ... in order, then a
// fixed shuffle tree (the loads of a lane are independent, so they overlap).
__global__ void policy_final_kernel(const double* part, int nblk, rl_pg_metrics* out) {
    const int k = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (k >= kPgFields) return;
    double s = 0.0;
    for (int b = lane; b < nblk; b += 32) s += part[static_cast<int64_t>(b) * kPgFields + k];
    s = warp_sum(s);
    if (lane != 0) return;
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

static int pg_blocks(int64_t T) {
    const int64_t want = (T / 4 + kPgThreads - 1) / kPgThreads;
    const int64_t cap = static_cast<int64_t>(num_sms()) * 2;   // 2 resident blocks per SM: one wave
    int64_t nb = want < cap ? want : cap;
    return nb < 1 ? 1 : static_cast<int>(nb);
}

size_t policy_ws_need(int64_t T) {
    return static_cast<size_t>(pg_blocks(T)) * kPgFields * sizeof(double);
}

size_t policy_ws_bytes(int64_t T) {
    (void)T;
    // enough block partials for 4 blocks per SM on any device up to 256 SMs
    return align_up(static_cast<size_t>(256 * 4) * kPgFields * sizeof(double), 256);
}

int policy_impl(const float* lt, const float* lo, const float* ls, const float* adv,
                const uint8_t* mask, int64_t T, const rl_pg_params* p, float* loss_ppo,
                float* loss_dec, float* grad_ppo, float* grad_dec, rl_pg_metrics* metrics,
                void* ws, cudaStream_t stream) {
    const int nb = pg_blocks(T);
    // rotation in whole warps: about 0.618 of the warps, with an odd residue near 0.6 x 32
    // modulo 32 warps, so successive rounds spread over the phases of any power-of-two
    // padding period instead of creeping by one warp
    const int64_t nwarps = static_cast<int64_t>(nb) * (kPgThreads / 32);
    int64_t kw = (nwarps * 618 / 1000) / 32 * 32 + 19;
    while (kw >= nwarps && kw > 0) kw -= 32;
    if (kw < 0) kw = 0;
    PgArgs a{lt, lo, ls, adv, mask, T, *p, loss_ppo, loss_dec, grad_ppo, grad_dec,
             static_cast<double*>(ws), kw * 32};
    if (static_cast<size_t>(nb) * kPgFields * sizeof(double) > policy_ws_bytes(T)) return RL_ERR_UNSUPPORTED;
    ProfScope ps(RL_PROF_POLICY, stream);
    policy_kernel<<<nb, kPgThreads, 0, stream>>>(a);
    count_launch();
    if (metrics) {
        policy_final_kernel<<<1, 32 * kPgFields, 0, stream>>>(a.part, nb, metrics);
        count_launch();
    }
    return cudaPeekAtLastError() == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}

}  // namespace rl
