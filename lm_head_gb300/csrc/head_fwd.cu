// Forward of the fused LM head + unified RL loss (prime-rl pull request #4233: the loss_t
// equation, the two estimator rules for u, "What changes").
//
//   1. validate_kernel     CSR sampler evidence -> status bits (GPU validation item)
//   2. gemm_tc<EpiStats>   z = X W^T / T by 128 x 256 tensor-core tiles; per row an online
//                          (max, sum e^{z-m}, sum e^{z-m}(z-m)) over the unit's vocab range,
//                          and the label / support logits gathered out of the tile
//   3. token_loss_kernel   one warp per token: combine the split statistics into
//                          logsumexp and entropy, renormalise over a replayed support,
//                          weights w and masks, centering, KL, loss_t, backward
//                          coefficients and per-token metric terms
//   4. metrics kernels     deterministic fp64 reduction of the metric terms
#include <cmath>
#include <climits>
#include <cstring>

#include <cuda_bf16.h>

#include "gemm_tc2.cuh"
#include "internal.h"

namespace rl {

// ----------------------------------------------------------------------------------
// Workspace / saved-state layouts
// ----------------------------------------------------------------------------------
SavedView saved_view(void* base, int64_t N, int64_t nnz, size_t* bytes) {
    Carve c(base);
    SavedView v;
    v.lse = c.take<float>(N);
    v.lse_s = c.take<float>(N);
    v.dcoef = c.take<float>(N);
    v.labcoef = c.take<float>(N);
    v.entcoef = c.take<float>(nnz > 0 ? nnz : 1);
    v.mterm = c.take<float>(N * 8);
    v.zlab = c.take<float>(N);
    v.zsup = c.take<float>(nnz > 0 ? nnz : 1);
    if (bytes) *bytes = align_up(c.off, 256);
    return v;
}

static int max_splits(int64_t V) {
    const int nb = static_cast<int>((V + kBN - 1) / kBN);
    return nb < 32 ? nb : 32;
}

FwdWs fwd_ws_view(void* base, int64_t N, int64_t H, int64_t V, int64_t nnz, size_t* bytes) {
    (void)H;
    Carve c(base);
    FwdWs w;
    w.splits = max_splits(V);   // each split holds one partial per column half
    w.part_m = c.take<float>(static_cast<size_t>(2 * w.splits) * N);
    w.part_s = c.take<float>(static_cast<size_t>(2 * w.splits) * N);
    w.part_u = c.take<float>(static_cast<size_t>(2 * w.splits) * N);
    w.mpart = c.take<double>(kMetricBlocks * kMetricFields);
    if (bytes) *bytes = align_up(c.off, 256);
    return w;
}

// Split count for the forward GEMM: units = m_blocks * splits spread over the SMs; pick
// the count that fills the last wave best (ties -> fewer splits).
static int choose_splits(int64_t N, int64_t V) {
    const int pair = gemm_pair_mode();
    const int m_blocks = static_cast<int>((N + (pair ? 2 * kBM : kBM) - 1) / (pair ? 2 * kBM : kBM));
    const int P = pair ? num_sms() / 2 : num_sms();
    const int smax = max_splits(V);
    int best = 1;
    double best_eff = 0.0;
    for (int s = 1; s <= smax; ++s) {
        const int64_t units = static_cast<int64_t>(m_blocks) * s;
        const int64_t waves = (units + P - 1) / P;
        const double eff = static_cast<double>(units) / static_cast<double>(waves * P);
        if (eff > best_eff + 0.01) {
            best_eff = eff;
            best = s;
        }
    }
    return best;
}

// ----------------------------------------------------------------------------------
// 1. Validation of the CSR sampler evidence
// ----------------------------------------------------------------------------------
struct ValidateArgs {
    int64_t N, V, nnz;
    const int64_t* offsets;
    const int32_t* ids;
    const float* logq;
    const uint8_t* replayed;
    const int32_t* labels;
    const float* label_logq;
    const uint8_t* loss_mask;
    int32_t* status;
};

__global__ void __launch_bounds__(256) validate_kernel(ValidateArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (t >= a.N) return;
    int32_t bad = 0;
    const int64_t b = a.offsets[t], e = a.offsets[t + 1];
    if (lane == 0) {
        if (t == 0 && b != 0) bad |= RL_STATUS_OFFSETS;
        if (t == a.N - 1 && e != a.nnz) bad |= RL_STATUS_OFFSETS;
    }
    if (b < 0 || e < b || e > a.nnz) {
        if (lane == 0) set_status(a.status, bad | RL_STATUS_OFFSETS);
        return;
    }
    const int32_t label = a.labels[t];
    const bool rl = a.loss_mask ? a.loss_mask[t] != 0 : true;
    const bool rep = a.replayed[t] != 0;
    if (lane == 0) {
        if (label < 0 || label >= a.V) bad |= RL_STATUS_ID_RANGE;
        const float llq = a.label_logq[t];
        if (!isfinite(llq) || llq > 1e-6f) bad |= RL_STATUS_LOGQ;
        if (rl && e == b) bad |= RL_STATUS_EMPTY_ROW;
    }
    float mass = 0.f;
    int found = 0;
    for (int64_t j = b + lane; j < e; j += 32) {
        const int32_t id = a.ids[j];
        const float lq = a.logq[j];
        if (id < 0 || id >= a.V) bad |= RL_STATUS_ID_RANGE;
        if (!isfinite(lq) || lq > 1e-6f) bad |= RL_STATUS_LOGQ;
        if (j > b) {
            const int32_t prev = a.ids[j - 1];
            if (rep ? (id <= prev) : (id < prev)) bad |= RL_STATUS_ROW_ORDER;
        }
        if (rep) mass += expf(lq);
        found |= (id == label);
    }
    mass = warp_sum(mass);
    found = __any_sync(0xffffffffu, found);
    bad = __reduce_or_sync(0xffffffffu, bad);
    if (lane == 0) {
        if (rep && rl) {
            if (!found) bad |= RL_STATUS_LABEL_MISSING;
            if (!(fabsf(mass - 1.f) <= 1e-3f)) bad |= RL_STATUS_SUPPORT_MASS;   // a NaN mass too
        }
        set_status(a.status, bad);
    }
}

int validate_impl(const rl_head_batch* b, int32_t* status, cudaStream_t stream) {
    if (b->N == 0) return RL_OK;
    ValidateArgs a{b->N, b->V, b->support.nnz, b->support.offsets, b->support.ids,
                   b->support.logq, b->support.replayed, b->labels, b->label_logq,
                   b->loss_mask, status};
    const int64_t blocks = (b->N + 7) / 8;
    ProfScope ps(RL_PROF_VALIDATE, stream);
    validate_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a);
    count_launch();
    return cudaPeekAtLastError() == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}

// ----------------------------------------------------------------------------------
// 2. GEMM epilogue: online logsumexp / entropy statistics + label & support gather
// ----------------------------------------------------------------------------------
RL_DEVINL float select32(const float (&v)[32], int idx) {
    float r = v[0];
#pragma unroll
    for (int k = 1; k < 32; ++k) r = (idx == k) ? v[k] : r;
    return r;
}
RL_DEVINL void kahan_add(float& s, float& c, float x) {
    const float y = x - c;
    const float t = s + y;
    c = (t - s) - y;
    s = t;
}

RL_DEVINL float max32(const float (&v)[32]) {
    float m[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) m[k] = fmaxf(v[k], v[k + 16]);
#pragma unroll
    for (int w = 8; w > 0; w >>= 1)
#pragma unroll
        for (int k = 0; k < w; ++k) m[k] = fmaxf(m[k], m[k + w]);
    return m[0];
}

// Per row and column half, an online (max, sum e^{z-m}, sum e^{z-m}(z-m)) over the unit's
// vocabulary tiles, kept in log2 units (m2 = m log2(e)): each logit costs one FFMA, one
// EX2, one FADD and one FFMA.  The partial is written in natural units.  Label and support
// logits are taken from the chunk that holds them: the row's CSR ids are ascending, so a
// pointer moves forward with the columns.
struct EpiStats {
    struct Params {
        int64_t N;
        int32_t V;
        float inv_T;
        float c2;          // log2(e) / T
        int64_t nnz;
        const int32_t* labels;
        const int64_t* offsets;
        const int32_t* ids;
        float* zlab;
        float* zsup;
        float* part_m;
        float* part_s;
        float* part_u;
        // fused forward + backward, bf16 gradient precision (Eb != nullptr): e relative to
        // the row reference cref, stored as bf16 in both layouts through TMA
        uint16_t* Eb;
        const float* cref;
        int* flag;
        CUtensorMap tmEb;    // over Eb [N, V]: box 32 rows x 32 columns, 64-byte swizzle
        CUtensorMap tmEbt;   // over Ebt [V, ldt]: box 32 vocabulary rows x 32 tokens, no swizzle
        // fused forward + backward, hi/lo gradient precision (E32 != nullptr): fp32 e relative
        // to the running max m2, which is stored per 32-column chunk [N, ldm]
        float* E32;
        float* M2;
        int64_t ldm;
        CUtensorMap tmE32;   // over E32 [N, V]: box 32 x 32, 128-byte swizzle
    };
    int64_t t;
    bool valid;
    float m2, s, sc, u2, uc;
    float cr;
    int64_t ptr, end;
    int32_t next_id;
    int32_t label;

    RL_DEVINL void begin_unit(const Params& p, int row, int half, int m_blk, int split, int col_begin) {
        (void)split;
        (void)half;
        t = static_cast<int64_t>(m_blk) * kBM + row;
        valid = t < p.N;
        m2 = -INFINITY;
        s = sc = u2 = uc = 0.f;
        cr = 0.f;
        ptr = end = 0;
        next_id = INT_MAX;
        label = -1;
        if (!valid) return;
        if (p.cref != nullptr) cr = p.cref[t];
        label = p.labels[t];
        int64_t b = p.offsets[t], e = p.offsets[t + 1];
        b = b < 0 ? 0 : (b > p.nnz ? p.nnz : b);
        e = e < b ? b : (e > p.nnz ? p.nnz : e);
        int64_t lo = b, hi = e;  // first entry with id >= col_begin
        while (lo < hi) {
            const int64_t mid = (lo + hi) >> 1;
            if (p.ids[mid] < col_begin)
                lo = mid + 1;
            else
                hi = mid;
        }
        ptr = lo;
        end = e;
        next_id = ptr < end ? p.ids[ptr] : INT_MAX;
    }

    RL_DEVINL void chunk(const Params& p, const uint32_t (&acc)[32], int col0, uint8_t* stage, int lane) {
        if (col0 >= p.V) return;   // uniform over the warp
        float ev[32];
        if (valid) {
            stats(p, acc, col0, ev);
        } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) ev[k] = 0.f;
        }
        if (p.Eb != nullptr)
            store_eb(p, ev, col0, stage, lane);
        else if (p.E32 != nullptr)
            store_e32(p, ev, col0, stage, lane);
    }

    // bf16 e relative to the row reference: 2^(z' - cref) = 2^(z' - m2) 2^(m2 - cref), one
    // EX2 per row and chunk.  The warp's 32 x 32 block goes through shared memory twice per
    // chunk: row-major (2 KB, 64-byte swizzle: 16-byte piece c of row r at c ^ ((r >> 1) & 3),
    // so the 32 lanes' 16-byte writes hit distinct banks) and transposed (2 KB, vocabulary
    // row k holds the 32 lanes' values at 2-byte steps), then two TMA stores.  Rows past N
    // and columns past V are clipped by the tensor maps.
    RL_DEVINL void store_eb(const Params& p, const float (&ev)[32], int col0, uint8_t* stage, int lane) {
        float kf = 0.f;
        if (valid) {
            const float dm = m2 - cr;
            if (dm > kRefRangeLog2) *p.flag = 1;   // beyond the bf16 store's range: recompute
            kf = exp2_approx(fminf(dm, 126.f));
        }
        uint32_t h[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const __nv_bfloat162 v = __floats2bfloat162_rn(ev[2 * k] * kf, ev[2 * k + 1] * kf);
            h[k] = *reinterpret_cast<const uint32_t*>(&v);
        }
        if (lane == 0) bulk_wait_read<0>();   // the previous chunk's stores have read the tiles
        __syncwarp();
        uint8_t* row = stage + lane * 64;
        const int sw = (lane >> 1) & 3;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(row + ((q ^ sw) << 4)) = make_uint4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
        uint16_t* col = reinterpret_cast<uint16_t*>(stage + 2048) + lane;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            col[(2 * k) * 32] = static_cast<uint16_t>(h[k] & 0xFFFFu);
            col[(2 * k + 1) * 32] = static_cast<uint16_t>(h[k] >> 16);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && t < p.N) {   // lane 0 holds the warp's first row
            // evict-first: e is read only by the backward GEMMs, after this kernel; keeping
            // it out of the way leaves L2 to the X and W tiles this kernel reuses
            tma_store_2d_evict_first(&p.tmEb, stage, col0, static_cast<int32_t>(t));
            tma_store_2d_evict_first(&p.tmEbt, stage + 2048, static_cast<int32_t>(t), col0);
            bulk_commit();
        }
    }

    // fp32 e relative to m2 (the running max at this chunk), one 32 x 32 tile per chunk
    // (4 KB, 128-byte swizzle: 16-byte piece c of row r at c ^ (r % 8)), and m2 itself.
    RL_DEVINL void store_e32(const Params& p, const float (&ev)[32], int col0, uint8_t* stage, int lane) {
        if (lane == 0) bulk_wait_read<0>();   // the previous store has read the tile
        __syncwarp();
        uint8_t* row = stage + lane * 128;
        const int sw = lane & 7;
#pragma unroll
        for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(row + ((q ^ sw) << 4)) =
                make_float4(ev[4 * q], ev[4 * q + 1], ev[4 * q + 2], ev[4 * q + 3]);
        if (valid) p.M2[t * p.ldm + (col0 >> 5)] = m2;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && t < p.N) {
            tma_store_2d(&p.tmE32, stage, col0, static_cast<int32_t>(t));
            bulk_commit();
        }
    }

    RL_DEVINL void stats(const Params& p, const uint32_t (&acc)[32], int col0, float (&ev)[32]) {
        float a[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) a[k] = __uint_as_float(acc[k]);
        const bool full = col0 + 32 <= p.V;
        if (!full) {
#pragma unroll
            for (int k = 0; k < 32; ++k)
                if (col0 + k >= p.V) a[k] = -INFINITY;
        }
        const float cm2 = max32(a) * p.c2;   // T > 0: the max of the raw accumulators is the max of z
        if (cm2 > m2) {
            if (m2 == -INFINITY) {
                s = sc = u2 = uc = 0.f;
            } else {
                const float f = exp2_approx(m2 - cm2);
                u2 = f * (u2 + (m2 - cm2) * s);
                uc *= f;
                s *= f;
                sc *= f;
            }
            m2 = cm2;
        }
        float cs0 = 0.f, cs1 = 0.f, cu0 = 0.f, cu1 = 0.f;
        if (full) {
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
                const float d0 = fmaf(a[k], p.c2, -m2);
                const float d1 = fmaf(a[k + 1], p.c2, -m2);
                ev[k] = exp2_approx(d0);
                ev[k + 1] = exp2_approx(d1);
                cs0 += ev[k];
                cs1 += ev[k + 1];
                cu0 = fmaf(ev[k], d0, cu0);
                cu1 = fmaf(ev[k + 1], d1, cu1);
            }
        } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const float d = fmaxf(fmaf(a[k], p.c2, -m2), -1e30f);
                ev[k] = exp2_approx(d);
                cs0 += ev[k];
                cu0 = fmaf(ev[k], d, cu0);
            }
        }
        kahan_add(s, sc, cs0 + cs1);
        kahan_add(u2, uc, cu0 + cu1);
        // z exactly as the backward's recompute forms it: one rounded multiply by 1/T
        if (static_cast<unsigned>(label - col0) < 32u)
            p.zlab[t] = __fmul_rn(select32(a, label - col0), p.inv_T);
        while (next_id < col0 + 32) {  // ids below col0 belong to the other column half
            if (next_id >= col0) p.zsup[ptr] = __fmul_rn(select32(a, next_id - col0), p.inv_T);
            ++ptr;
            next_id = ptr < end ? p.ids[ptr] : INT_MAX;
        }
    }

    RL_DEVINL void end_unit(const Params& p, int split, int half) {
        if (!valid) return;
        const int64_t i = static_cast<int64_t>(2 * split + half) * p.N + t;
        p.part_m[i] = m2 * kLn2;
        p.part_s[i] = s - sc;
        p.part_u[i] = (u2 - uc) * kLn2;
    }
};

// ----------------------------------------------------------------------------------
// 3. Per-token loss assembly (one warp per token)
// ----------------------------------------------------------------------------------
struct TokenArgs {
    int64_t N;
    int32_t V;
    int32_t S;
    int64_t nnz;
    int64_t pstride;   // distance between the partials of consecutive splits (N, or 3 N for shard triplets)
    const float* part_m;
    const float* part_s;
    const float* part_u;
    const float* zlab;
    const float* zsup;
    const int32_t* labels;
    const float* label_logq;
    const float* adv;
    const uint8_t* loss_mask;
    const int32_t* age;
    const int64_t* offsets;
    const int32_t* ids;
    const float* logq;
    const uint8_t* replayed;
    int32_t loss_type, kl_est, kl_stale, sparse;
    float eps, cap, lo, hi, adv_tau, kl_coeff, ent_coeff;
    float* loss;
    float* logp_label;
    float* logp_support;
    float* entropy;
    float* lse_out;
    uint8_t* mask_label;
    uint8_t* mask_support;
    SavedView sv;
    int32_t* status;
    // fused forward + backward with bf16 e (rs != nullptr): the row scale of the stored e
    const float* cref;
    const float* dloss;
    float inv_T;
    float* rs;
    int* flag;
};

struct WeightOut {
    float w;
    float r;
    bool keep, low, high;
};

// w of pull request #4233 ("What changes": ipo / icepop / reinforce) with the probability
// band of "Masking by Probability, Not Ratio".  Decisions are taken in fp32 and re-taken
// in fp64 (from the same fp32 log-probs) when the fp32 value lies within 1e-5 of a
// threshold, so the keep bit equals the fp64 predicate evaluated on these log-probs.
RL_DEVINL WeightOut rl_weight(float logP, float logq, const TokenArgs& a) {
    WeightOut o;
    o.r = expf(logP - logq);
    if (a.loss_type == RL_LOSS_IPO) {
        float diff = expf(logP) - expf(logq);
        bool keep;
        if (fabsf(fabsf(diff) - a.eps) <= 1e-5f) {
            const double dd = exp(static_cast<double>(logP)) - exp(static_cast<double>(logq));
            keep = fabs(dd) <= static_cast<double>(a.eps);
            diff = dd < 0 ? -1.f : (dd > 0 ? 1.f : 0.f);
        } else {
            keep = fabsf(diff) <= a.eps;
        }
        o.keep = keep;
        o.w = keep ? fminf(o.r, a.cap) : 0.f;
        o.low = !keep && diff < 0.f;
        o.high = !keep && diff > 0.f;
    } else if (a.loss_type == RL_LOSS_ICEPOP) {
        bool ge_lo, le_hi;
        if (fabsf(o.r - a.lo) <= 1e-5f * a.lo || fabsf(o.r - a.hi) <= 1e-5f * a.hi) {
            const double rd = exp(static_cast<double>(logP) - static_cast<double>(logq));
            ge_lo = rd >= static_cast<double>(a.lo);
            le_hi = rd <= static_cast<double>(a.hi);
        } else {
            ge_lo = o.r >= a.lo;
            le_hi = o.r <= a.hi;
        }
        o.keep = ge_lo && le_hi;
        o.w = o.keep ? o.r : 0.f;
        o.low = !ge_lo;
        o.high = !le_hi;
    } else {
        o.keep = true;
        o.w = 1.f;
        o.low = o.high = false;
    }
    return o;
}

__global__ void __launch_bounds__(256) token_loss_kernel(TokenArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (t >= a.N) return;
    // combine the per-split (m, s, u) statistics: logsumexp and entropy of the full row
    float M = -INFINITY;
    for (int i = lane; i < a.S; i += 32) M = fmaxf(M, a.part_m[static_cast<int64_t>(i) * a.pstride + t]);
    M = warp_max(M);
    float s = 0.f, u = 0.f;
    for (int i = lane; i < a.S; i += 32) {
        const int64_t k = static_cast<int64_t>(i) * a.pstride + t;
        const float mi = a.part_m[k], si = a.part_s[k], ui = a.part_u[k];
        const float f = expf(mi - M);
        s += f * si;
        u += f * (ui + (mi - M) * si);
    }
    s = warp_sum(s);
    u = warp_sum(u);
    const float logs = logf(s);
    const float lse = M + logs;
    const float ent = logs - u / s;

    int64_t b = a.offsets[t], e = a.offsets[t + 1];
    b = b < 0 ? 0 : (b > a.nnz ? a.nnz : b);
    e = e < b ? b : (e > a.nnz ? a.nnz : e);
    const int K = static_cast<int>(e - b);
    const bool rep = a.replayed[t] != 0;
    const bool rl = a.loss_mask ? a.loss_mask[t] != 0 : true;
    const int32_t label = a.labels[t];
    const bool label_ok = label >= 0 && label < a.V;

    // READING: a replayed token's P is the trainer softmax renormalised over S
    float lse_s = lse;
    if (rep) {
        float mx = -INFINITY;
        for (int64_t j = b + lane; j < e; j += 32) {
            const int32_t id = a.ids[j];
            if (id >= 0 && id < a.V) mx = fmaxf(mx, a.zsup[j]);
        }
        mx = warp_max(mx);
        float ss = 0.f;
        for (int64_t j = b + lane; j < e; j += 32) {
            const int32_t id = a.ids[j];
            if (id >= 0 && id < a.V) ss += expf(a.zsup[j] - mx);
        }
        ss = warp_sum(ss);
        if (ss > 0.f) lse_s = mx + logf(ss);
    }

    // pass 1 over the support: log P, u, w, sums
    const float inv_K = K > 0 ? 1.f / static_cast<float>(K) : 0.f;
    float C = 0.f, U = 0.f, cen = 0.f, klx = 0.f, smass = 0.f, mtv = 0.f;
    for (int64_t j = b + lane; j < e; j += 32) {
        const int32_t id = a.ids[j];
        const float lq = a.logq[j];
        const bool ok = id >= 0 && id < a.V && isfinite(lq);
        const float zj = ok ? a.zsup[j] : 0.f;
        const float logP = zj - lse_s;
        float uj = rep ? expf(lq) : inv_K;
        WeightOut wo = rl_weight(logP, lq, a);
        if (!ok) {
            uj = 0.f;
            wo.w = 0.f;
            wo.keep = false;
            wo.r = 0.f;
        }
        const float c = uj * wo.w;
        C += c;
        U += uj;
        cen = fmaf(c, logP, cen);
        klx = fmaf(uj, lq - logP, klx);
        if (ok) smass = fmaf(uj, expf((zj - lse) - lq), smass);
        if (!wo.keep) mtv = fmaf(uj, wo.r, mtv);
        if (a.logp_support) a.logp_support[j] = ok ? logP : 0.f;
        if (a.mask_support) a.mask_support[j] = wo.keep ? 1 : 0;
        a.sv.entcoef[j] = c;  // pass 2 turns this into the spike coefficient
    }
    C = warp_sum(C);
    U = warp_sum(U);
    cen = warp_sum(cen);
    klx = warp_sum(klx);
    smass = warp_sum(smass);
    mtv = warp_sum(mtv);

    const float llq = a.label_logq[t];
    const float logP_lab = label_ok ? a.zlab[t] - lse_s : 0.f;
    WeightOut wl = rl_weight(logP_lab, llq, a);
    const int age = a.age ? a.age[t] : 0;
    const float beta = a.kl_stale == RL_STALE_INV_SQRT
                           ? a.kl_coeff / sqrtf(1.f + static_cast<float>(age))
                           : a.kl_coeff;
    const bool exact = a.kl_est == RL_KL_EXACT;
    const float kl = exact ? klx : (llq - logP_lab);
    const float A = a.adv[t];
    const float at = a.adv_tau * A;
    float loss = -at * (wl.w * logP_lab - cen) + beta * kl;
    // exploration regulariser ("10-KL-clip-entropy", section 3): loss -= c H, full-vocab H
    if (a.ent_coeff != 0.f) loss = fmaf(-a.ent_coeff, ent, loss);
    // d loss / d z_j = d * P_j + spikes; d multiplies the (full or renormalised) softmax
    const float d = at * (wl.w - C) + beta * (exact ? U : 1.f);
    float labc = -at * wl.w - (exact ? 0.f : beta);
    float dco = rep ? 0.f : d;
    const bool eligible = rep || (a.loss_type == RL_LOSS_REINFORCE && beta == 0.f);
    if (a.sparse) {
        if (eligible)
            dco = 0.f;
        else if (rl && lane == 0)
            set_status(a.status, RL_STATUS_SPARSE_INELIGIBLE);
    }
    if (!rl) {
        loss = 0.f;
        dco = 0.f;
        labc = 0.f;
    }

    // pass 2: spike coefficient per entry (same lane touches the same j as in pass 1)
    for (int64_t j = b + lane; j < e; j += 32) {
        float ec = 0.f;
        if (rl) {
            const int32_t id = a.ids[j];
            const float lq = a.logq[j];
            const bool ok = id >= 0 && id < a.V && isfinite(lq);
            if (ok) {
                const float c = a.sv.entcoef[j];
                const float uj = rep ? expf(lq) : inv_K;
                ec = at * c - (exact ? beta * uj : 0.f);
                if (rep) ec = fmaf(d, expf(a.zsup[j] - lse_s), ec);
            }
        }
        a.sv.entcoef[j] = ec;
    }

    if (lane == 0) {
        a.loss[t] = loss;
        if (a.logp_label) a.logp_label[t] = logP_lab;
        if (a.entropy) a.entropy[t] = ent;
        if (a.lse_out) a.lse_out[t] = lse;
        if (a.mask_label) a.mask_label[t] = wl.keep ? 1 : 0;
        a.sv.lse[t] = lse;
        a.sv.lse_s[t] = lse_s;
        a.sv.dcoef[t] = dco;
        a.sv.labcoef[t] = labc;
        float* mt = a.sv.mterm + t * 8;
        int flags = 0;
        if (rl) {
            flags = 1 | (wl.keep ? 0 : 2) | (wl.low ? 4 : 0) | (wl.high ? 8 : 0) | (age == 0 ? 16 : 0);
        }
        mt[0] = loss;
        mt[1] = llq - logP_lab;
        mt[2] = smass;
        mt[3] = mtv;
        mt[4] = kl;
        mt[5] = beta;
        mt[6] = ent;
        mt[7] = __int_as_float(flags);
        if (!isfinite(lse) || !isfinite(loss)) set_status(a.status, RL_STATUS_NONFINITE);
        if (a.rs != nullptr) {
            // G = alpha exp(z - lse) = rs e with e = 2^(z log2(e) - cref); alpha is formed as
            // the backward forms it (dloss dcoef / T, rounded in that order)
            const float alpha = __fmul_rn(__fmul_rn(a.dloss[t], dco), a.inv_T);
            float r = 0.f;
            if (alpha != 0.f) {
                const float gap = __fsub_rn(a.cref[t], __fmul_rn(lse, kLog2e));
                r = __fmul_rn(alpha, exp2_approx(gap));
                if (!(gap >= -kRefRangeLog2 && gap <= kRefRangeLog2) || !isfinite(r)) *a.flag = 1;
            }
            a.rs[t] = r;
        }
    }
}

// ----------------------------------------------------------------------------------
// 4. Deterministic metric reduction
// ----------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) metrics_partial_kernel(const float* mterm, int64_t N,
                                                              double* part) {
    __shared__ double sh[256];
    const int64_t per = (N + gridDim.x - 1) / gridDim.x;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * per;
    const int64_t t1 = t0 + per < N ? t0 + per : N;
    double acc[kMetricFields];
#pragma unroll
    for (int k = 0; k < kMetricFields; ++k) acc[k] = 0.0;
    for (int64_t t = t0 + threadIdx.x; t < t1; t += blockDim.x) {
        const float* mt = mterm + t * 8;
        const int flags = __float_as_int(mt[7]);
        if (!(flags & 1)) continue;
        acc[0] += mt[0];
        acc[1] += mt[1];
        acc[2] += mt[2];
        acc[3] += mt[3];
        acc[4] += mt[4];
        acc[5] += mt[5];
        if (flags & 16) acc[6] += mt[4];
        acc[7] += mt[6];
        acc[8] += 1.0;
        acc[9] += (flags & 2) ? 1.0 : 0.0;
        acc[10] += (flags & 4) ? 1.0 : 0.0;
        acc[11] += (flags & 8) ? 1.0 : 0.0;
        acc[12] += (flags & 16) ? 1.0 : 0.0;
    }
    for (int k = 0; k < kMetricFields; ++k) {
        sh[threadIdx.x] = acc[k];
        __syncthreads();
        for (int w = blockDim.x / 2; w > 0; w >>= 1) {
            if (threadIdx.x < w) sh[threadIdx.x] += sh[threadIdx.x + w];
            __syncthreads();
        }
        if (threadIdx.x == 0) part[blockIdx.x * kMetricFields + k] = sh[0];
        __syncthreads();
    }
}

// One warp per field: lane l sums the block partials b = l, l + 32, ... in order, then a
// fixed shuffle tree.
__global__ void metrics_final_kernel(const double* part, int nblk, const int* flags, int nflags,
                                     rl_head_metrics* out) {
    const int k = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (k >= kMetricFields) return;
    double s = 0.0;
    for (int b = lane; b < nblk; b += 32) s += part[b * kMetricFields + k];
    s = warp_sum(s);
    if (lane != 0) return;
    switch (k) {
        case 0: out->loss = s; break;
        case 1: out->mismatch_kl = s; break;
        case 2: out->support_mass = s; break;
        case 3: out->mask_tv = s; break;
        case 4: out->kl = s; break;
        case 5: out->beta = s; break;
        case 6: out->kl_age0 = s; break;
        case 7: out->entropy = s; break;
        case 8: out->n_rl = static_cast<int64_t>(s); break;
        case 9: out->masked = static_cast<int64_t>(s); break;
        case 10: out->masked_low = static_cast<int64_t>(s); break;
        case 11: out->masked_high = static_cast<int64_t>(s); break;
        case 12: out->n_age0 = static_cast<int64_t>(s); break;
        case 13: {
            int64_t r = 0;
            for (int c = 0; c < nflags; ++c) r += flags[c] != 0 ? 1 : 0;
            out->recomputed_chunks = r;
            break;
        }
        default: break;
    }
}

int metrics_impl(const rl_head_batch* b, const void* saved, rl_head_metrics* metrics, void* ws,
                 cudaStream_t stream) {
    const FwdWs w = fwd_ws_view(ws, b->N, b->H, b->V, b->support.nnz, nullptr);
    return metrics_run(b, saved, metrics, w.mpart, stream);
}

int metrics_run(const rl_head_batch* b, const void* saved, rl_head_metrics* metrics, double* mpart,
                cudaStream_t stream, const int* flags, int nflags) {
    const SavedView sv = saved_view(const_cast<void*>(saved), b->N, b->support.nnz, nullptr);
    ProfScope ps(RL_PROF_METRICS, stream);
    metrics_partial_kernel<<<kMetricBlocks, 256, 0, stream>>>(sv.mterm, b->N, mpart);
    metrics_final_kernel<<<1, 32 * kMetricFields, 0, stream>>>(mpart, kMetricBlocks, flags, nflags, metrics);
    count_launch(2);
    return cudaPeekAtLastError() == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}

// ----------------------------------------------------------------------------------
// Entry
// ----------------------------------------------------------------------------------
// GEMM + per-token loss for token rows [c0, c0 + n): per-token pointers are offset by c0,
// CSR entry arrays stay absolute.  With `es` (fused forward + backward) the GEMM also
// stores e for the backward, in the layout EStore describes.
int fwd_rows(const rl_head_batch* b, const rl_params* prm, const rl_head_outputs* out, const SavedView& sv,
             const FwdWs& w, int64_t c0, int64_t n, const EStore* es, int sparse, int32_t* status,
             cudaStream_t stream) {
    const int64_t H = b->H, V = b->V, nnz = b->support.nnz;
    if (n <= 0) return RL_OK;
    const int S = choose_splits(n, V);
    CUtensorMap tmX, tmW;
    const uint16_t* Xc = static_cast<const uint16_t*>(b->hidden) + c0 * H;
    int rc = make_tmap_bf16(&tmX, Xc, n, H, H, kBM);
    if (rc != RL_OK) return rc;
    rc = make_tmap_b(&tmW, b->weight, V, H, H);
    if (rc != RL_OK) return rc;
    const GemmPlan plan = make_plan_auto(n, V, H, 1, S, 1, status);
    EpiStats::Params ep;
    std::memset(&ep, 0, sizeof(ep));
    ep.N = n;
    ep.V = static_cast<int32_t>(V);
    ep.inv_T = 1.0f / prm->temperature;
    ep.c2 = kLog2e / prm->temperature;
    ep.nnz = nnz;
    ep.labels = b->labels + c0;
    ep.offsets = b->support.offsets + c0;
    ep.ids = b->support.ids;
    ep.zlab = sv.zlab + c0;
    ep.zsup = sv.zsup;
    ep.part_m = w.part_m;
    ep.part_s = w.part_s;
    ep.part_u = w.part_u;
    ep.ldm = (V + 31) / 32;
    if (es != nullptr && es->Eb != nullptr) {
        ep.Eb = es->Eb;
        ep.cref = es->cref;
        ep.flag = es->flag;
        if ((rc = make_tmap_2d(&ep.tmEb, es->Eb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, n, V, V, 32, 32, 64)) != RL_OK)
            return rc;
        if ((rc = make_tmap_2d(&ep.tmEbt, es->Ebt, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, V, n, es->ldt, 32, 32, 0)) !=
            RL_OK)
            return rc;
    } else if (es != nullptr && es->E32 != nullptr) {
        ep.E32 = es->E32;
        ep.M2 = es->M2;
        if ((rc = make_tmap_2d(&ep.tmE32, es->E32, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, n, V, V, 32, 32, 128)) != RL_OK)
            return rc;
    }
    {
        ProfScope ps(RL_PROF_GEMM_FWD, stream);
        rc = launch_gemm_auto<EpiStats>(tmX, tmX, tmW, plan, ep, stream);
    }
    count_launch();
    if (rc != RL_OK) return rc;

    auto off = [c0](auto* p) { return p ? p + c0 : p; };
    TokenArgs ta;
    ta.N = n;
    ta.V = static_cast<int32_t>(V);
    ta.S = 2 * plan.n_splits;
    ta.nnz = nnz;
    ta.pstride = n;
    ta.part_m = w.part_m;
    ta.part_s = w.part_s;
    ta.part_u = w.part_u;
    ta.zlab = sv.zlab + c0;
    ta.zsup = sv.zsup;
    ta.labels = b->labels + c0;
    ta.label_logq = b->label_logq + c0;
    ta.adv = b->adv + c0;
    ta.loss_mask = off(b->loss_mask);
    ta.age = off(b->age);
    ta.offsets = b->support.offsets + c0;
    ta.ids = b->support.ids;
    ta.logq = b->support.logq;
    ta.replayed = b->support.replayed + c0;
    ta.loss_type = prm->loss_type;
    ta.kl_est = prm->kl_estimator;
    ta.kl_stale = prm->kl_staleness;
    ta.sparse = sparse;
    ta.eps = prm->eps;
    ta.cap = prm->max_importance_ratio;
    ta.lo = prm->icepop_low;
    ta.hi = prm->icepop_high;
    ta.adv_tau = prm->adv_tau;
    ta.kl_coeff = prm->kl_coeff;
    ta.ent_coeff = prm->entropy_coeff;
    ta.loss = out->loss + c0;
    ta.logp_label = off(out->logp_label);
    ta.logp_support = out->logp_support;
    ta.entropy = off(out->entropy);
    ta.lse_out = off(out->lse);
    ta.mask_label = off(out->mask_label);
    ta.mask_support = out->mask_support;
    ta.sv = sv;
    ta.sv.lse = sv.lse + c0;
    ta.sv.lse_s = sv.lse_s + c0;
    ta.sv.dcoef = sv.dcoef + c0;
    ta.sv.labcoef = sv.labcoef + c0;
    ta.sv.mterm = sv.mterm + c0 * 8;
    ta.sv.zlab = sv.zlab + c0;
    ta.status = status;
    const bool rows_scale = es != nullptr && es->Eb != nullptr;
    ta.cref = rows_scale ? es->cref : nullptr;
    ta.dloss = rows_scale ? es->dloss : nullptr;
    ta.inv_T = 1.0f / prm->temperature;
    ta.rs = rows_scale ? es->rs : nullptr;
    ta.flag = rows_scale ? es->flag : nullptr;
    {
        ProfScope ps(RL_PROF_TOKEN_LOSS, stream);
        token_loss_kernel<<<static_cast<unsigned>((n + 7) / 8), 256, 0, stream>>>(ta);
    }
    count_launch();
    return cudaPeekAtLastError() == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}

// ----------------------------------------------------------------------------------
// Vocabulary shards: the head split by rows of W (each rank a contiguous vocabulary range)
// ----------------------------------------------------------------------------------
// Global ids to a shard's local ids: id - v0 inside [v0, v1), -1 below, v1 - v0 above, so a
// row's ids stay in ascending order and the ids the shard does not own never match one of
// its columns.
__global__ void shard_remap_kernel(const int32_t* in, int64_t n, int32_t v0, int32_t v1, int32_t* out) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int32_t id = in[i];
    out[i] = id < v0 ? -1 : (id >= v1 ? v1 - v0 : id - v0);
}

// One (m, s, u) per token over the shard's columns from the GEMM's split partials (the same
// combination as token_loss_kernel's); stats [3][N]: m, then s, then u.
__global__ void shard_combine_kernel(const float* pm, const float* ps, const float* pu, int32_t S, int64_t N,
                                     float* stats) {
    const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t >= N) return;
    float M = -INFINITY;
    for (int i = 0; i < S; ++i) M = fmaxf(M, pm[static_cast<int64_t>(i) * N + t]);
    float sv = 0.f, uv = 0.f;
    for (int i = 0; i < S; ++i) {
        const int64_t k = static_cast<int64_t>(i) * N + t;
        const float f = expf(pm[k] - M);
        sv += f * ps[k];
        uv += f * (pu[k] + (pm[k] - M) * ps[k]);
    }
    stats[t] = M;
    stats[N + t] = sv;
    stats[2 * N + t] = uv;
}

int shard_remap_impl(const int32_t* in, int64_t n, int64_t v0, int64_t v1, int32_t* out, cudaStream_t stream) {
    if (n <= 0) return RL_OK;
    ProfScope ps(RL_PROF_OTHER, stream);
    shard_remap_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(
        in, n, static_cast<int32_t>(v0), static_cast<int32_t>(v1), out);
    count_launch();
    return cudaPeekAtLastError() == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}

int shard_stats_impl(const rl_head_batch* b, const rl_params* prm, float* stats, float* zlab, float* zsup, void* ws,
                     int32_t* status, cudaStream_t stream) {
    const int64_t N = b->N, H = b->H, V = b->V, nnz = b->support.nnz;
    if (N == 0) return RL_OK;
    const FwdWs w = fwd_ws_view(ws, N, H, V, nnz, nullptr);
    if (cudaMemsetAsync(zlab, 0, N * sizeof(float), stream) != cudaSuccess) return RL_ERR_CUDA;
    if (nnz > 0 && cudaMemsetAsync(zsup, 0, nnz * sizeof(float), stream) != cudaSuccess) return RL_ERR_CUDA;
    const int S = choose_splits(N, V);
    CUtensorMap tmX, tmW;
    int rc = make_tmap_bf16(&tmX, b->hidden, N, H, H, kBM);
    if (rc != RL_OK) return rc;
    rc = make_tmap_b(&tmW, b->weight, V, H, H);
    if (rc != RL_OK) return rc;
    const GemmPlan plan = make_plan_auto(N, V, H, 1, S, 1, status);
    EpiStats::Params ep;
    std::memset(&ep, 0, sizeof(ep));
    ep.N = N;
    ep.V = static_cast<int32_t>(V);
    ep.inv_T = 1.0f / prm->temperature;
    ep.c2 = kLog2e / prm->temperature;
    ep.nnz = nnz;
    ep.labels = b->labels;
    ep.offsets = b->support.offsets;
    ep.ids = b->support.ids;
    ep.zlab = zlab;
    ep.zsup = zsup;
    ep.part_m = w.part_m;
    ep.part_s = w.part_s;
    ep.part_u = w.part_u;
    ep.ldm = (V + 31) / 32;
    {
        ProfScope ps(RL_PROF_GEMM_FWD, stream);
        rc = launch_gemm_auto<EpiStats>(tmX, tmX, tmW, plan, ep, stream);
    }
    count_launch();
    if (rc != RL_OK) return rc;
    {
        ProfScope ps(RL_PROF_TOKEN_LOSS, stream);
        shard_combine_kernel<<<static_cast<unsigned>((N + 255) / 256), 256, 0, stream>>>(
            w.part_m, w.part_s, w.part_u, 2 * plan.n_splits, N, stats);
    }
    count_launch();
    return cudaPeekAtLastError() == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}

int loss_from_shards_impl(const rl_head_batch* b, const rl_params* prm, int32_t R, const float* stats_all,
                          const float* zlab, const float* zsup, const rl_head_outputs* out, void* saved, void* ws,
                          int32_t* status, cudaStream_t stream) {
    const int64_t N = b->N, nnz = b->support.nnz;
    int rc = validate_impl(b, status, stream);
    if (rc != RL_OK) return rc;
    if (N == 0) return RL_OK;
    const SavedView sv = saved_view(saved, N, nnz, nullptr);
    if (cudaMemcpyAsync(sv.zlab, zlab, N * sizeof(float), cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
        return RL_ERR_CUDA;
    if (nnz > 0 && cudaMemcpyAsync(sv.zsup, zsup, nnz * sizeof(float), cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
        return RL_ERR_CUDA;
    auto opt = [](auto* p) { return p; };
    TokenArgs ta;
    std::memset(&ta, 0, sizeof(ta));
    ta.N = N;
    ta.V = static_cast<int32_t>(b->V);
    ta.S = R;
    ta.nnz = nnz;
    ta.pstride = 3 * N;
    ta.part_m = stats_all;
    ta.part_s = stats_all + N;
    ta.part_u = stats_all + 2 * N;
    ta.zlab = sv.zlab;
    ta.zsup = sv.zsup;
    ta.labels = b->labels;
    ta.label_logq = b->label_logq;
    ta.adv = b->adv;
    ta.loss_mask = b->loss_mask;
    ta.age = b->age;
    ta.offsets = b->support.offsets;
    ta.ids = b->support.ids;
    ta.logq = b->support.logq;
    ta.replayed = b->support.replayed;
    ta.loss_type = prm->loss_type;
    ta.kl_est = prm->kl_estimator;
    ta.kl_stale = prm->kl_staleness;
    ta.sparse = !bwd_is_dense(prm);
    ta.eps = prm->eps;
    ta.cap = prm->max_importance_ratio;
    ta.lo = prm->icepop_low;
    ta.hi = prm->icepop_high;
    ta.adv_tau = prm->adv_tau;
    ta.kl_coeff = prm->kl_coeff;
    ta.ent_coeff = prm->entropy_coeff;
    ta.loss = out->loss;
    ta.logp_label = opt(out->logp_label);
    ta.logp_support = out->logp_support;
    ta.entropy = opt(out->entropy);
    ta.lse_out = opt(out->lse);
    ta.mask_label = opt(out->mask_label);
    ta.mask_support = out->mask_support;
    ta.sv = sv;
    ta.status = status;
    ta.inv_T = 1.0f / prm->temperature;
    {
        ProfScope ps(RL_PROF_TOKEN_LOSS, stream);
        token_loss_kernel<<<static_cast<unsigned>((N + 7) / 8), 256, 0, stream>>>(ta);
    }
    count_launch();
    if (cudaPeekAtLastError() != cudaSuccess) return RL_ERR_CUDA;
    if (out->metrics) return metrics_impl(b, saved, out->metrics, ws, stream);
    return RL_OK;
}

int head_fwd_impl(const rl_head_batch* b, const rl_params* prm, const rl_head_outputs* out,
                  void* saved, void* ws, int32_t* status, cudaStream_t stream) {
    if (keep_e_active(prm)) return head_fwd_kept(b, prm, out, saved, ws, status, stream);
    const int64_t N = b->N, H = b->H, V = b->V, nnz = b->support.nnz;
    int rc = validate_impl(b, status, stream);
    if (rc != RL_OK) return rc;
    if (N == 0) return RL_OK;
    const SavedView sv = saved_view(saved, N, nnz, nullptr);
    const FwdWs w = fwd_ws_view(ws, N, H, V, nnz, nullptr);
    rc = fwd_rows(b, prm, out, sv, w, 0, N, nullptr, !bwd_is_dense(prm), status, stream);
    if (rc != RL_OK) return rc;
    if (out->metrics) return metrics_impl(b, saved, out->metrics, ws, stream);
    return RL_OK;
}

}  // namespace rl
