// Backward of the fused LM head + unified RL loss (prime-rl pull request #4233, "Sparse
// LM-head backward": dense softmax-gradient GEMMs, or a deterministic CSR matmul when
// every logit gradient lies on the label and the support).
//
// With g_t = dloss_t the logit gradient of token t splits into
//     G_tj = alpha_t * P_full,tj  +  sum over spikes (label, support entries)
// where alpha_t = g_t * dcoef_t / T is non-zero only on untruncated rows whose gradient
// has a dense softmax part (the forward folds a replayed row's renormalised-softmax term
// into its support entries).  In the two-call path (and the fused hi/lo path) the spikes
// go through the sparse path exactly:
//     dX_t += sum_e c_e W[v_e],    dW[v] += sum_{e: v_e = v} c_e x_t     (fixed order)
// and the dense part, chunk by chunk over tokens, through three tcgen05 GEMMs:
//     G_c  = alpha * exp(X_c W^T / T - lse)      (EpiGrad: writes G_c [n, V] and G_c^T)
//     dX_c = G_c * W   (+ sparse dX, -> bf16)    (A = G_c, B = W^T copy, K = V)
//     dW  += G_c^T X_c                           (A = G_c^T, B = X_c^T copy, K = n)
#include <climits>
#include <cmath>


#include "gemm_tc2.cuh"
#include "internal.h"

namespace rl {

bool bwd_is_dense(const rl_params* prm) {
    if (prm->bwd_mode == RL_BWD_DENSE) return true;
    if (prm->bwd_mode == RL_BWD_SPARSE) return false;
    if (prm->entropy_coeff != 0.f) return true;   // the entropy gradient is dense
    const bool knobs_sparse = prm->loss_type == RL_LOSS_REINFORCE && prm->kl_coeff == 0.f;
    return !(knobs_sparse || prm->all_replayed != 0);
}

// Default token chunk of the backward (and of the fused forward + backward): the first
// multiple of the GEMM's row tile at or above 8192 tokens at which the dX GEMM's tiles
// (row blocks x H / 256 column tiles) fill whole waves of the GEMM's units (SM pairs, or
// SMs): 9728 with H = 2048 on 152 SMs (38 row blocks x 8 = 4 waves of 76 pairs), where 8192
// left a last wave 37 % full.  At the 64k-token batch 9728 took 83.4 / 84.2 ms against
// 84.1 / 85.8 at 8192 in alternating runs (dX 24.8 / 25.0 ms against 27.5 / 28.1); 16384
// held 4.7 GiB more for the same time as 8192, 4096 took 4 % longer.  Falls back to 8192
// if no such multiple lies below 16384.
static int64_t gcd64(int64_t a, int64_t b) {
    while (b != 0) {
        const int64_t t = a % b;
        a = b;
        b = t;
    }
    return a;
}
int64_t bwd_chunk(int64_t N, int64_t H, const rl_params* prm) {
    int64_t c = prm->token_chunk;
    if (c <= 0) {
        const bool pair = gemm_pair_mode() != 0;
        const int64_t units = pair ? num_sms() / 2 : num_sms();
        const int64_t rows = pair ? 2 * kBM : kBM;
        const int64_t cols = (H + kBN - 1) / kBN;
        const int64_t step = units / gcd64(units, cols > 0 ? cols : 1);   // row blocks per whole-wave set
        const int64_t rb = (8192 / rows + step - 1) / step * step;
        c = rb * rows;
        if (c < 8192 || c >= 16384) c = 8192;
    }
    c = (c + kBM - 1) / kBM * kBM;
    const int64_t n128 = (N + kBM - 1) / kBM * kBM;
    if (c > n128) c = n128;
    return c < kBM ? kBM : c;
}

constexpr int kSortTile = 2048;
constexpr int kDigitBits = 9;
constexpr int kDigits = 1 << kDigitBits;

BwdWs bwd_ws_view(void* base, int64_t N, int64_t H, int64_t V, int64_t nnz, const rl_params* prm,
                  size_t* bytes) {
    Carve c(base);
    BwdWs w{};
    w.dense = bwd_is_dense(prm);
    w.split = prm->grad_precision == RL_GRAD_SPLIT;
    w.chunk = bwd_chunk(N, H, prm);
    const int64_t items = nnz + N;
    if (w.dense) {
        w.Wt = c.take<uint16_t>(static_cast<size_t>(V) * H);
        w.Xt = c.take<uint16_t>(static_cast<size_t>(H) * w.chunk);
        w.G = c.take<uint16_t>(static_cast<size_t>(w.chunk) * V);
        w.Gt = c.take<uint16_t>(static_cast<size_t>(V) * w.chunk);
        if (w.split) {
            w.G_lo = c.take<uint16_t>(static_cast<size_t>(w.chunk) * V);
            w.Gt_lo = c.take<uint16_t>(static_cast<size_t>(V) * w.chunk);
        }
        w.dxs = c.take<float>(static_cast<size_t>(N) * H);
        w.resid = c.take<float>(nnz + N);
    }
    w.item_tok = c.take<int32_t>(items);
    w.keys_a = c.take<int32_t>(items);
    w.vals_a = c.take<int32_t>(items);
    w.keys_b = c.take<int32_t>(items);
    w.vals_b = c.take<int32_t>(items);
    const int64_t tiles = (items + kSortTile - 1) / kSortTile;
    w.hist = c.take<int32_t>(static_cast<size_t>(tiles > 0 ? tiles : 1) * kDigits);
    w.bucket = c.take<int64_t>(V + 2);
    if (bytes) *bytes = align_up(c.off, 256);
    return w;
}

// ----------------------------------------------------------------------------------
// GEMM epilogues
// ----------------------------------------------------------------------------------
RL_DEVINL uint32_t pack_bf16x2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// The dense softmax-gradient value alpha * exp(z - lse), with every rounding explicit so
// that the GEMM epilogue and the sparse path compute the same fp32 number.
RL_DEVINL float dense_alpha(float dloss, float dcoef, float inv_T) {
    return __fmul_rn(__fmul_rn(dloss, dcoef), inv_T);
}
RL_DEVINL float dense_grad(float alpha, float z, float lse) {
    if (alpha == 0.f) return 0.f;
    return __fmul_rn(alpha, exp2_approx(__fmul_rn(__fsub_rn(z, lse), kLog2e)));
}
// With the entropy regulariser ("10-KL-clip-entropy", section 3: loss -= c H) the dense
// part of G also holds (dloss / T) c p (log p + H): kappa = dloss c / T on an RL token
// (bit 0 of the saved metric flags), 0 otherwise; x = z - lse = log p.
RL_DEVINL float dense_kappa(float dloss, float ent_coeff, float inv_T, float mflags) {
    if (ent_coeff == 0.f || (__float_as_int(mflags) & 1) == 0) return 0.f;
    return __fmul_rn(__fmul_rn(dloss, ent_coeff), inv_T);
}
RL_DEVINL float dense_grad2(float alpha, float kappa, float ent, float z, float lse) {
    if (kappa == 0.f) return dense_grad(alpha, z, lse);
    const float x = __fsub_rn(z, lse);
    const float pv = exp2_approx(__fmul_rn(x, kLog2e));
    return __fmul_rn(pv, fmaf(kappa, __fadd_rn(x, ent), alpha));
}
// G = alpha_t * exp(z - lse_t) for the tile, written as G [n, V] (row-major, ld V) and
// G^T [V, ldt]; with `split`, also the bf16 remainder G - bf16(G) into G_lo / Gt_lo.
struct EpiGrad {
    struct Params {
        int64_t n;       // valid tokens of the chunk
        int32_t V;
        float inv_T;
        const float* lse;     // chunk-relative
        const float* dloss;   // chunk-relative
        const float* dcoef;   // chunk-relative
        uint16_t* G;
        uint16_t* Gt;
        uint16_t* G_lo;
        uint16_t* Gt_lo;
        int64_t ldt;
        const int* gate;      // fused path: run only when the chunk's range flag is set
        const float* mterm;   // chunk-relative [n, 8] saved metric terms (entropy, flags)
        float ent_coeff;
    };
    int64_t t;
    bool valid;
    float alpha, lse, kappa, ent;

    RL_DEVINL void begin_unit(const Params& p, int row, int, int m_blk, int, int) {
        t = static_cast<int64_t>(m_blk) * kBM + row;
        valid = t < p.n;
        alpha = 0.f;
        lse = 0.f;
        kappa = 0.f;
        ent = 0.f;
        if (valid) {
            alpha = dense_alpha(p.dloss[t], p.dcoef[t], p.inv_T);
            lse = p.lse[t];
            if (p.ent_coeff != 0.f) {
                kappa = dense_kappa(p.dloss[t], p.ent_coeff, p.inv_T, p.mterm[t * 8 + 7]);
                ent = p.mterm[t * 8 + 6];
            }
        }
    }
    RL_DEVINL void chunk(const Params& p, const uint32_t (&acc)[32], int col0, uint8_t*, int) {
        if (!valid || col0 >= p.V) return;
        const int nvalid = p.V - col0 < 32 ? p.V - col0 : 32;  // multiple of 8
        float g[32];
#pragma unroll
        for (int k = 0; k < 32; ++k)
            g[k] = dense_grad2(alpha, kappa, ent, __fmul_rn(__uint_as_float(acc[k]), p.inv_T), lse);
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            hi[k] = pack_bf16x2(g[2 * k], g[2 * k + 1]);
            if (p.G_lo) {
                const float h0 = bf16_bits_to_float(static_cast<uint16_t>(hi[k] & 0xFFFFu));
                const float h1 = bf16_bits_to_float(static_cast<uint16_t>(hi[k] >> 16));
                lo[k] = pack_bf16x2(g[2 * k] - h0, g[2 * k + 1] - h1);
            }
        }
        uint4* grow = reinterpret_cast<uint4*>(p.G + t * p.V + col0);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (q * 8 < nvalid) grow[q] = make_uint4(hi[4 * q], hi[4 * q + 1], hi[4 * q + 2], hi[4 * q + 3]);
        if (p.G_lo) {
            uint4* lrow = reinterpret_cast<uint4*>(p.G_lo + t * p.V + col0);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (q * 8 < nvalid) lrow[q] = make_uint4(lo[4 * q], lo[4 * q + 1], lo[4 * q + 2], lo[4 * q + 3]);
        }
        // transposed copy: for each column, the 32 lanes (consecutive tokens) write 64 B
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            if (k < nvalid) {
                const uint16_t hv = static_cast<uint16_t>((k & 1) ? (hi[k >> 1] >> 16) : (hi[k >> 1] & 0xFFFFu));
                p.Gt[static_cast<int64_t>(col0 + k) * p.ldt + t] = hv;
                if (p.Gt_lo) {
                    const uint16_t lv = static_cast<uint16_t>((k & 1) ? (lo[k >> 1] >> 16) : (lo[k >> 1] & 0xFFFFu));
                    p.Gt_lo[static_cast<int64_t>(col0 + k) * p.ldt + t] = lv;
                }
            }
        }
    }
    RL_DEVINL void end_unit(const Params&, int, int) {}
};

// dX rows of the chunk: bf16(rs_t acc + dxs) for columns < H, where rs_t is the row scale
// of the stored e (fused path; 1 when rs is absent or the chunk's range flag is set).
struct EpiDx {
    struct Params {
        int64_t n;
        int32_t H;
        const float* dxs;   // chunk-relative [n, H]
        uint16_t* out;      // chunk-relative [n, H] bf16
        const float* rs;    // chunk-relative [n], or nullptr
        const int* flag;    // with rs
        const int* dxs_gate;   // optional: dxs holds data only when *dxs_gate != 0
    };
    int64_t t;
    bool valid, with_dxs;
    float scale;
    RL_DEVINL void begin_unit(const Params& p, int row, int, int m_blk, int, int) {
        t = static_cast<int64_t>(m_blk) * kBM + row;
        valid = t < p.n;
        scale = 1.f;
        if (valid && p.rs != nullptr && *p.flag == 0) scale = p.rs[t];
        with_dxs = p.dxs_gate == nullptr || *p.dxs_gate != 0;
    }
    RL_DEVINL void chunk(const Params& p, const uint32_t (&acc)[32], int col0, uint8_t*, int) {
        if (!valid || col0 >= p.H) return;
        const float4* s = reinterpret_cast<const float4*>(p.dxs + t * p.H + col0);
        uint4* o = reinterpret_cast<uint4*>(p.out + t * p.H + col0);
        const float c = scale;
        const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 a = with_dxs ? s[2 * q] : zero, b = with_dxs ? s[2 * q + 1] : zero;
            o[q] = make_uint4(pack_bf16x2(fmaf(__uint_as_float(acc[8 * q + 0]), c, a.x), fmaf(__uint_as_float(acc[8 * q + 1]), c, a.y)),
                              pack_bf16x2(fmaf(__uint_as_float(acc[8 * q + 2]), c, a.z), fmaf(__uint_as_float(acc[8 * q + 3]), c, a.w)),
                              pack_bf16x2(fmaf(__uint_as_float(acc[8 * q + 4]), c, b.x), fmaf(__uint_as_float(acc[8 * q + 5]), c, b.y)),
                              pack_bf16x2(fmaf(__uint_as_float(acc[8 * q + 6]), c, b.z), fmaf(__uint_as_float(acc[8 * q + 7]), c, b.w)));
        }
    }
    RL_DEVINL void end_unit(const Params&, int, int) {}
};

// dW rows: dW = (accumulate ? dW : 0) + acc for columns < H, rows < V.
struct EpiDw {
    struct Params {
        int64_t V;
        int32_t H;
        int32_t accumulate;
        float* dW;
    };
    int64_t v;
    bool valid;
    RL_DEVINL void begin_unit(const Params& p, int row, int, int m_blk, int, int) {
        v = static_cast<int64_t>(m_blk) * kBM + row;
        valid = v < p.V;
    }
    RL_DEVINL void chunk(const Params& p, const uint32_t (&acc)[32], int col0, uint8_t*, int) {
        if (!valid || col0 >= p.H) return;
        float4* d = reinterpret_cast<float4*>(p.dW + v * p.H + col0);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float4 r = make_float4(__uint_as_float(acc[4 * q]), __uint_as_float(acc[4 * q + 1]),
                                   __uint_as_float(acc[4 * q + 2]), __uint_as_float(acc[4 * q + 3]));
            if (p.accumulate) {
                const float4 o = d[q];
                r.x += o.x;
                r.y += o.y;
                r.z += o.z;
                r.w += o.w;
            }
            d[q] = r;
        }
    }
    RL_DEVINL void end_unit(const Params&, int, int) {}
};

// ----------------------------------------------------------------------------------
// Transpose (bf16): out[c, r] = in[r, c] for r < rows, c < cols; with a row scale,
// out[c, r] = bf16(rs_r in[r, c]) (rs ignored when *flag is set)
// ----------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) transpose_bf16_kernel(const uint16_t* in, int64_t rows,
                                                             int64_t cols, int64_t ld_in,
                                                             uint16_t* out, int64_t ld_out,
                                                             const float* rs, const int* flag) {
    // 64 x 64 tile; 16-byte global loads and stores (8 elements), the transpose in shared
    // memory with a 65-element pitch (the rows 8 apart that a warp's lanes gather fall in
    // distinct banks)
    __shared__ uint16_t tile[64][65];
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 64;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 64;
    const bool scaled = rs != nullptr && *flag == 0;
    const bool vec_in = ((ld_in & 7) == 0) && ((reinterpret_cast<uintptr_t>(in) & 15) == 0);
    const bool vec_out = ((ld_out & 7) == 0) && ((reinterpret_cast<uintptr_t>(out) & 15) == 0);
    const int cv = (threadIdx.x & 7) * 8;   // column group of 8
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int i = (threadIdx.x >> 3) + 32 * k;   // tile row
        const int64_t r = r0 + i, c = c0 + cv;
        uint16_t v[8];
        if (r < rows && vec_in && c + 8 <= cols) {
            const uint4 q = *reinterpret_cast<const uint4*>(in + r * ld_in + c);
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[2 * j] = static_cast<uint16_t>(w[j] & 0xFFFFu);
                v[2 * j + 1] = static_cast<uint16_t>(w[j] >> 16);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = (r < rows && c + j < cols) ? in[r * ld_in + c + j] : 0;
        }
        if (scaled && r < rows) {
            const float sc = rs[r];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                v[j] = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(sc, bf16_bits_to_float(v[j]))));
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) tile[i][cv + j] = v[j];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int i = (threadIdx.x >> 3) + 32 * k;   // output row = input column c0 + i
        const int64_t c = c0 + i, r = r0 + cv;
        if (c >= cols) continue;
        uint16_t v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = tile[cv + j][i];
        if (vec_out && r + 8 <= rows) {
            uint4 q;
            q.x = v[0] | (static_cast<uint32_t>(v[1]) << 16);
            q.y = v[2] | (static_cast<uint32_t>(v[3]) << 16);
            q.z = v[4] | (static_cast<uint32_t>(v[5]) << 16);
            q.w = v[6] | (static_cast<uint32_t>(v[7]) << 16);
            *reinterpret_cast<uint4*>(out + c * ld_out + r) = q;
        } else {
            for (int j = 0; j < 8 && r + j < rows; ++j) out[c * ld_out + r + j] = v[j];
        }
    }
}

static int transpose_bf16(const void* in, int64_t rows, int64_t cols, int64_t ld_in, void* out,
                          int64_t ld_out, cudaStream_t s, const float* rs = nullptr, const int* flag = nullptr) {
    if (rows <= 0 || cols <= 0) return RL_OK;
    dim3 grid(static_cast<unsigned>((cols + 63) / 64), static_cast<unsigned>((rows + 63) / 64));
    if (grid.y > 65535u) return RL_ERR_UNSUPPORTED;
    ProfScope ps(RL_PROF_TRANSPOSE, s);
    transpose_bf16_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(in), rows, cols, ld_in,
                                               static_cast<uint16_t*>(out), ld_out, rs, flag);
    count_launch();
    return cudaPeekAtLastError() == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}

// ----------------------------------------------------------------------------------
// Sparse dX: dX_t = (g_t / T) (labcoef_t W[a_t] + sum_e entcoef_e W[v_e])
// One block per token; thread i owns hidden columns [8 i, 8 i + 8) (+ 2048 strides).
// ----------------------------------------------------------------------------------
struct SparseArgs {
    int64_t N, H, V, nnz;
    const uint16_t* W;
    const uint16_t* X;
    const int32_t* labels;
    const int64_t* offsets;
    const int32_t* ids;
    const float* dloss;
    const float* labcoef;
    const float* entcoef;
    float inv_T;
    // dense mode only (nullptr otherwise): per gradient item, what the bf16 dense GEMM
    // operand dropped at that (token, vocab id); non-zero once per distinct pair
    const float* resid;
    // optional: the sparse kernels do nothing unless *gate != 0 (device-side decision)
    const int* gate;
};

RL_DEVINL bool gate_closed(const int* gate) { return gate != nullptr && *gate == 0; }

// True when `v` occurs among ids[b, e) (ascending).
RL_DEVINL bool row_contains(const int32_t* ids, int64_t b, int64_t e, int32_t v) {
    int64_t lo = b, hi = e;
    while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if (ids[mid] < v)
            lo = mid + 1;
        else
            hi = mid;
    }
    return lo < e && ids[lo] == v;
}

// Residual at one spike: the exact fp32 dense value g_true = alpha exp(z - lse) minus what
// the dense GEMMs consume there (bf16 hi, and lo with the split), where g_gemm is either
// g_true itself (recompute path) or F * e from the stored fp32 e (fused path, hi/lo).
RL_DEVINL float spike_residual(float g_true, float g_gemm, bool split) {
    const float hi = __bfloat162float(__float2bfloat16_rn(g_gemm));
    float r = __fsub_rn(g_true, hi);
    if (split) r = __fsub_rn(r, __bfloat162float(__float2bfloat16_rn(__fsub_rn(g_gemm, hi))));
    return r;
}
// Per-row factor of the fused path: G = F * e with F = alpha 2^(m2 - lse log2(e)).
RL_DEVINL float fused_factor(float alpha, float m2, float lse) {
    if (alpha == 0.f) return 0.f;
    return __fmul_rn(alpha, exp2_approx(__fsub_rn(m2, __fmul_rn(lse, kLog2e))));
}
// G of one element on the fused hi/lo path, e = 2^(z log2(e) - m2): F e, plus the entropy
// term kappa p (log p + H) with p = 2^(m2 - lse log2(e)) e.
RL_DEVINL float fused_grad(float F, float kappa, float ent, float m2, float lse, float e) {
    if (kappa == 0.f) return __fmul_rn(F, e);
    if (e == 0.f) return 0.f;
    const float l2 = __fsub_rn(m2, __fmul_rn(lse, kLog2e));
    const float pv = __fmul_rn(exp2_approx(l2), e);
    const float lnp = __fmul_rn(__fadd_rn(__log2f(e), l2), 0.6931471805599453f);
    return fmaf(__fmul_rn(pv, kappa), __fadd_rn(lnp, ent), __fmul_rn(F, e));
}

struct ResidArgs {
    int64_t t0, n, V, nnz;
    const int32_t* labels;    // absolute
    const int64_t* offsets;   // absolute
    const int32_t* ids;
    const float* dloss;       // absolute
    const float* dcoef;       // absolute
    const float* lse;         // absolute
    const float* zlab;        // absolute
    const float* zsup;
    float inv_T;
    int split;
    float* resid;             // [nnz + N]
    // fused path, hi/lo: fp32 e [n, V] and m2 [n, ldm], chunk-relative
    const float* E32;
    const float* M2;
    int64_t ldm;
    // fused path, bf16: e [n, V] relative to the row reference, row scale rs [n], range flag
    const uint16_t* Eb;
    const float* rs;
    const int* flag;
    // none of the above: recompute path
    const float* mterm;       // absolute [N, 8]: entropy and flags for the entropy term
    float ent_coeff;
};

// One warp per token of [t0, t0 + n): residual at the label and at the first entry of each
// distinct support id; 0 elsewhere (duplicates, rows without a dense part).
__global__ void __launch_bounds__(256) resid_kernel(ResidArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (r >= a.n) return;
    const int64_t t = a.t0 + r;
    int64_t b = a.offsets[t], e = a.offsets[t + 1];
    b = b < 0 ? 0 : (b > a.nnz ? a.nnz : b);
    e = e < b ? b : (e > a.nnz ? a.nnz : e);
    const float alpha = dense_alpha(a.dloss[t], a.dcoef[t], a.inv_T);
    const float lse = a.lse[t];
    const float kappa = a.ent_coeff != 0.f ? dense_kappa(a.dloss[t], a.ent_coeff, a.inv_T, a.mterm[t * 8 + 7]) : 0.f;
    const float ent = a.ent_coeff != 0.f ? a.mterm[t * 8 + 6] : 0.f;
    const float sc = (a.Eb != nullptr && *a.flag == 0) ? a.rs[r] : 1.f;
    auto resid_at = [&](int32_t v, float z) -> float {
        if ((alpha == 0.f && kappa == 0.f) || v < 0 || v >= a.V) return 0.f;
        const float g_true = dense_grad2(alpha, kappa, ent, z, lse);
        if (a.Eb != nullptr)   // the GEMMs use sc * e (e = G itself after a recompute)
            return __fsub_rn(g_true, __fmul_rn(sc, bf16_bits_to_float(a.Eb[r * a.V + v])));
        float g_gemm = g_true;
        if (a.E32 != nullptr) {
            const float m2 = a.M2[r * a.ldm + (v >> 5)];
            g_gemm = fused_grad(fused_factor(alpha, m2, lse), kappa, ent, m2, lse, a.E32[r * a.V + v]);
        }
        return spike_residual(g_true, g_gemm, a.split != 0);
    };
    for (int64_t j = b + lane; j < e; j += 32) {
        const int32_t id = a.ids[j];
        const bool first = (j == b) || (a.ids[j - 1] != id);
        a.resid[j] = first ? resid_at(id, a.zsup[j]) : 0.f;
    }
    if (lane == 0) {
        const int32_t lab = a.labels[t];
        a.resid[a.nnz + t] = row_contains(a.ids, b, e, lab) ? 0.f : resid_at(lab, a.zlab[t]);
    }
}

static int launch_resid(const ResidArgs& a, cudaStream_t s) {
    if (a.n <= 0) return RL_OK;
    ProfScope ps(RL_PROF_RESID, s);
    resid_kernel<<<static_cast<unsigned>((a.n + 7) / 8), 256, 0, s>>>(a);
    count_launch();
    return cudaPeekAtLastError() == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}

RL_DEVINL void fma_row8(float (&acc)[8], const uint16_t* row, float c) {
    const uint4 v = *reinterpret_cast<const uint4*>(row);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        acc[2 * k] = fmaf(c, __uint_as_float(w[k] << 16), acc[2 * k]);
        acc[2 * k + 1] = fmaf(c, __uint_as_float(w[k] & 0xFFFF0000u), acc[2 * k + 1]);
    }
}

template <bool kToBf16>
__global__ void __launch_bounds__(256) sparse_dx_kernel(SparseArgs a, int64_t t0, float* dxs, uint16_t* dx_bf16) {
    if (gate_closed(a.gate)) return;
    const int64_t t = t0 + blockIdx.x;   // output row blockIdx.x (chunk-relative)
    const float g = a.dloss[t] * a.inv_T;
    int64_t b = a.offsets[t], e = a.offsets[t + 1];
    b = b < 0 ? 0 : (b > a.nnz ? a.nnz : b);
    e = e < b ? b : (e > a.nnz ? a.nnz : e);
    const int32_t lab = a.labels[t];
    float cl = g * a.labcoef[t];
    if (a.resid) cl += a.resid[a.nnz + t];
    for (int64_t h0 = static_cast<int64_t>(threadIdx.x) * 8; h0 < a.H; h0 += 256 * 8) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (g != 0.f) {
            if (lab >= 0 && lab < a.V && cl != 0.f) fma_row8(acc, a.W + lab * a.H + h0, cl);
            for (int64_t j = b; j < e; ++j) {
                const int32_t id = a.ids[j];
                float c = g * a.entcoef[j];
                if (a.resid) c += a.resid[j];
                if (id >= 0 && id < a.V && c != 0.f) fma_row8(acc, a.W + id * a.H + h0, c);
            }
        }
        if (kToBf16) {
            uint4 o = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                 pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
            *reinterpret_cast<uint4*>(dx_bf16 + t * a.H + h0) = o;
        } else {
            float4* o = reinterpret_cast<float4*>(dxs + static_cast<int64_t>(blockIdx.x) * a.H + h0);
            o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
    }
}

// ----------------------------------------------------------------------------------
// Sparse dW: stable LSD radix sort of the gradient items by vocab id, then one block per
// vocab id sums its items in item order (items: support entries 0..nnz-1, then labels).
// ----------------------------------------------------------------------------------
__global__ void items_init_kernel(SparseArgs a, int32_t* item_tok, int32_t* keys, int32_t* vals) {
    if (gate_closed(a.gate)) return;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= a.N) return;
    int64_t b = a.offsets[t], e = a.offsets[t + 1];
    b = b < 0 ? 0 : (b > a.nnz ? a.nnz : b);
    e = e < b ? b : (e > a.nnz ? a.nnz : e);
    for (int64_t j = b + lane; j < e; j += 32) {
        const int32_t id = a.ids[j];
        item_tok[j] = static_cast<int32_t>(t);
        keys[j] = (id >= 0 && id < a.V) ? id : static_cast<int32_t>(a.V);
        vals[j] = static_cast<int32_t>(j);
    }
    if (lane == 0) {
        const int64_t i = a.nnz + t;
        const int32_t lab = a.labels[t];
        item_tok[i] = static_cast<int32_t>(t);
        keys[i] = (lab >= 0 && lab < a.V) ? lab : static_cast<int32_t>(a.V);
        vals[i] = static_cast<int32_t>(i);
    }
}

// Entries with a corrupt row range never get a token; mark them out of range.
__global__ void items_guard_kernel(const int64_t* offsets, int64_t N, int64_t nnz, int32_t V,
                                   int32_t* item_tok, int32_t* keys, const int* gate) {
    if (gate_closed(gate)) return;
    const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (j >= nnz) return;
    const int32_t t = item_tok[j];
    bool ok = t >= 0 && t < N;
    if (ok) {
        const int64_t b = offsets[t], e = offsets[t + 1];
        ok = j >= b && j < e;
    }
    if (!ok) {
        item_tok[j] = 0;
        keys[j] = V;
    }
}

__global__ void __launch_bounds__(256) radix_hist_kernel(const int32_t* keys, int64_t n, int shift,
                                                         int32_t* hist, int64_t tiles, const int* gate) {
    if (gate_closed(gate)) return;
    __shared__ int cnt[kDigits];
    for (int i = threadIdx.x; i < kDigits; i += blockDim.x) cnt[i] = 0;
    __syncthreads();
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kSortTile;
    for (int i = threadIdx.x; i < kSortTile; i += blockDim.x) {
        const int64_t j = t0 + i;
        if (j < n) atomicAdd(&cnt[(keys[j] >> shift) & (kDigits - 1)], 1);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kDigits; i += blockDim.x) hist[static_cast<int64_t>(i) * tiles + blockIdx.x] = cnt[i];
}

// Exclusive scan over hist in digit-major order (single block).  Each thread takes a
// contiguous run of entries (16-byte loads, four in flight), the runs' sums are scanned
// across the block with warp shuffles, then each thread writes its run's prefixes.
__global__ void __launch_bounds__(1024) radix_scan_kernel(int32_t* hist, int64_t len, const int* gate) {
    if (gate_closed(gate)) return;
    __shared__ int64_t wtot[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // len is a multiple of kDigits, so every run starts and ends on a 16-byte boundary
    const int64_t per = ((len + blockDim.x - 1) / blockDim.x + 3) & ~int64_t(3);
    const int64_t b = static_cast<int64_t>(threadIdx.x) * per;
    const int64_t e = b + per < len ? b + per : len;
    int64_t s = 0;
#pragma unroll 4
    for (int64_t i = b; i < e; i += 4) {
        const int4 v = *reinterpret_cast<const int4*>(hist + i);
        s += static_cast<int64_t>(v.x) + v.y + v.z + v.w;
    }
    // exclusive scan of the runs' sums over the block
    int64_t x = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wtot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int64_t t = lane < static_cast<int>(blockDim.x >> 5) ? wtot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        wtot[lane] = t;   // inclusive over warps
    }
    __syncthreads();
    int64_t run = x - s + (warp > 0 ? wtot[warp - 1] : 0);
#pragma unroll 4
    for (int64_t i = b; i < e; i += 4) {
        int4 v = *reinterpret_cast<const int4*>(hist + i);
        int4 o;
        o.x = static_cast<int32_t>(run);
        run += v.x;
        o.y = static_cast<int32_t>(run);
        run += v.y;
        o.z = static_cast<int32_t>(run);
        run += v.z;
        o.w = static_cast<int32_t>(run);
        run += v.w;
        *reinterpret_cast<int4*>(hist + i) = o;
    }
}

// One block of eight warps per tile; warp w takes the tile's items [256 w, 256 w + 256) in
// order.  The warps' digit counts, scanned over the warps in order on top of the tile's
// base from hist, give each warp its own running base per digit; within a warp the rank
// among equal digits of each group of 32 comes from match.any.  Items keep their order
// within a digit: stable.
constexpr int kScatterWarps = kSortTile / 256;
static_assert(kScatterWarps * 256 == kSortTile && kScatterWarps <= 32, "tiles of whole 256-item warp shares");
__global__ void __launch_bounds__(256) radix_scatter_kernel(const int32_t* keys_in, const int32_t* vals_in,
                                                            int64_t n, int shift, const int32_t* hist,
                                                            int64_t tiles, int32_t* keys_out,
                                                            int32_t* vals_out, const int* gate) {
    if (gate_closed(gate)) return;
    __shared__ int cnt[kScatterWarps][kDigits];   // counts, then running bases
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kScatterWarps * kDigits; i += blockDim.x) (&cnt[0][0])[i] = 0;
    // the warp's 256 items, eight per lane, all loads in flight
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kSortTile + warp * 256;
    int32_t k[8], v[8];
    int dg[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int64_t j = t0 + r * 32 + lane;
        const bool act = j < n;
        k[r] = act ? keys_in[j] : 0;
        v[r] = act ? vals_in[j] : 0;
        dg[r] = act ? ((k[r] >> shift) & (kDigits - 1)) : kDigits;   // inactive lanes: their own group
    }
    __syncthreads();   // counters zeroed
#pragma unroll
    for (int r = 0; r < 8; ++r)
        if (dg[r] < kDigits) atomicAdd(&cnt[warp][dg[r]], 1);
    __syncthreads();
    for (int d = threadIdx.x; d < kDigits; d += blockDim.x) {
        int run = hist[static_cast<int64_t>(d) * tiles + blockIdx.x];
        for (int w = 0; w < kScatterWarps; ++w) {
            const int c = cnt[w][d];
            cnt[w][d] = run;
            run += c;
        }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const bool act = dg[r] < kDigits;
        const unsigned peers = __match_any_sync(0xffffffffu, dg[r]);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        int pos = 0;
        if (act) pos = cnt[warp][dg[r]] + rank;
        __syncwarp();
        const int leader_hi = 31 - __clz(peers);   // highest lane of the group updates the base
        if (act && lane == leader_hi) cnt[warp][dg[r]] += __popc(peers);
        __syncwarp();
        if (act) {
            keys_out[pos] = k[r];
            vals_out[pos] = v[r];
        }
    }
}

// bucket[v] = first sorted position whose key >= v, for v in [0, V + 1].
__global__ void bucket_kernel(const int32_t* keys, int64_t n, int32_t V, int64_t* bucket, const int* gate) {
    if (gate_closed(gate)) return;
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i > n) return;
    const int64_t prev = i == 0 ? -1 : keys[i - 1];
    const int64_t cur = i == n ? static_cast<int64_t>(V) + 1 : keys[i];
    for (int64_t v = prev + 1; v <= cur && v <= V + 1; ++v) bucket[v] = i;
}

// Four vocabulary rows per 256-thread block, 64 threads per row (8 columns per thread per
// pass over the row's items, H / 512 passes): four times the rows in flight per SM of a
// block per row, whose short life (two bucket loads, a few items, one 8 KB store) left
// the SMs waiting on latency.
constexpr int kDwRowsPerBlock = 4;
__global__ void __launch_bounds__(256) sparse_dw_kernel(SparseArgs a, const int32_t* vals,
                                                        const int32_t* item_tok, const int64_t* bucket,
                                                        float* dW, int overwrite) {
    if (gate_closed(a.gate)) return;
    constexpr int kRowThreads = 256 / kDwRowsPerBlock;
    const int64_t v = static_cast<int64_t>(blockIdx.x) * kDwRowsPerBlock + threadIdx.x / kRowThreads;
    if (v >= a.V) return;
    const int64_t b = bucket[v], e = bucket[v + 1];
    if (e <= b && !overwrite) return;   // overwrite: a row no item touches is written as zeros
    for (int64_t h0 = static_cast<int64_t>(threadIdx.x % kRowThreads) * 8; h0 < a.H; h0 += kRowThreads * 8) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int64_t i = b; i < e; ++i) {
            const int32_t item = vals[i];
            const int32_t t = item_tok[item];
            const float g = a.dloss[t] * a.inv_T;
            float c = g * (item < a.nnz ? a.entcoef[item] : a.labcoef[t]);
            if (a.resid) c += a.resid[item];
            if (c != 0.f) fma_row8(acc, a.X + static_cast<int64_t>(t) * a.H + h0, c);
        }
        float4* d = reinterpret_cast<float4*>(dW + v * a.H + h0);
        if (overwrite) {
            d[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            d[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
            continue;
        }
        float4 o0 = d[0], o1 = d[1];
        o0.x += acc[0];
        o0.y += acc[1];
        o0.z += acc[2];
        o0.w += acc[3];
        o1.x += acc[4];
        o1.y += acc[5];
        o1.z += acc[6];
        o1.w += acc[7];
        d[0] = o0;
        d[1] = o1;
    }
}

// overwrite: dW = the sparse part (every row written, no memset and no read of dW first);
// else dW += the sparse part.
static int sparse_dw(const SparseArgs& a, const BwdWs& w, float* dW, cudaStream_t s, int overwrite = 0) {
    const int64_t n = a.nnz + a.N;
    if (n >= (int64_t(1) << 31)) {
        set_last_error("sparse gradient items exceed 2^31");
        return RL_ERR_UNSUPPORTED;
    }
    ProfScope ps(RL_PROF_SPARSE_DW, s);
    items_init_kernel<<<static_cast<unsigned>((a.N + 7) / 8), 256, 0, s>>>(a, w.item_tok, w.keys_a, w.vals_a);
    if (a.nnz > 0)
        items_guard_kernel<<<static_cast<unsigned>((a.nnz + 255) / 256), 256, 0, s>>>(
            a.offsets, a.N, a.nnz, static_cast<int32_t>(a.V), w.item_tok, w.keys_a, a.gate);
    count_launch(2);
    const int64_t tiles = (n + kSortTile - 1) / kSortTile;
    int bits = 1;
    while ((int64_t(1) << bits) <= a.V) ++bits;  // keys in [0, V]
    const int passes = (bits + kDigitBits - 1) / kDigitBits;
    int32_t *kin = w.keys_a, *vin = w.vals_a, *kout = w.keys_b, *vout = w.vals_b;
    for (int p = 0; p < passes; ++p) {
        const int shift = p * kDigitBits;
        radix_hist_kernel<<<static_cast<unsigned>(tiles), 256, 0, s>>>(kin, n, shift, w.hist, tiles, a.gate);
        radix_scan_kernel<<<1, 1024, 0, s>>>(w.hist, tiles * kDigits, a.gate);
        radix_scatter_kernel<<<static_cast<unsigned>(tiles), 256, 0, s>>>(kin, vin, n, shift, w.hist, tiles, kout,
                                                                         vout, a.gate);
        count_launch(3);
        int32_t* tk = kin;
        kin = kout;
        kout = tk;
        int32_t* tv = vin;
        vin = vout;
        vout = tv;
    }
    bucket_kernel<<<static_cast<unsigned>((n + 1 + 255) / 256), 256, 0, s>>>(kin, n, static_cast<int32_t>(a.V), w.bucket,
                                                                             a.gate);
    sparse_dw_kernel<<<static_cast<unsigned>((a.V + kDwRowsPerBlock - 1) / kDwRowsPerBlock), 256, 0, s>>>(
        a, vin, w.item_tok, w.bucket, dW, overwrite);
    count_launch(2);
    return cudaPeekAtLastError() == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}

// ----------------------------------------------------------------------------------
// Entry
// ----------------------------------------------------------------------------------
static int head_bwd_kept(const rl_head_batch* b, const rl_params* prm, const void* saved, const float* dloss,
                         void* dhidden, float* dW, int accumulate, void* ws, int32_t* status, cudaStream_t stream);

int head_bwd_impl(const rl_head_batch* b, const rl_params* prm, const void* saved,
                  const float* dloss, void* dhidden, float* dW, int accumulate, void* ws,
                  int32_t* status, cudaStream_t stream) {
    if (keep_e_active(prm)) return head_bwd_kept(b, prm, saved, dloss, dhidden, dW, accumulate, ws, status, stream);
    const int64_t N = b->N, H = b->H, V = b->V, nnz = b->support.nnz;
    if (N == 0) {
        if (!accumulate && V > 0)
            if (cudaMemsetAsync(dW, 0, static_cast<size_t>(V) * H * sizeof(float), stream) != cudaSuccess)
                return RL_ERR_CUDA;
        return RL_OK;
    }
    const SavedView sv = saved_view(const_cast<void*>(saved), N, nnz, nullptr);
    const BwdWs w = bwd_ws_view(ws, N, H, V, nnz, prm, nullptr);
    SparseArgs sa{N, H, V, nnz,
                  static_cast<const uint16_t*>(b->weight), static_cast<const uint16_t*>(b->hidden),
                  b->labels, b->support.offsets, b->support.ids, dloss, sv.labcoef, sv.entcoef,
                  1.0f / prm->temperature, w.dense ? w.resid : nullptr};
    int rc;
    if (!w.dense) {
        {
            ProfScope ps(RL_PROF_SPARSE_DX, stream);
            sparse_dx_kernel<true><<<static_cast<unsigned>(N), 256, 0, stream>>>(sa, 0, nullptr, static_cast<uint16_t*>(dhidden));
        }
        count_launch();
        return sparse_dw(sa, w, dW, stream, accumulate ? 0 : 1);
    }

    ResidArgs ra{0, N, V, nnz, b->labels, b->support.offsets, b->support.ids, dloss, sv.dcoef, sv.lse,
                 sv.zlab, sv.zsup, 1.0f / prm->temperature, w.split ? 1 : 0, w.resid,
                 nullptr, nullptr, 0, nullptr, nullptr, nullptr, sv.mterm, prm->entropy_coeff};
    if ((rc = launch_resid(ra, stream)) != RL_OK) return rc;
    {
        ProfScope ps(RL_PROF_SPARSE_DX, stream);
        sparse_dx_kernel<false><<<static_cast<unsigned>(N), 256, 0, stream>>>(sa, 0, w.dxs, nullptr);
    }
    count_launch();
    rc = transpose_bf16(b->weight, V, H, H, w.Wt, V, stream);
    if (rc != RL_OK) return rc;

    CUtensorMap tmW, tmWt;
    rc = make_tmap_b(&tmW, b->weight, V, H, H);
    if (rc != RL_OK) return rc;
    rc = make_tmap_b(&tmWt, w.Wt, H, V, V);
    if (rc != RL_OK) return rc;
    const int passes = w.split ? 2 : 1;
    for (int64_t c0 = 0; c0 < N; c0 += w.chunk) {
        const int64_t n = N - c0 < w.chunk ? N - c0 : w.chunk;
        const uint16_t* Xc = static_cast<const uint16_t*>(b->hidden) + c0 * H;
        rc = transpose_bf16(Xc, n, H, H, w.Xt, w.chunk, stream);
        if (rc != RL_OK) return rc;
        CUtensorMap tmX, tmG, tmGlo, tmGt, tmGtlo, tmXt;
        if ((rc = make_tmap_bf16(&tmX, Xc, n, H, H, kBM)) != RL_OK) return rc;
        if ((rc = make_tmap_bf16(&tmG, w.G, n, V, V, kBM)) != RL_OK) return rc;
        if ((rc = make_tmap_bf16(&tmGt, w.Gt, V, n, w.chunk, kBM)) != RL_OK) return rc;
        if ((rc = make_tmap_b(&tmXt, w.Xt, H, n, w.chunk)) != RL_OK) return rc;
        tmGlo = tmG;
        tmGtlo = tmGt;
        if (w.split) {
            if ((rc = make_tmap_bf16(&tmGlo, w.G_lo, n, V, V, kBM)) != RL_OK) return rc;
            if ((rc = make_tmap_bf16(&tmGtlo, w.Gt_lo, V, n, w.chunk, kBM)) != RL_OK) return rc;
        }
        // G chunk (recomputed logits -> softmax gradient), both layouts
        EpiGrad::Params gp{n, static_cast<int32_t>(V), 1.0f / prm->temperature, sv.lse + c0, dloss + c0,
                           sv.dcoef + c0, static_cast<uint16_t*>(w.G), static_cast<uint16_t*>(w.Gt),
                           static_cast<uint16_t*>(w.G_lo), static_cast<uint16_t*>(w.Gt_lo), w.chunk, nullptr,
                           sv.mterm + c0 * 8, prm->entropy_coeff};
        const GemmPlan p1 = make_plan_auto(n, V, H, 1, 1 << 30, 1, status);
        {
            ProfScope ps(RL_PROF_GEMM_GRAD, stream);
            if ((rc = launch_gemm_auto<EpiGrad>(tmX, tmX, tmW, p1, gp, stream)) != RL_OK) return rc;
        }
        // dX chunk = G W + sparse part
        EpiDx::Params dp{n, static_cast<int32_t>(H), w.dxs + c0 * H, static_cast<uint16_t*>(dhidden) + c0 * H};
        const GemmPlan p2 = make_plan_auto(n, H, V, passes, 1 << 30, 0, status);
        {
            ProfScope ps(RL_PROF_GEMM_DX, stream);
            if ((rc = launch_gemm_auto<EpiDx>(tmG, tmGlo, tmWt, p2, dp, stream)) != RL_OK) return rc;
        }
        // dW += G^T X
        EpiDw::Params wp{V, static_cast<int32_t>(H), (c0 > 0 || accumulate) ? 1 : 0, dW};
        const GemmPlan p3 = make_plan_auto(V, H, n, passes, 1 << 30, 0, status);
        {
            ProfScope ps(RL_PROF_GEMM_DW, stream);
            if ((rc = launch_gemm_auto<EpiDw>(tmGt, tmGtlo, tmXt, p3, wp, stream)) != RL_OK) return rc;
        }
        count_launch(3);
    }
    return sparse_dw(sa, w, dW, stream);
}

// ----------------------------------------------------------------------------------
// Fused forward + backward (dloss known before the forward): no logit recompute.
//
// bf16 gradient precision.  Before a chunk's forward GEMM, each row gets a reference
// cref = z_label log2(e) (ref_logit_kernel).  The GEMM epilogue stores
// e = 2^(z log2(e) - cref) in bf16 twice, as Eb [n, V] and Ebt [V, n], and once the
// chunk's logsumexp is known the dense softmax gradient is G = rs * e with one scale per
// row, rs = alpha 2^(cref - lse log2(e)).  The scale is applied where it is free: in the
// dX epilogue (dX = rs * (e W)) and in the copy of X^T that dW consumes
// (dW += e^T (rs X)).  So the backward reads e straight from the forward's output.
// If a row's logits leave the range of that representation (max logit more than 2^64
// above the reference, or a scale out of range) the chunk's flag is set and a gated GEMM
// recomputes G into Eb / Ebt with rs = 1 (the two-call path's arithmetic).  The spikes
// are then folded into e (fold_kernel), so the dense GEMMs carry the whole gradient and
// the sparse kernels run (gated) only for rows without a dense part.
//
// hi/lo gradient precision.  The forward stores e = 2^(z log2(e) - m2) in fp32 with its
// running-max reference per 32-column chunk, and grad_from_e_kernel forms
// G = alpha 2^(m2 - lse log2(e)) e and its bf16 hi/lo split in both layouts.
// 6 N H V tensor flops per step either way (x2 for the dX / dW GEMMs with hi/lo).
// ----------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) ref_logit_kernel(const uint16_t* X, const uint16_t* W, const int32_t* labels,
                                                        int64_t n, int64_t H, int64_t V, float c2, float* cref,
                                                        int* flag) {
    const int lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (blockIdx.x == 0 && threadIdx.x == 0) *flag = 0;
    if (t >= n) return;
    const int32_t lab = labels[t];
    const bool ok = lab >= 0 && lab < V;
    float acc = 0.f;
    if (ok) {
        const uint16_t* x = X + t * H;
        const uint16_t* w = W + static_cast<int64_t>(lab) * H;
        for (int64_t h = lane * 8; h < H; h += 256) {
            const uint4 xv = *reinterpret_cast<const uint4*>(x + h);
            const uint4 wv = *reinterpret_cast<const uint4*>(w + h);
            const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w}, wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                acc = fmaf(__uint_as_float(xa[k] << 16), __uint_as_float(wa[k] << 16), acc);
                acc = fmaf(__uint_as_float(xa[k] & 0xFFFF0000u), __uint_as_float(wa[k] & 0xFFFF0000u), acc);
            }
        }
    }
    acc = warp_sum(acc);
    if (lane == 0) {
        const float c = acc * c2;
        cref[t] = (ok && isfinite(c)) ? c : 0.f;
    }
}

// Spikes (label and support coefficients, pull request #4233's loss_t differentiated with
// w, c, u held constant) folded into the stored e of their row: with the dense gradient
// G = rs e, the total gradient at (t, v) is rs (e + c / rs), so e[t, v] becomes
// bf16(e + c / rs) in both layouts and the dense GEMMs carry the spikes too.  e is
// re-formed there in fp32 from the forward's fp32 logit (zsup / zlab), so the stored
// value is rounded to bf16 once.  c sums every coefficient at that id (duplicate draws, a
// label that is also a support id) in entry order.  After a recompute (flag set) the
// stored value is G itself (rs = 1) and the fp32 value is alpha exp(z - lse).  A row with
// rs = 0 (no dense part: replayed, or a zero coefficient) cannot fold; its spikes stay on
// the sparse path, which gets dls_t = dloss_t for it (0 for folded rows), and the chunk's
// and the call's sparse gates open.  One warp per token.
struct FoldArgs {
    int64_t t0, n, V, nnz, ldt;
    const int32_t* labels;    // absolute
    const int64_t* offsets;   // absolute
    const int32_t* ids;
    const float* dloss;       // absolute
    const float* labcoef;     // absolute
    const float* entcoef;
    const float* zlab;        // absolute
    const float* zsup;
    const float* dcoef;       // absolute
    const float* lse;         // absolute
    float inv_T;
    const float* cref;        // chunk-relative
    const float* rs;          // chunk-relative
    const int* flag;
    uint16_t* Eb;             // [n, V] chunk
    uint16_t* Ebt;            // [V, ldt] chunk
    float* dls;               // absolute [N]
    int* open_chunk;
    int* open_any;
    const float* mterm;       // absolute [N, 8]
    float ent_coeff;
};

RL_DEVINL void fold_at(const FoldArgs& a, int64_t r, int32_t v, float x) {
    const uint16_t nv = __bfloat16_as_ushort(__float2bfloat16_rn(x));
    a.Eb[r * a.V + v] = nv;
    a.Ebt[static_cast<int64_t>(v) * a.ldt + r] = nv;
}

__global__ void __launch_bounds__(256) fold_kernel(FoldArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (r >= a.n) return;
    const int64_t t = a.t0 + r;
    int64_t b = a.offsets[t], e = a.offsets[t + 1];
    b = b < 0 ? 0 : (b > a.nnz ? a.nnz : b);
    e = e < b ? b : (e > a.nnz ? a.nnz : e);
    const float g = a.dloss[t] * a.inv_T;   // as the sparse path forms it
    const float sc = *a.flag != 0 ? 1.f : a.rs[r];
    const int32_t lab = a.labels[t];
    const float cl = g * a.labcoef[t];
    if (sc == 0.f) {
        bool any = false;
        for (int64_t j = b + lane; j < e; j += 32) any |= g * a.entcoef[j] != 0.f;
        any = __any_sync(0xffffffffu, any) || cl != 0.f;
        if (lane == 0) {
            a.dls[t] = a.dloss[t];
            if (any) {
                *a.open_chunk = 1;
                *a.open_any = 1;
            }
        }
        return;
    }
    if (lane == 0) a.dls[t] = 0.f;
    const bool rec = *a.flag != 0;
    const float alpha = dense_alpha(a.dloss[t], a.dcoef[t], a.inv_T);
    const float lse = a.lse[t], cr = a.cref[r];
    const float kappa = a.ent_coeff != 0.f ? dense_kappa(a.dloss[t], a.ent_coeff, a.inv_T, a.mterm[t * 8 + 7]) : 0.f;
    const float ent = a.ent_coeff != 0.f ? a.mterm[t * 8 + 6] : 0.f;
    auto dense_at = [&](float z) -> float {   // the stored quantity before rounding
        return rec ? dense_grad2(alpha, kappa, ent, z, lse) : exp2_approx(__fsub_rn(__fmul_rn(z, kLog2e), cr));
    };
    for (int64_t j = b + lane; j < e; j += 32) {
        const int32_t id = a.ids[j];
        if ((j > b && a.ids[j - 1] == id) || id < 0 || id >= a.V) continue;   // first entry of its id only
        float c = 0.f;
        for (int64_t k = j; k < e && a.ids[k] == id; ++k) c = __fadd_rn(c, g * a.entcoef[k]);
        if (id == lab) c = __fadd_rn(c, cl);
        if (c != 0.f) fold_at(a, r, id, __fadd_rn(dense_at(a.zsup[j]), c / sc));
    }
    if (lane == 0 && lab >= 0 && lab < a.V && cl != 0.f && !row_contains(a.ids, b, e, lab))
        fold_at(a, r, lab, __fadd_rn(dense_at(a.zlab[t]), cl / sc));
}

struct GradEArgs {
    int64_t n, V, ldm, ldt;
    const float* E32;     // fp32 e
    const float* M2;
    const float* dloss;   // chunk-relative
    const float* dcoef;
    const float* lse;
    float inv_T;
    uint16_t* G;
    uint16_t* Gt;
    uint16_t* G_lo;
    uint16_t* Gt_lo;
    const float* mterm;   // chunk-relative [n, 8]
    float ent_coeff;
};

constexpr int kGradTileT = 64;    // tokens per block
constexpr int kGradTileV = 128;   // vocabulary ids per block
constexpr int kGradPitch = 72;    // smem row pitch (halfwords): 144 B keeps 16-byte rows

// G = F e with one factor F = alpha 2^(m2 - lse log2 e) per row and 32-column chunk, and
// its bf16 hi/lo split.  Row-major pass: 16 threads cover one token's 128 columns (8
// each), so loads of e and stores of G are full row segments.  The tile is kept
// transposed in shared memory (token index XOR-swizzled by 8 per 8-column group against
// bank conflicts) and written as G^T with 16-byte stores, 8 threads per vocabulary row.
__global__ void __launch_bounds__(256) grad_from_e_kernel(GradEArgs a) {
    __shared__ __align__(16) uint16_t th[kGradTileV][kGradPitch];
    __shared__ __align__(16) uint16_t tl[kGradTileV][kGradPitch];
    const int tid = threadIdx.x;
    const int g = tid & 15;
    const int sw = (g & 7) << 3;
    const int64_t v = static_cast<int64_t>(blockIdx.x) * kGradTileV + g * 8;
    for (int pass = 0; pass < kGradTileT / 16; ++pass) {
        const int r = pass * 16 + (tid >> 4);
        const int64_t t = static_cast<int64_t>(blockIdx.y) * kGradTileT + r;
        uint32_t hi[4] = {0u, 0u, 0u, 0u}, lo[4] = {0u, 0u, 0u, 0u};
        if (t < a.n && v < a.V) {
            const float alpha = dense_alpha(a.dloss[t], a.dcoef[t], a.inv_T);
            const float m2 = a.M2[t * a.ldm + (v >> 5)];
            const float F = fused_factor(alpha, m2, a.lse[t]);
            const float kappa =
                a.ent_coeff != 0.f ? dense_kappa(a.dloss[t], a.ent_coeff, a.inv_T, a.mterm[t * 8 + 7]) : 0.f;
            const float ent = a.ent_coeff != 0.f ? a.mterm[t * 8 + 6] : 0.f;
            const float4* src = reinterpret_cast<const float4*>(a.E32 + t * a.V + v);
            const float4 x0 = src[0], x1 = src[1];
            const float e[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float g0 = fused_grad(F, kappa, ent, m2, a.lse[t], e[2 * k]);
                const float g1 = fused_grad(F, kappa, ent, m2, a.lse[t], e[2 * k + 1]);
                hi[k] = pack_bf16x2(g0, g1);
                const float h0 = bf16_bits_to_float(static_cast<uint16_t>(hi[k] & 0xFFFFu));
                const float h1 = bf16_bits_to_float(static_cast<uint16_t>(hi[k] >> 16));
                lo[k] = pack_bf16x2(g0 - h0, g1 - h1);
            }
            *reinterpret_cast<uint4*>(a.G + t * a.V + v) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(a.G_lo + t * a.V + v) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            th[g * 8 + k][r ^ sw] = static_cast<uint16_t>((k & 1) ? (hi[k >> 1] >> 16) : (hi[k >> 1] & 0xFFFFu));
            tl[g * 8 + k][r ^ sw] = static_cast<uint16_t>((k & 1) ? (lo[k >> 1] >> 16) : (lo[k >> 1] & 0xFFFFu));
        }
    }
    __syncthreads();
    const int64_t tbase = static_cast<int64_t>(blockIdx.y) * kGradTileT;
    for (int row = tid >> 3; row < kGradTileV; row += 32) {
        const int64_t vr = static_cast<int64_t>(blockIdx.x) * kGradTileV + row;
        if (vr >= a.V) continue;
        const int j = (tid & 7) * 8;
        const int jp = j ^ (((row >> 3) & 7) << 3);
        const int64_t tt = tbase + j;
        if (tt + 8 <= a.n) {
            *reinterpret_cast<uint4*>(a.Gt + vr * a.ldt + tt) = *reinterpret_cast<const uint4*>(&th[row][jp]);
            *reinterpret_cast<uint4*>(a.Gt_lo + vr * a.ldt + tt) = *reinterpret_cast<const uint4*>(&tl[row][jp]);
        } else {
            for (int k = 0; k < 8 && tt + k < a.n; ++k) {
                a.Gt[vr * a.ldt + tt + k] = th[row][jp + k];
                a.Gt_lo[vr * a.ldt + tt + k] = tl[row][jp + k];
            }
        }
    }
}

struct FusedWs {
    int64_t chunk;
    int64_t nchunks;
    FwdWs fw;
    // bf16 gradient precision
    uint16_t* Eb;    // [chunk, V]
    uint16_t* Ebt;   // [V, chunk]
    float* cref;     // [chunk]
    float* rs;       // [chunk]
    float* dls;      // [N] dloss for the rows whose spikes stay on the sparse path, else 0
    int* gates;      // [nchunks + 1] sparse-path gate per chunk, then for the whole call
    int* flags;      // [nchunks] range flag per chunk
    // hi/lo gradient precision
    float* E32;      // [chunk, V]
    float* M2;       // [chunk, ldm]
    int64_t ldm;
    BwdWs bw;   // Wt, Xt, dxs [chunk, H], resid, sort buffers; G, Gt, G_lo, Gt_lo with hi/lo
};

// kept: the backward of the kept-numerator two-call path, whose e / e^T and reference
// logits live in the saved state: no forward workspace and no chunk copies of them here.
static FusedWs fused_ws_view(void* base, int64_t N, int64_t H, int64_t V, int64_t nnz, const rl_params* prm,
                             size_t* bytes, bool kept = false) {
    FusedWs f{};
    f.chunk = bwd_chunk(N, H, prm);
    f.nchunks = (N + f.chunk - 1) / f.chunk;
    size_t fb = 0;
    if (!kept) f.fw = fwd_ws_view(base, f.chunk, H, V, nnz, &fb);
    Carve c(base ? static_cast<uint8_t*>(base) + fb : nullptr);
    c.off = 0;
    f.ldm = (V + 31) / 32;
    BwdWs& w = f.bw;
    w.dense = true;
    w.split = prm->grad_precision == RL_GRAD_SPLIT;
    w.chunk = f.chunk;
    if (w.split) {
        f.E32 = c.take<float>(static_cast<size_t>(f.chunk) * V);
        f.M2 = c.take<float>(static_cast<size_t>(f.chunk) * f.ldm);
        w.G = c.take<uint16_t>(static_cast<size_t>(f.chunk) * V);
        w.Gt = c.take<uint16_t>(static_cast<size_t>(V) * f.chunk);
        w.G_lo = c.take<uint16_t>(static_cast<size_t>(f.chunk) * V);
        w.Gt_lo = c.take<uint16_t>(static_cast<size_t>(V) * f.chunk);
    } else {
        if (!kept) {
            f.Eb = c.take<uint16_t>(static_cast<size_t>(f.chunk) * V);
            f.Ebt = c.take<uint16_t>(static_cast<size_t>(V) * f.chunk);
            f.cref = c.take<float>(f.chunk);
        }
        f.rs = c.take<float>(f.chunk);
        f.dls = c.take<float>(N);
        f.gates = c.take<int>(f.nchunks + 1);
    }
    f.flags = c.take<int>(f.nchunks > 0 ? f.nchunks : 1);
    w.Wt = c.take<uint16_t>(static_cast<size_t>(V) * H);
    w.Xt = c.take<uint16_t>(static_cast<size_t>(H) * f.chunk);
    w.dxs = c.take<float>(static_cast<size_t>(f.chunk) * H);
    w.resid = c.take<float>(nnz + N);
    const int64_t items = nnz + N;
    w.item_tok = c.take<int32_t>(items);
    w.keys_a = c.take<int32_t>(items);
    w.vals_a = c.take<int32_t>(items);
    w.keys_b = c.take<int32_t>(items);
    w.vals_b = c.take<int32_t>(items);
    const int64_t tiles = (items + kSortTile - 1) / kSortTile;
    w.hist = c.take<int32_t>(static_cast<size_t>(tiles > 0 ? tiles : 1) * kDigits);
    w.bucket = c.take<int64_t>(V + 2);
    if (bytes) *bytes = align_up(fb + c.off, 256);
    return f;
}

size_t fused_ws_bytes(int64_t N, int64_t H, int64_t V, int64_t nnz, const rl_params* prm) {
    if (!bwd_is_dense(prm)) {   // no dense GEMMs: the forward, then the sparse backward
        size_t a = 0, b = 0;
        fwd_ws_view(nullptr, N, H, V, nnz, &a);
        bwd_ws_view(nullptr, N, H, V, nnz, prm, &b);
        return a > b ? a : b;
    }
    size_t bytes = 0;
    fused_ws_view(nullptr, N, H, V, nnz, prm, &bytes);
    return bytes;
}

// The BF16 backward of one token chunk from its softmax numerators e / e^T (the fused
// call's chunk buffers, or the ones the forward kept for every token), once the row scales
// rs are formed: the gated logit recompute for a chunk whose range flag is up, the spikes
// folded into e, X^T scaled by rs, the sparse part of the rows that cannot fold, dX and dW.
struct ChunkE {
    uint16_t* Eb;        // [n, V] from the chunk's first token
    uint16_t* Ebt;       // [V, ldt] from the chunk's first token's column
    int64_t ldt;
    const float* cref;   // [n]
    float* rs;           // [n]
    int* flag;           // the chunk's range flag
};
static int bf16_chunk_bwd(const rl_head_batch* b, const rl_params* prm, const SavedView& sv, const float* dloss,
                          int64_t c0, int64_t n, int64_t ci, const FusedWs& f, const ChunkE& ce, const SparseArgs& sa,
                          const CUtensorMap& tmW, const CUtensorMap& tmWt, void* dhidden, float* dW, int accumulate,
                          int32_t* status, cudaStream_t stream) {
    const int64_t H = b->H, V = b->V, nnz = b->support.nnz;
    const BwdWs& w = f.bw;
    const float inv_T = 1.0f / prm->temperature;
    const uint16_t* Xc = static_cast<const uint16_t*>(b->hidden) + c0 * H;
    int rc;
    // out-of-range chunk only: G recomputed from the logits into Eb / Ebt (rs := 1)
    CUtensorMap tmX;
    if ((rc = make_tmap_bf16(&tmX, Xc, n, H, H, kBM)) != RL_OK) return rc;
    EpiGrad::Params gp{n, static_cast<int32_t>(V), inv_T, sv.lse + c0, dloss + c0, sv.dcoef + c0,
                       ce.Eb, ce.Ebt, nullptr, nullptr, ce.ldt, ce.flag, sv.mterm + c0 * 8, prm->entropy_coeff};
    const GemmPlan pg = make_plan_auto(n, V, H, 1, 1 << 30, 1, status);
    {
        ProfScope ps(RL_PROF_GEMM_GRAD, stream);
        if ((rc = launch_gemm_auto<EpiGrad>(tmX, tmX, tmW, pg, gp, stream)) != RL_OK) return rc;
    }
    count_launch();
    {
        FoldArgs fa{c0, n, V, nnz, ce.ldt, b->labels, b->support.offsets, b->support.ids, dloss,
                    sv.labcoef, sv.entcoef, sv.zlab, sv.zsup, sv.dcoef, sv.lse, inv_T, ce.cref, ce.rs, ce.flag,
                    ce.Eb, ce.Ebt, f.dls, f.gates + ci, f.gates + f.nchunks, sv.mterm, prm->entropy_coeff};
        ProfScope ps(RL_PROF_RESID, stream);
        fold_kernel<<<static_cast<unsigned>((n + 7) / 8), 256, 0, stream>>>(fa);
        count_launch();
    }
    if ((rc = transpose_bf16(Xc, n, H, H, w.Xt, f.chunk, stream, ce.rs, ce.flag)) != RL_OK) return rc;
    CUtensorMap tmA, tmAt, tmXt;
    if ((rc = make_tmap_bf16(&tmA, ce.Eb, n, V, V, kBM)) != RL_OK) return rc;
    if ((rc = make_tmap_bf16(&tmAt, ce.Ebt, V, n, ce.ldt, kBM)) != RL_OK) return rc;
    {
        SparseArgs sc = sa;
        sc.gate = f.gates + ci;
        ProfScope ps(RL_PROF_SPARSE_DX, stream);
        sparse_dx_kernel<false><<<static_cast<unsigned>(n), 256, 0, stream>>>(sc, c0, w.dxs, nullptr);
        count_launch();
    }
    if ((rc = make_tmap_b(&tmXt, w.Xt, H, n, f.chunk)) != RL_OK) return rc;
    EpiDx::Params dp{n, static_cast<int32_t>(H), w.dxs, static_cast<uint16_t*>(dhidden) + c0 * H, ce.rs, ce.flag,
                     f.gates + ci};
    const GemmPlan p2 = make_plan_auto(n, H, V, 1, 1 << 30, 0, status);
    {
        ProfScope ps(RL_PROF_GEMM_DX, stream);
        if ((rc = launch_gemm_auto<EpiDx>(tmA, tmA, tmWt, p2, dp, stream)) != RL_OK) return rc;
    }
    EpiDw::Params wp{V, static_cast<int32_t>(H), (c0 > 0 || accumulate) ? 1 : 0, dW};
    const GemmPlan p3 = make_plan_auto(V, H, n, 1, 1 << 30, 0, status);
    {
        ProfScope ps(RL_PROF_GEMM_DW, stream);
        if ((rc = launch_gemm_auto<EpiDw>(tmAt, tmAt, tmXt, p3, wp, stream)) != RL_OK) return rc;
    }
    count_launch(2);
    return RL_OK;
}

// ----------------------------------------------------------------------------------
// Kept numerators (rl_params.keep_e): the two-call path without the logit recompute
// ----------------------------------------------------------------------------------
bool keep_e_active(const rl_params* prm) {
    return prm != nullptr && prm->keep_e != 0 && bwd_is_dense(prm) && prm->grad_precision == RL_GRAD_BF16 &&
           prm->entropy_coeff == 0.f;
}

KeptView kept_view(void* saved, int64_t N, int64_t nnz, int64_t V, const rl_params* prm, size_t* bytes) {
    size_t sb = 0;
    saved_view(nullptr, N, nnz, &sb);
    Carve c(saved ? static_cast<uint8_t*>(saved) + sb : nullptr);
    KeptView k{};
    k.chunks_max = (N + kBM - 1) / kBM;   // the smallest chunk is one row tile
    k.ldt = (N + kBM - 1) / kBM * kBM;
    k.Eb = c.take<uint16_t>(static_cast<size_t>(N) * V);
    k.Ebt = c.take<uint16_t>(static_cast<size_t>(V) * k.ldt);
    k.cref = c.take<float>(N);
    k.flags = c.take<int>(k.chunks_max > 0 ? k.chunks_max : 1);
    if (bytes) *bytes = align_up(sb + c.off, 256);
    return k;
}

size_t kept_bwd_ws_bytes(int64_t N, int64_t H, int64_t V, int64_t nnz, const rl_params* prm) {
    size_t bytes = 0;
    fused_ws_view(nullptr, N, H, V, nnz, prm, &bytes, true);
    return bytes;
}

// Forward with keep_e: per token chunk, the reference logits, then the forward GEMM that
// also stores e (row-major, from the chunk's first row) and e^T (columns from the chunk's
// first token, leading dimension N rounded up to 128) into the saved state and raises the chunk's flag when
// a row's logits leave the bf16 range around its reference.  Everything else as the plain
// forward.
int head_fwd_kept(const rl_head_batch* b, const rl_params* prm, const rl_head_outputs* out, void* saved,
                  void* ws, int32_t* status, cudaStream_t stream) {
    const int64_t N = b->N, H = b->H, V = b->V, nnz = b->support.nnz;
    int rc = validate_impl(b, status, stream);
    if (rc != RL_OK) return rc;
    if (N == 0) return RL_OK;
    const SavedView sv = saved_view(saved, N, nnz, nullptr);
    const KeptView k = kept_view(saved, N, nnz, V, prm, nullptr);
    const FwdWs w = fwd_ws_view(ws, N, H, V, nnz, nullptr);
    const float inv_T = 1.0f / prm->temperature;
    const int64_t chunk = bwd_chunk(N, H, prm);   // the backward's chunk
    const int64_t nchunks = (N + chunk - 1) / chunk;
    if (cudaMemsetAsync(k.flags, 0, sizeof(int) * nchunks, stream) != cudaSuccess) return RL_ERR_CUDA;
    for (int64_t c0 = 0, ci = 0; c0 < N; c0 += chunk, ++ci) {
        const int64_t n = N - c0 < chunk ? N - c0 : chunk;
        const uint16_t* Xc = static_cast<const uint16_t*>(b->hidden) + c0 * H;
        {
            ProfScope ps(RL_PROF_REF_LOGIT, stream);
            ref_logit_kernel<<<static_cast<unsigned>((n + 7) / 8), 256, 0, stream>>>(
                Xc, static_cast<const uint16_t*>(b->weight), b->labels + c0, n, H, V, kLog2e * inv_T, k.cref + c0,
                k.flags + ci);
            count_launch();
        }
        EStore es;
        es.Eb = k.Eb + c0 * V;
        es.Ebt = k.Ebt + c0;
        es.ldt = k.ldt;
        es.cref = k.cref + c0;
        es.flag = k.flags + ci;
        es.rs = nullptr;      // the row scales need dloss: the backward forms them
        es.dloss = nullptr;
        if ((rc = fwd_rows(b, prm, out, sv, w, c0, n, &es, 0, status, stream)) != RL_OK) return rc;
    }
    if (out->metrics) return metrics_impl(b, saved, out->metrics, ws, stream);
    return RL_OK;
}

// rs_t = alpha 2^(cref_t - lse_t log2 e) with alpha = dloss_t dcoef_t / T, formed as the
// fused call's token pass forms it (the same bits); a gap outside the bf16 range, or a
// non-finite factor, raises the chunk's recompute flag.  Chunk-relative arrays.
__global__ void __launch_bounds__(256) rs_kernel(const float* dloss, const float* dcoef, const float* lse,
                                                 const float* cref, float inv_T, int64_t n, float* rs, int* flag) {
    const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (r >= n) return;
    const float alpha = __fmul_rn(__fmul_rn(dloss[r], dcoef[r]), inv_T);
    float v = 0.f;
    if (alpha != 0.f) {
        const float gap = __fsub_rn(cref[r], __fmul_rn(lse[r], kLog2e));
        v = __fmul_rn(alpha, exp2_approx(gap));
        if (!(gap >= -kRefRangeLog2 && gap <= kRefRangeLog2) || !isfinite(v)) *flag = 1;
    }
    rs[r] = v;
}

// Backward with keep_e: the fused call's backward, chunk by chunk, on the kept numerators.
static int head_bwd_kept(const rl_head_batch* b, const rl_params* prm, const void* saved, const float* dloss,
                         void* dhidden, float* dW, int accumulate, void* ws, int32_t* status, cudaStream_t stream) {
    const int64_t N = b->N, H = b->H, V = b->V, nnz = b->support.nnz;
    if (N == 0) {
        if (!accumulate && V > 0 &&
            cudaMemsetAsync(dW, 0, static_cast<size_t>(V) * H * sizeof(float), stream) != cudaSuccess)
            return RL_ERR_CUDA;
        return RL_OK;
    }
    void* sp = const_cast<void*>(saved);
    const SavedView sv = saved_view(sp, N, nnz, nullptr);
    const KeptView k = kept_view(sp, N, nnz, V, prm, nullptr);
    const FusedWs f = fused_ws_view(ws, N, H, V, nnz, prm, nullptr, true);
    const float inv_T = 1.0f / prm->temperature;
    SparseArgs sa{N, H, V, nnz,
                  static_cast<const uint16_t*>(b->weight), static_cast<const uint16_t*>(b->hidden),
                  b->labels, b->support.offsets, b->support.ids, f.dls, sv.labcoef, sv.entcoef,
                  inv_T, nullptr, f.gates + f.nchunks};
    if (cudaMemsetAsync(f.gates, 0, sizeof(int) * (f.nchunks + 1), stream) != cudaSuccess) return RL_ERR_CUDA;
    int rc = transpose_bf16(b->weight, V, H, H, f.bw.Wt, V, stream);
    if (rc != RL_OK) return rc;
    CUtensorMap tmW, tmWt;
    if ((rc = make_tmap_b(&tmW, b->weight, V, H, H)) != RL_OK) return rc;
    if ((rc = make_tmap_b(&tmWt, f.bw.Wt, H, V, V)) != RL_OK) return rc;
    for (int64_t c0 = 0, ci = 0; c0 < N; c0 += f.chunk, ++ci) {
        const int64_t n = N - c0 < f.chunk ? N - c0 : f.chunk;
        {
            ProfScope ps(RL_PROF_TOKEN_LOSS, stream);
            rs_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(
                dloss + c0, sv.dcoef + c0, sv.lse + c0, k.cref + c0, inv_T, n, f.rs, k.flags + ci);
            count_launch();
        }
        const ChunkE ce{k.Eb + c0 * V, k.Ebt + c0, k.ldt, k.cref + c0, f.rs, k.flags + ci};
        if ((rc = bf16_chunk_bwd(b, prm, sv, dloss, c0, n, ci, f, ce, sa, tmW, tmWt, dhidden, dW, accumulate,
                                 status, stream)) != RL_OK)
            return rc;
    }
    return sparse_dw(sa, f.bw, dW, stream);
}

int head_fused_impl(const rl_head_batch* b, const rl_params* prm, const rl_head_outputs* out,
                    const float* dloss, void* dhidden, float* dW, int accumulate, void* saved, void* ws,
                    int32_t* status, cudaStream_t stream) {
    const int64_t N = b->N, H = b->H, V = b->V, nnz = b->support.nnz;
    if (!bwd_is_dense(prm)) {
        int rc = head_fwd_impl(b, prm, out, saved, ws, status, stream);
        if (rc != RL_OK) return rc;
        return head_bwd_impl(b, prm, saved, dloss, dhidden, dW, accumulate, ws, status, stream);
    }
    int rc = validate_impl(b, status, stream);
    if (rc != RL_OK) return rc;
    if (N == 0) {
        if (!accumulate && cudaMemsetAsync(dW, 0, static_cast<size_t>(V) * H * sizeof(float), stream) != cudaSuccess)
            return RL_ERR_CUDA;
        return RL_OK;
    }
    const SavedView sv = saved_view(saved, N, nnz, nullptr);
    const FusedWs f = fused_ws_view(ws, N, H, V, nnz, prm, nullptr);
    const BwdWs& w = f.bw;
    const float inv_T = 1.0f / prm->temperature;
    // hi/lo: exact spikes on the sparse path (with the residuals of the dense operands);
    // bf16: spikes folded into e, the sparse path only for rows that cannot fold
    SparseArgs sa{N, H, V, nnz,
                  static_cast<const uint16_t*>(b->weight), static_cast<const uint16_t*>(b->hidden),
                  b->labels, b->support.offsets, b->support.ids, w.split ? dloss : f.dls, sv.labcoef, sv.entcoef,
                  inv_T, w.split ? w.resid : nullptr, w.split ? nullptr : f.gates + f.nchunks};
    if (!w.split && cudaMemsetAsync(f.gates, 0, sizeof(int) * (f.nchunks + 1), stream) != cudaSuccess)
        return RL_ERR_CUDA;
    rc = transpose_bf16(b->weight, V, H, H, w.Wt, V, stream);
    if (rc != RL_OK) return rc;
    CUtensorMap tmW, tmWt;
    if ((rc = make_tmap_b(&tmW, b->weight, V, H, H)) != RL_OK) return rc;
    if ((rc = make_tmap_b(&tmWt, w.Wt, H, V, V)) != RL_OK) return rc;
    const int passes = w.split ? 2 : 1;
    for (int64_t c0 = 0, ci = 0; c0 < N; c0 += f.chunk, ++ci) {
        const int64_t n = N - c0 < f.chunk ? N - c0 : f.chunk;
        const uint16_t* Xc = static_cast<const uint16_t*>(b->hidden) + c0 * H;
        int* flag = f.flags + ci;
        CUtensorMap tmA, tmAlo, tmAt, tmAtlo, tmXt;
        EStore es;
        if (!w.split) {
            es.Eb = f.Eb;
            es.Ebt = f.Ebt;
            es.ldt = f.chunk;
            es.cref = f.cref;
            es.flag = flag;
            es.rs = f.rs;
            es.dloss = dloss + c0;
            {
                ProfScope ps(RL_PROF_REF_LOGIT, stream);
                ref_logit_kernel<<<static_cast<unsigned>((n + 7) / 8), 256, 0, stream>>>(
                    Xc, static_cast<const uint16_t*>(b->weight), b->labels + c0, n, H, V, kLog2e * inv_T, f.cref, flag);
                count_launch();
            }
        } else {
            es.E32 = f.E32;
            es.M2 = f.M2;
        }
        // forward GEMM (+ e store) and per-token loss for the chunk
        if ((rc = fwd_rows(b, prm, out, sv, f.fw, c0, n, &es, 0, status, stream)) != RL_OK) return rc;
        // the entropy term is not a row scale of e: such a chunk takes the recompute path
        if (!w.split && prm->entropy_coeff != 0.f && cudaMemsetAsync(flag, 1, 1, stream) != cudaSuccess)
            return RL_ERR_CUDA;
        if (!w.split) {
            const ChunkE ce{f.Eb, f.Ebt, f.chunk, f.cref, f.rs, flag};
            if ((rc = bf16_chunk_bwd(b, prm, sv, dloss, c0, n, ci, f, ce, sa, tmW, tmWt, dhidden, dW, accumulate,
                                     status, stream)) != RL_OK)
                return rc;
            continue;
        } else {
            // spike residuals of the chunk's tokens, then G / G^T (hi/lo) from e
            ResidArgs ra{c0, n, V, nnz, b->labels, b->support.offsets, b->support.ids, dloss, sv.dcoef, sv.lse,
                         sv.zlab, sv.zsup, inv_T, 1, w.resid, f.E32, f.M2, f.ldm, nullptr, nullptr, nullptr,
                         sv.mterm, prm->entropy_coeff};
            if ((rc = launch_resid(ra, stream)) != RL_OK) return rc;
            {
                GradEArgs ga{n, V, f.ldm, f.chunk, f.E32, f.M2, dloss + c0, sv.dcoef + c0, sv.lse + c0, inv_T,
                             static_cast<uint16_t*>(w.G), static_cast<uint16_t*>(w.Gt),
                             static_cast<uint16_t*>(w.G_lo), static_cast<uint16_t*>(w.Gt_lo), sv.mterm + c0 * 8,
                             prm->entropy_coeff};
                dim3 grid(static_cast<unsigned>((V + kGradTileV - 1) / kGradTileV),
                          static_cast<unsigned>((n + kGradTileT - 1) / kGradTileT));
                ProfScope ps(RL_PROF_GRAD_E, stream);
                grad_from_e_kernel<<<grid, 256, 0, stream>>>(ga);
                count_launch();
            }
            if ((rc = transpose_bf16(Xc, n, H, H, w.Xt, f.chunk, stream)) != RL_OK) return rc;
            if ((rc = make_tmap_bf16(&tmA, w.G, n, V, V, kBM)) != RL_OK) return rc;
            if ((rc = make_tmap_bf16(&tmAt, w.Gt, V, n, f.chunk, kBM)) != RL_OK) return rc;
            if ((rc = make_tmap_bf16(&tmAlo, w.G_lo, n, V, V, kBM)) != RL_OK) return rc;
            if ((rc = make_tmap_bf16(&tmAtlo, w.Gt_lo, V, n, f.chunk, kBM)) != RL_OK) return rc;
        }
        {
            SparseArgs sc = sa;
            if (!w.split) sc.gate = f.gates + ci;
            ProfScope ps(RL_PROF_SPARSE_DX, stream);
            sparse_dx_kernel<false><<<static_cast<unsigned>(n), 256, 0, stream>>>(sc, c0, w.dxs, nullptr);
            count_launch();
        }
        if ((rc = make_tmap_b(&tmXt, w.Xt, H, n, f.chunk)) != RL_OK) return rc;
        EpiDx::Params dp{n, static_cast<int32_t>(H), w.dxs, static_cast<uint16_t*>(dhidden) + c0 * H,
                         w.split ? nullptr : f.rs, flag, w.split ? nullptr : f.gates + ci};
        const GemmPlan p2 = make_plan_auto(n, H, V, passes, 1 << 30, 0, status);
        {
            ProfScope ps(RL_PROF_GEMM_DX, stream);
            if ((rc = launch_gemm_auto<EpiDx>(tmA, tmAlo, tmWt, p2, dp, stream)) != RL_OK) return rc;
        }
        EpiDw::Params wp{V, static_cast<int32_t>(H), (c0 > 0 || accumulate) ? 1 : 0, dW};
        const GemmPlan p3 = make_plan_auto(V, H, n, passes, 1 << 30, 0, status);
        {
            ProfScope ps(RL_PROF_GEMM_DW, stream);
            if ((rc = launch_gemm_auto<EpiDw>(tmAt, tmAtlo, tmXt, p3, wp, stream)) != RL_OK) return rc;
        }
        count_launch(2);
    }
    if ((rc = sparse_dw(sa, w, dW, stream)) != RL_OK) return rc;
    if (out->metrics)
        return metrics_run(b, saved, out->metrics, f.fw.mpart, stream, w.split ? nullptr : f.flags,
                           w.split ? 0 : static_cast<int>(f.nchunks));
    return RL_OK;
}

}  // namespace rl
