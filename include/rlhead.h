/*
 * rlhead.h -- C ABI of the GB300 (sm_103a) fused LM head + unified RL loss library.
 *
 * The operation (prime-rl pull request #4233, the loss_t equation and "What changes"):
 * for every RL token t with hidden row h_t, logits z_t = W h_t / T over the whole
 * vocabulary, and a ragged sampler support S_t (CSR row: int32 ids, sampler log q),
 *
 *   loss_t = -adv_tau * A_t * ( w(a_t) log P_t(a_t) - sum_{e in S_t} sg[u_e w_e] log P_t(v_e) )
 *            + beta_t * KL_t(q || P_t)
 *
 *   w:  ipo       1(|P - q| <= eps) * min(P/q, max_importance_ratio)
 *       icepop    1(low <= P/q <= high) * P/q
 *       reinforce 1
 *   u:  q_e on a replayed (truncated top-p / top-k) support; 1/K on K i.i.d. sampler draws
 *   P:  the trainer softmax at temperature T; on a replayed support the softmax
 *       renormalised over S_t (the trainer distribution under the replayed truncation)
 *   KL: exact = sum_e u_e (log q_e - log P(v_e));  k1 = log q(a) - log P(a)
 *   beta_t = kl_coeff * (1, or 1/sqrt(1 + age_t) for inv_sqrt staleness)
 *
 * The [N, V] logits are never materialised: the forward streams vocabulary tiles through
 * tcgen05 tensor-core tiles with an online logsumexp.  The backward is dense
 * (softmax-gradient GEMMs for dX and dW) or sparse (a deterministic CSR matmul) when every
 * logit gradient lies on the label and the support ("Sparse LM-head backward").
 *
 * Conventions for every entry point:
 *   - Pointers marked "device" point to GPU global memory of the current CUDA device;
 *     "host" pointers to CPU memory.  The caller allocates and owns every buffer,
 *     including workspaces and the forward->backward saved state; the library never
 *     allocates and never synchronises the host (except rl_status_read).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  All work is enqueued
 *     on it in order.
 *   - Return value: RL_OK, or an RL_ERR_* code for errors visible on the host (bad
 *     argument, workspace too small, unsupported shape, CUDA launch failure).  When an
 *     error is returned nothing was enqueued, except for RL_ERR_CUDA.
 *   - Data errors found on the device (a corrupt CSR, an out-of-range id, a wait that
 *     ran out) are OR-ed into *dev_status as RL_STATUS_* bits; kernels never trap.
 *     Read them with rl_status_read after the stream is synchronised ("checked once per
 *     step before the optimizer", pull request #4233, GPU sampler-evidence validation).
 *     The library never clears *dev_status; the caller zeroes it.
 *   - Same inputs, same device => bitwise-identical outputs (no float atomics; fixed
 *     reduction orders).
 *   - Layouts are dense row-major; bf16 is IEEE bfloat16 (2 bytes).
 */
#ifndef RLHEAD_H
#define RLHEAD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- host return codes ---------------------------------------------------------- */
#define RL_OK               0
#define RL_ERR_ARG          1   /* null pointer, negative size, bad enum or knob        */
#define RL_ERR_WORKSPACE    2   /* ws_bytes smaller than the matching *_workspace_bytes */
#define RL_ERR_UNSUPPORTED  3   /* H % 64 != 0, V % 8 != 0, or no sm_100-family device  */
#define RL_ERR_CUDA         4   /* a CUDA call or kernel launch failed                   */

/* ---- device status bits (OR-ed into *dev_status) -------------------------------- */
#define RL_STATUS_OFFSETS            0x0001  /* offsets[0]!=0, decreasing, or offsets[N]!=nnz */
#define RL_STATUS_ID_RANGE           0x0002  /* a support id or label outside [0, V)          */
#define RL_STATUS_LOGQ               0x0004  /* a log q not finite or > 1e-6                  */
#define RL_STATUS_LABEL_MISSING      0x0008  /* replayed row does not contain its label      */
#define RL_STATUS_SUPPORT_MASS       0x0010  /* replayed row: |sum exp(log q) - 1| > 1e-3     */
#define RL_STATUS_EMPTY_ROW          0x0020  /* an RL token with an empty support row        */
#define RL_STATUS_ROW_ORDER          0x0040  /* ids not ascending (strictly, when replayed)  */
#define RL_STATUS_SPARSE_INELIGIBLE  0x0080  /* sparse backward asked for, but a token's
                                                gradient has a dense softmax part            */
#define RL_STATUS_NONFINITE          0x0100  /* a non-finite loss or logsumexp               */
#define RL_STATUS_TIMEOUT            0x0200  /* a kernel's bounded wait ran out; outputs invalid */

/* ---- knobs ---------------------------------------------------------------------- */
typedef enum { RL_LOSS_IPO = 0, RL_LOSS_ICEPOP = 1, RL_LOSS_REINFORCE = 2 } rl_loss_type;
typedef enum { RL_KL_EXACT = 0, RL_KL_K1 = 1 } rl_kl_estimator;
typedef enum { RL_STALE_NONE = 0, RL_STALE_INV_SQRT = 1 } rl_kl_staleness;
/* AUTO = SPARSE when the knobs alone make every gradient lie on label + support
 * (reinforce with kl_coeff == 0) or the caller asserts all_replayed; DENSE otherwise. */
typedef enum { RL_BWD_AUTO = 0, RL_BWD_DENSE = 1, RL_BWD_SPARSE = 2 } rl_bwd_mode;
/* Precision of the softmax-gradient operand G fed to the dX / dW tensor-core GEMMs:
 * BF16 rounds G once to bf16; SPLIT feeds G as bf16 hi + bf16 lo (two GEMM passes),
 * which carries ~16 significant bits. */
typedef enum { RL_GRAD_BF16 = 0, RL_GRAD_SPLIT = 1 } rl_grad_precision;

typedef struct rl_params {
    int32_t loss_type;            /* rl_loss_type */
    int32_t kl_estimator;         /* rl_kl_estimator */
    int32_t kl_staleness;         /* rl_kl_staleness */
    int32_t bwd_mode;             /* rl_bwd_mode */
    int32_t grad_precision;       /* rl_grad_precision */
    int32_t all_replayed;         /* caller's assertion that every row is replayed (AUTO) */
    float eps;                    /* ipo band half-width in probability (>= 0); default 0.3 */
    float max_importance_ratio;   /* ipo ratio cap (> 0); default 10 */
    float icepop_low;             /* icepop band, 0 <= low <= high */
    float icepop_high;
    float adv_tau;                /* advantage scale */
    float temperature;            /* T > 0; logits are (W h) / T */
    float kl_coeff;               /* >= 0; default 0 */
    int32_t token_chunk;          /* backward token chunk (multiple of 128); 0 = library default
                                     (rl_head_token_chunk: the first multiple of the GEMM row tile
                                     at or above 8192 at which the dX GEMM fills whole waves of
                                     the device, 9728 with H = 2048 on 152 SMs): memory held grows
                                     with it (about chunk x V x 4 bytes for the bf16 softmax
                                     numerators of the fused call) */
    float entropy_coeff;          /* >= 0; default 0.  "10-KL-clip-entropy", section 3: the
                                     exploration regulariser, loss_t -= entropy_coeff * H_t with
                                     H_t the full-vocabulary token entropy; its gradient is dense
                                     over the vocabulary, so a nonzero value rules out the sparse
                                     backward (RL_BWD_SPARSE then returns RL_ERR_ARG) and makes
                                     the fused BF16 backward recompute the logits (8 N H V) */
    int32_t keep_e;               /* 1: rl_head_loss_fwd keeps the bf16 softmax numerators
                                     e = exp(z - z_label) of every token, in both layouts (2 N V
                                     bf16 values), in the saved state, and rl_head_loss_bwd runs
                                     the fused call's backward on them: 6 N H V of tensor work for
                                     the two calls instead of 8 (no logit recompute), the same
                                     bits as rl_head_loss_fwd_bwd.  The saved state is then
                                     rl_head_saved_bytes_ex bytes, and one backward consumes it
                                     (it folds the gradient's spikes into the kept values).
                                     Takes effect with a dense backward, BF16 gradients and no
                                     entropy term; ignored otherwise.  Default 0. */
} rl_params;

/* Ragged per-token sampler support, CSR over tokens ("TokenSupport", pull request #4233,
 * "What changes": int32 ids, int64 offsets, replayed flag, sampler logprobs).
 * Row t holds entries [offsets[t], offsets[t+1]); ids ascending within a row (strictly
 * ascending when replayed; repeated draws adjacent otherwise). */
typedef struct rl_support {
    const int64_t* offsets;   /* device [N+1] */
    const int32_t* ids;       /* device [nnz] */
    const float*   logq;      /* device [nnz] sampler log q of each entry (renormalised over
                                 S on a replayed row) */
    const uint8_t* replayed;  /* device [N]; 1 = truncated support replayed with u = q */
    int64_t nnz;
} rl_support;

typedef struct rl_head_batch {
    const void* hidden;       /* device [N, H] bf16 */
    const void* weight;       /* device [V, H] bf16 (LM-head rows) */
    int64_t N, H, V;
    const int32_t* labels;    /* device [N] sampled token a_t */
    const float* label_logq;  /* device [N] sampler log q(a_t) */
    const float* adv;         /* device [N] advantage A_t */
    const uint8_t* loss_mask; /* device [N] 1 = RL token; NULL = every token is an RL token */
    const int32_t* age;       /* device [N] policy age for kl_staleness; NULL = all 0 */
    rl_support support;
} rl_head_batch;

/* Metric sums over RL tokens (pull request #4233, metrics item: support_mass = E_q[p/q],
 * mask_tv, kl, kl/beta, kl/age0; "IPO ...": mismatch_kl).  Divide by the counts on the
 * host; sums compose across micro-batches. */
typedef struct rl_head_metrics {
    double loss;          /* sum_t loss_t */
    double mismatch_kl;   /* sum_t (log q(a) - log P(a)) */
    double support_mass;  /* sum_t sum_e u_e exp(log p_full(v_e) - log q_e) */
    double mask_tv;       /* sum_t sum_e u_e (1 - m_e) P(v_e)/q_e */
    double kl;            /* sum_t KL_t */
    double beta;          /* sum_t beta_t */
    double kl_age0;       /* sum of KL_t over age_t == 0 */
    double entropy;       /* sum_t H(p_t) (full-vocab trainer entropy) */
    int64_t n_rl;         /* RL tokens */
    int64_t masked;       /* RL tokens whose label weight was masked */
    int64_t masked_low;   /* ... with P below the band (ipo: P < q - eps; icepop: r < low) */
    int64_t masked_high;  /* ... with P above the band */
    int64_t n_age0;       /* RL tokens with age 0 */
    int64_t recomputed_chunks; /* rl_head_loss_fwd_bwd, bf16 gradients: token chunks whose dense
                                  backward recomputed the logits because a row's stored softmax
                                  numerators left their range (0 elsewhere) */
} rl_head_metrics;

typedef struct rl_head_outputs {
    float*   loss;          /* device [N] per-token loss (0 for non-RL tokens); required */
    float*   logp_label;    /* device [N] log P(a_t); NULL to skip */
    float*   logp_support;  /* device [nnz] log P(v_e); NULL to skip */
    float*   entropy;       /* device [N] full-vocab entropy of p_t; NULL to skip */
    float*   lse;           /* device [N] logsumexp_v z_tv; NULL to skip */
    uint8_t* mask_label;    /* device [N] keep bit of the label weight; NULL to skip */
    uint8_t* mask_support;  /* device [nnz] keep bit of each entry weight; NULL to skip */
    rl_head_metrics* metrics; /* device, one struct, overwritten; NULL to skip */
} rl_head_outputs;

/* Bytes of the caller-owned state the forward saves for the backward. */
size_t rl_head_saved_bytes(int64_t N, int64_t nnz);
/* The token chunk the backward and the fused call use for these sizes and params on the
 * current device (params->token_chunk if set; see rl_params.token_chunk). */
int64_t rl_head_token_chunk(int64_t N, int64_t H, const rl_params* params);
/* Saved-state bytes for these params: rl_head_saved_bytes, plus with keep_e in effect the
 * kept numerators (e [N, V] and e^T [V, N rounded up to 128] bf16), a reference logit per
 * token and a flag per token chunk. */
size_t rl_head_saved_bytes_ex(int64_t N, int64_t nnz, int64_t V, const rl_params* params);
/* Workspace bytes of rl_head_loss_fwd / rl_head_loss_bwd for these sizes and knobs. */
size_t rl_head_fwd_workspace_bytes(int64_t N, int64_t H, int64_t V, int64_t nnz,
                                   const rl_params* params);
size_t rl_head_bwd_workspace_bytes(int64_t N, int64_t H, int64_t V, int64_t nnz,
                                   const rl_params* params);

/* Validate the CSR sampler evidence on the device (pull request #4233, GPU validation of
 * the sampler evidence): sets RL_STATUS_OFFSETS / ID_RANGE / LOGQ / LABEL_MISSING /
 * SUPPORT_MASS / EMPTY_ROW / ROW_ORDER bits.  rl_head_loss_fwd runs it first. */
int rl_validate_support(const rl_head_batch* batch, int32_t* dev_status, void* stream);

/* Forward: per-token loss, label / support log-probs, entropy, masks, metrics, and the
 * saved state (`saved`, device, rl_head_saved_bytes_ex: rl_head_saved_bytes unless keep_e) for
 * the backward. */
int rl_head_loss_fwd(const rl_head_batch* batch, const rl_params* params,
                     const rl_head_outputs* out, void* saved, void* ws, size_t ws_bytes,
                     int32_t* dev_status, void* stream);

/* Backward of sum_t dloss[t] * loss_t.  dloss: device [N] fp32 (the caller's aggregation,
 * e.g. 1 / #RL tokens for a token mean).  dhidden: device [N, H] bf16, overwritten.
 * dW: device [V, H] fp32; accumulate_dW != 0 adds into it, else it is overwritten.
 * params must be the forward's.  With keep_e in effect it runs on the numerators the
 * forward kept (no logit recompute) and leaves them changed: call it once per forward. */
int rl_head_loss_bwd(const rl_head_batch* batch, const rl_params* params, const void* saved,
                     const float* dloss, void* dhidden, float* dW, int accumulate_dW,
                     void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* Forward and backward in one call, for callers whose loss aggregation is known before
 * the forward (dloss_t = the weight of loss_t in the scalar objective, e.g. 1 / #RL tokens
 * for a token mean; an autograd caller then scales dhidden and dW by the upstream
 * gradient of that scalar).  Same outputs as rl_head_loss_fwd (incl. `saved`, usable by a
 * later rl_head_loss_bwd) plus the gradients of rl_head_loss_bwd, without recomputing
 * the logits: per token chunk the forward tiles keep the softmax numerators (fp16,
 * relative to the running row max) and the dense backward consumes them.  Dense-mode
 * tensor work is 6 N H V flops instead of 8.  Sparse-mode knobs run the forward and
 * the sparse backward.  Workspace: rl_head_fwd_bwd_workspace_bytes. */
size_t rl_head_fwd_bwd_workspace_bytes(int64_t N, int64_t H, int64_t V, int64_t nnz,
                                       const rl_params* params);
int rl_head_loss_fwd_bwd(const rl_head_batch* batch, const rl_params* params,
                         const rl_head_outputs* out, const float* dloss, void* dhidden, float* dW,
                         int accumulate_dW, void* saved, void* ws, size_t ws_bytes,
                         int32_t* dev_status, void* stream);

/* ---- the head split by vocabulary across ranks ---------------------------------------
 * Each of R ranks holds a contiguous range [vocab_begin, vocab_end) of W's rows (pull request
 * #4233, "What changes": the support is sharded with the head); every rank holds the whole
 * batch.  Per step (lm_head_gb300/vocab_parallel.py drives it with torch.distributed):
 *   forward   1. rl_head_shard_remap: the labels' and support ids' local numbering;
 *             2. rl_head_shard_stats on the rank's rows: per token the logsumexp statistics
 *                over its columns (m = max z, s = sum e^(z - m), u = sum e^(z - m)(z - m))
 *                and the label / support logits it owns (0 for the others);
 *             3. all-gather of the statistics (rank order), all-reduce (sum) of the owned
 *                logits: every logit is nonzero on exactly its owner;
 *             4. rl_head_loss_from_shard_stats on every rank: the loss, log-probs, masks,
 *                metrics and saved state, combining the R statistics as the single-GPU
 *                forward combines its vocabulary splits (the same bits on every rank).
 *   backward  rl_head_loss_bwd on the rank's rows with the local ids and the saved state of
 *             step 4: dW of its rows, and its part of dX (bf16), which the ranks all-reduce.
 * keep_e does not apply: rl_head_shard_stats and rl_head_loss_from_shard_stats return
 * RL_ERR_ARG when it would take effect (their saved state holds no numerators).
 * Unmeasured on hardware with more than one GPU: one process here emulates the ranks. */

/* ids_local[i] = ids[i] - vocab_begin for an id inside [vocab_begin, vocab_end), -1 below
 * the range, vocab_end - vocab_begin above it (a row stays in ascending order; an id the
 * shard does not own matches none of its columns).  Device arrays of n int32. */
int rl_head_shard_remap(const int32_t* ids, int64_t n, int64_t vocab_begin, int64_t vocab_end, int32_t* ids_local,
                        void* stream);
/* shard: the batch with weight = the rank's rows of W (V = their count) and labels / support
 * ids in local numbering (rl_head_shard_remap); params: temperature only.  Outputs, device:
 * stats [3][N] fp32 (m, then s, then u, per token over the shard's columns), zlab [N] and
 * zsup [nnz] fp32 (the logits / T of the labels and entries the shard owns, 0 elsewhere).
 * Workspace: rl_head_fwd_workspace_bytes(N, H, V_shard, nnz).  No validation here. */
int rl_head_shard_stats(const rl_head_batch* shard, const rl_params* params, float* stats, float* zlab, float* zsup,
                        void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);
/* batch: the whole batch in global numbering (weight unused, may be NULL; V the full
 * vocabulary); stats_all [n_shards][3][N]: the shards' statistics in rank order; zlab, zsup:
 * the owned logits summed over the ranks.  Outputs and saved state as rl_head_loss_fwd
 * (validation included); workspace rl_head_fwd_workspace_bytes(N, H, V, nnz). */
int rl_head_loss_from_shard_stats(const rl_head_batch* batch, const rl_params* params, int32_t n_shards,
                                  const float* stats_all, const float* zlab, const float* zsup,
                                  const rl_head_outputs* out, void* saved, void* ws, size_t ws_bytes,
                                  int32_t* dev_status, void* stream);

/* Reduce the per-token metric terms in `saved` (written by rl_head_loss_fwd for the same
 * batch) into *metrics (device).  rl_head_loss_fwd calls it when out->metrics != NULL. */
int rl_mismatch_metrics(const rl_head_batch* batch, const void* saved,
                        rl_head_metrics* metrics, void* ws, size_t ws_bytes, void* stream);

/* ---- elementwise PPO / decoupled-TIS / mismatch path --------------------------------
 * "Rollout Correction Methods", "Algorithms" (standard, bypass and decoupled 3-policy PPO)
 * and "Mismatch Metrics"; "10-KL-clip-entropy", section 2 (clip, dual clip, metrics);
 * "IPO (INTELLECT Policy Optimization)", "Choosing eps" (masked fraction vs eps).
 * Per token i with r = exp(lp_theta - lp_old):
 *   l1 = -A r, l2 = -A clip(r, 1 - clip_ratio_low, 1 + clip_ratio_high), lc = max(l1, l2)
 *   loss_ppo = A < 0 ? min(lc, -A clip_ratio_c) : lc          (dual clip)
 *   loss_dec = min(exp(lp_old - lp_samp), tis_upper) * lc      (decoupled, TIS truncate)
 *   grad_*   = d loss_* / d lp_theta
 * Bypass PPO is the same call with lp_old := lp_samp. */
#define RL_PG_MAX_CURVE 16
typedef struct rl_pg_params {
    float clip_ratio_low, clip_ratio_high, clip_ratio_c;  /* defaults 0.2, 0.2, 3.0 */
    float tis_upper;                                      /* TIS truncation bound */
    float icepop_low, icepop_high;                        /* ratio band for the IcePop count */
    int32_t n_curve;                                      /* 0..RL_PG_MAX_CURVE */
    float curve_eps[RL_PG_MAX_CURVE];                     /* IPO eps values */
} rl_pg_params;

typedef struct rl_pg_metrics {
    double loss_ppo, loss_dec;   /* sums over valid tokens */
    double ppo_kl;               /* sum (lp_old - lp_theta) */
    double mis_kl;               /* sum (lp_samp - lp_old) */
    double k3;                   /* sum (e^d - d - 1), d = lp_old - lp_samp */
    double tis_sum;              /* sum of truncated TIS weights */
    int64_t n_valid, n_clip, n_clip_lower, icepop_low, icepop_high, n_tis_trunc;
    int64_t ipo_curve[RL_PG_MAX_CURVE];   /* count of |e^lp_old - e^lp_samp| > curve_eps[k] */
    int64_t status;              /* RL_STATUS_* bits: RL_STATUS_TIMEOUT if a wait for a copy ran
                                    out (the outputs and metrics are then incomplete) */
} rl_pg_metrics;

/* Workspace bytes for T tokens: 4096 (an arrival counter, a status word, a range flag, a
 * stage-claim counter and the batch's metric accumulators, one 128-byte line each; the
 * workspace 8-byte aligned), for any T and device.  The argument stays so that callers
 * need not change if a later layout depends on T.  Zero the workspace once before its
 * first use (a cudaMemset when it is allocated): every call is one kernel launch whose
 * last block sets all of it back to zero, so later calls need no clearing.  Calls that
 * overlap on the GPU must not share a workspace. */
size_t rl_policy_workspace_bytes(int64_t T);
/* All arrays device [T] fp32 (mask uint8, 1 = valid response token; any nonzero byte
 * counts as valid).  A masked slot's inputs are never used, whatever they hold (NaN and
 * inf included).  mask == NULL: packed input, every one of the T slots is a valid token
 * (the response tokens of a batch laid end to end, as for the sequences' cumulative
 * lengths; nothing is read for the mask).  Output arrays may be NULL to skip; masked
 * tokens get 0.  metrics: device, overwritten; NULL to skip. */
int rl_policy_loss_elementwise(const float* lp_theta, const float* lp_old, const float* lp_samp,
                               const float* adv, const uint8_t* mask, int64_t T,
                               const rl_pg_params* params, float* loss_ppo, float* loss_dec,
                               float* grad_ppo, float* grad_dec, rl_pg_metrics* metrics,
                               void* ws, size_t ws_bytes, void* stream);

/* The same computation as rl_policy_loss_elementwise, for callers that cannot allocate
 * device memory.  The pages have no counterpart of this entry point.  Some callers hold
 * only their input and output buffers: for example a metrics or loss hook inside a
 * trainer or inference engine whose device memory is reserved up front by its own pool,
 * where an extra cudaMalloc would fail or compete with that pool, or plain C code with
 * no device allocator at hand.  This variant takes no workspace and allocates nothing:
 * its scratch (the counters, flags and metric accumulators) is a file-scope device
 * array of 4096 bytes, the size rl_policy_workspace_bytes returns.
 *   - Every GPU that loads the library holds that array until the process exits.
 *   - The first call on a device looks the array's device address up (once per
 *     device); make that first call before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents.  The array
 *     starts at zero when the library is loaded; every block of a call adds its partial
 *     before the last block reads the totals, and that last block sets the whole array
 *     back to zero, so each call leaves the array ready for the next.  Calls one after
 *     another on one stream are therefore safe; calls that overlap on the GPU (other
 *     streams, other threads) race on the array: serialise them.
 * Arguments, outputs and errors as rl_policy_loss_elementwise, without ws / ws_bytes. */
int rl_policy_loss_elementwise_noalloc(const float* lp_theta, const float* lp_old,
                                       const float* lp_samp, const float* adv,
                                       const uint8_t* mask, int64_t T,
                                       const rl_pg_params* params, float* loss_ppo,
                                       float* loss_dec, float* grad_ppo, float* grad_dec,
                                       rl_pg_metrics* metrics, void* stream);

/* ---- rollout correction: IS / RS weights and mismatch metrics over sequences -------
 * "Rollout Correction Methods": "Config keys", "Importance Sampling", "Rejection
 * Sampling" (with the veto) and "Mismatch Metrics".  Per response token i of sequence s,
 * d_i = lp_train_i - lp_rollout_i (lp_train: the trainer's log-probs, pi_old; lp_rollout:
 * the inference engine's):
 *   IS weight  w_i = exp(d_i) (token) | exp(sum_s d) (sequence) | exp(mean_s d) (geometric)
 *   bounding   truncate: min(w, U); clip: clamp(w, L, U); mask: w if L <= w <= U else 0
 *   RS         reject token i if exp(d_i) is outside [rL, rU] (token), or all of s if its
 *              mean token weight (sequence) / geometric-mean weight (geometric) is
 *   veto       reject all of s if some exp(d_i) < veto (whatever use_tis / use_rs say)
 *   keep_i     = response token, not rejected; weights_i = w'_i * factor on kept tokens,
 *              0 elsewhere; factor = 1, or (batch normalisation) n_kept / sum_kept w'.
 * A weight equal to a bound is inside it.  Every decision (bounds, RS, veto) is the exact
 * predicate on the fp32 inputs (the log-ratio sums carried in float-float); weight values
 * are fp32 (a raw sequence weight past the fp32 range is inf, its bounded value exact).
 * The metric struct holds sums and counts (they compose across calls); the named
 * metrics of "Mismatch Metrics" come from them through rl_rollout_metrics_named. */
typedef enum { RL_TIS_TRUNCATE = 0, RL_TIS_CLIP = 1, RL_TIS_MASK = 2 } rl_tis_mode;
typedef enum { RL_LEVEL_TOKEN = 0, RL_LEVEL_SEQUENCE = 1, RL_LEVEL_GEOMETRIC = 2 } rl_is_level;
typedef struct rl_rc_params {
    int32_t use_tis;                  /* 0: weights 1 on kept tokens (RS, veto, metrics only) */
    int32_t tis_mode;                 /* rl_tis_mode */
    int32_t tis_level;                /* rl_is_level */
    int32_t tis_batch_normalize;      /* 1: kept weights scaled to mean 1 */
    float tis_lower_bound, tis_upper_bound;   /* L, U; 0 <= L <= U */
    int32_t use_rs;
    int32_t rs_level;                 /* rl_is_level */
    float rs_lower_bound, rs_upper_bound;     /* NaN: the tis bound */
    float rs_veto_threshold;          /* <= 0 or NaN: no veto */
} rl_rc_params;

typedef struct rl_rc_metrics {
    /* IS / RS (sums over response tokens unless noted) */
    double w_before_sum;        /* raw IS weights at tis_level */
    double w_after_sum;         /* bounded weights */
    double kept_w_sum;          /* bounded weights of kept tokens */
    double batch_norm_factor;   /* factor (1 when off) */
    double final_sum, final_min, final_max;   /* final weights of kept tokens */
    /* mismatch monitoring */
    double mis_kl_sum;          /* sum (lp_rollout - lp_train) */
    double k3_sum;              /* sum (e^d - d - 1) */
    double abs_diff_sum;        /* sum |d| */
    double chi2_token_sum;      /* sum e^(2d) */
    double train_lppl_sum;      /* over sequences: -mean_s lp_train */
    double rollout_lppl_sum;    /* over sequences: -mean_s lp_rollout */
    double lppl_diff_sum;       /* over sequences: train - rollout log-ppl */
    double lppl_abs_diff_sum;   /* over sequences: |train - rollout log-ppl| */
    double ppl_ratio_sum;       /* over sequences: exp(train - rollout log-ppl) */
    double chi2_seq_sum;        /* over sequences: exp(2 sum_s d) */
    int64_t n_valid;            /* response tokens */
    int64_t n_seq;              /* sequences with at least one response token */
    int64_t n_kept;             /* kept tokens */
    int64_t n_tis_low, n_tis_high;     /* response tokens with raw weight < L / > U */
    int64_t n_rs_low, n_rs_high;       /* response tokens rejected by RS below / above */
    int64_t n_cat_tokens;       /* response tokens with exp(d) < veto */
    int64_t n_cat_seqs;         /* sequences holding one */
    int64_t status;             /* RL_STATUS_OFFSETS if seq_offsets was not a partition of
                                   [0, T) (bad sequences then count as empty) */
} rl_rc_metrics;

/* Workspace bytes for B sequences: a small header (counters, status, factor), per-sequence
 * and per-group partial sums, per-group counters.  Zero the workspace once before its first
 * use (8-byte aligned): every call leaves its counters and status word at zero again, so
 * later calls need no clearing.  Calls that overlap on the GPU must not share a workspace. */
size_t rl_rollout_correction_workspace_bytes(int64_t B);
/* lp_train, lp_rollout: device [T] fp32; mask: device [T] uint8 (1 = response token);
 * seq_offsets: device [B + 1] int64, sequence s = tokens [seq_offsets[s], seq_offsets[s+1])
 * (padded rows: s * row_length; packed: cumulative lengths).  A token whose mask byte is 0
 * is not a response token and its log-probs are never used (NaN and inf included).
 * Outputs, device: weights [T] fp32 and keep [T] uint8 (either may be NULL), metrics
 * (overwritten, may be NULL).  Sums: per sequence in fp32 (fp64 for the sequence-level
 * terms), then over the sequences in fp64 in a fixed order (groups of 32 in sequence order,
 * then the groups in order), so results are reproducible; the batch-normalisation factor
 * n_kept / (sum of kept weights) comes from those totals.
 * Errors: RL_ERR_ARG (NULL input, B < 0, T < 0, B == 0 with T > 0, bad enum, L > U or
 * negative bound), RL_ERR_WORKSPACE; bad offsets are reported in metrics->status, not
 * trapped. */
int rl_rollout_correction(const float* lp_train, const float* lp_rollout, const uint8_t* mask,
                          const int64_t* seq_offsets, int64_t B, int64_t T,
                          const rl_rc_params* params, float* weights, uint8_t* keep,
                          rl_rc_metrics* metrics, void* ws, size_t ws_bytes, void* stream);

/* The named metrics of "Rollout Correction Methods", "Mismatch Metrics" (the "Mismatch
 * Monitoring Metrics" and "IS/RS Correction Metrics" tables), under the names the page
 * logs them by without the mis_ prefix.  Readings where the page names a metric without
 * a formula:
 *   - a mean E[.] is over response tokens; the log-perplexities are per sequence (mean of
 *     -log pi over its response tokens) averaged over the sequences holding one; the
 *     perplexity is exp of that average; the log-perplexity difference (training minus
 *     rollout), its absolute value and the perplexity ratio exp(difference) are taken per
 *     sequence and averaged over sequences;
 *   - chi^2 of the two policies, estimated under the rollout policy, is E[w^2] - 1 with
 *     w = exp(lp_train - lp_rollout) per token (token) or exp of the sequence's summed
 *     log-ratio (sequence, averaged over sequences);
 *   - the fractions count response tokens (catastrophic sequences: sequences);
 *   - is_ratio_mean_after_tis_rs and the final mean / min / max are over kept tokens.
 * A mean over an empty set is 0 (a perplexity over no sequence is exp(0) = 1).  A metric
 * the page emits only under some settings ("Emitted when": use_tis for the IS/RS weight
 * statistics, the tis_mode for its fractions, use_rs, a set veto threshold) is NaN when
 * the settings given here do not emit it. */
typedef struct rl_rc_named {
    /* Mismatch Monitoring Metrics (always emitted) */
    double training_log_ppl, training_ppl, rollout_log_ppl, rollout_ppl;
    double kl;                  /* E[lp_rollout - lp_train] */
    double k3_kl;               /* E[e^d - d - 1], d = lp_train - lp_rollout */
    double log_ppl_diff, log_ppl_abs_diff, ppl_ratio;
    double chi2_token, chi2_seq;
    double train_rollout_logprob_abs_diff;   /* E|d| */
    /* IS/RS Correction Metrics */
    double tis_weight_before_bound, tis_weight_after_bound;      /* use_tis: token means */
    double tis_truncate_fraction;                                /* use_tis, truncate */
    double tis_clip_fraction_low, tis_clip_fraction_high;        /* use_tis, clip */
    double tis_mask_fraction_low, tis_mask_fraction_high;        /* use_tis, mask */
    double rs_mask_fraction_low, rs_mask_fraction_high;          /* use_rs */
    double rs_catastrophic_token_fraction, rs_catastrophic_seq_fraction;   /* veto set */
    double is_ratio_mean_after_tis_rs, batch_norm_factor;        /* use_tis */
    double is_ratio_mean_final, is_ratio_min_final, is_ratio_max_final;    /* use_tis */
} rl_rc_named;

/* metrics: device, as rl_rollout_correction wrote it (or sums the caller added up over
 * several calls, with the min / max / factor fields of one of them); params: host, the
 * settings of those calls; named: device, overwritten.  One device thread, enqueued on
 * `stream` after the call that wrote `metrics`.  Errors: RL_ERR_ARG (NULL pointer, bad
 * enum). */
int rl_rollout_metrics_named(const rl_rc_metrics* metrics, const rl_rc_params* params,
                             rl_rc_named* named, void* stream);

/* ---- utilities ------------------------------------------------------------------ */
/* The head contraction alone: D[M, N] fp32 = A[M, K] * B[N, K]^T, A and B bf16 row-major
 * (K contiguous), device pointers, 16-byte aligned; K % 8 == 0, N % 4 == 0.  Same tcgen05
 * tensor-core pipeline as rl_head_loss_fwd with a plain store epilogue; for unit tests and
 * for timing the contraction in isolation.  Status bits: RL_STATUS_TIMEOUT only. */
int rl_gemm_bf16_tn(const void* A, const void* B, int64_t M, int64_t N, int64_t K, float* D,
                    int32_t* dev_status, void* stream);
/* General layouts of the same contraction: A is [M, K] (a_mn_major = 0) or [K, M]
 * (a_mn_major = 1), B is [N, K] or [K, N]; the contiguous extent of each operand must be a
 * multiple of 8; N % 4 == 0.  D[M, N] fp32 = A * B^T in the K-major naming. */
int rl_gemm_bf16(const void* A, int a_mn_major, const void* B, int b_mn_major, int64_t M, int64_t N,
                 int64_t K, float* D, int32_t* dev_status, void* stream);

/* Per-kernel timing: when enabled, the library records a CUDA event pair on the caller's
 * stream around each of its kernel launches, grouped by kind (RL_PROF_* below).
 * rl_profile_enable(1) also clears the counters.  rl_profile_read waits for the recorded
 * events, then fills ms[k] (summed device milliseconds) and launches[k] for every kind
 * k < RL_PROF_KINDS; either pointer may be NULL.  Host arrays. */
#define RL_PROF_KINDS 18
enum { RL_PROF_VALIDATE = 0, RL_PROF_GEMM_FWD = 1, RL_PROF_TOKEN_LOSS = 2, RL_PROF_METRICS = 3,
       RL_PROF_TRANSPOSE = 4, RL_PROF_GEMM_GRAD = 5, RL_PROF_GEMM_DX = 6, RL_PROF_GEMM_DW = 7,
       RL_PROF_SPARSE_DX = 8, RL_PROF_SPARSE_DW = 9, RL_PROF_POLICY = 10, RL_PROF_GEMM_UTIL = 11,
       RL_PROF_MEMSET = 12, RL_PROF_OTHER = 13, RL_PROF_RESID = 14, RL_PROF_GRAD_E = 15,
       RL_PROF_REF_LOGIT = 16, RL_PROF_ROLLOUT = 17 };
int rl_profile_enable(int on);
int rl_profile_read(double* ms, int64_t* launches);
const char* rl_profile_kind_name(int kind);

/* Library options (process-wide, host side, read when a call enqueues its kernels).
 *   RL_OPT_GEMM_PAIR: 1 (the default) runs the tensor-core GEMMs on pairs of SMs (two-CTA
 *     clusters, tcgen05 cta_group::2, 256 x 256 tiles); 0 on single SMs (128 x 256 tiles).
 *     Results are the same to fp32 rounding.
 *   RL_OPT_WAIT_LIMIT_US: how long (microseconds, 1 .. 10,000,000; default 1,000,000) a
 *     kernel's wait for its own copies or tensor-core work may last before it gives up,
 *     ORs RL_STATUS_TIMEOUT into the status word (rl_pg_metrics.status for the
 *     elementwise path) and unwinds; the outputs of that call are then invalid.  An
 *     unwinding kernel still waits (up to 1 s, whatever this option says) for the copies
 *     and MMAs it has in flight before it releases its shared memory and TMEM, so a short
 *     limit makes a call fail, never fault.  A limit below a few milliseconds is for tests.
 * rl_set_option returns RL_ERR_ARG for an unknown key or a value out of range;
 * rl_get_option returns -1 for an unknown key. */
#define RL_OPT_GEMM_PAIR 1
#define RL_OPT_WAIT_LIMIT_US 2
int rl_set_option(int key, int value);
int rl_get_option(int key);

/* Self-test of the bounded waits: one block waits on a shared-memory mbarrier that nothing
 * ever signals, with the RL_OPT_WAIT_LIMIT_US limit; the wait runs out, ORs
 * RL_STATUS_TIMEOUT into *dev_status (device) and the kernel returns normally, so the
 * context stays usable.  This is the failure path of every wait in the library
 * ("checked once per step before the optimizer": pull request #4233, GPU validation of the
 * sampler evidence, whose device status word this reuses), made to happen on purpose
 * without a fault.  Takes about the limit to run. */
int rl_wait_selftest(int32_t* dev_status, void* stream);

/* Synchronous device->host copy of the status word.  Call after the stream is done. */
int rl_status_read(const int32_t* dev_status, int32_t* host_out);
/* Kernels this library has launched in this process (for launch accounting). */
int64_t rl_kernel_launch_count(void);
/* Static text for an RL_ERR_* code; the last error's detail in rl_last_error(). */
const char* rl_error_string(int code);
const char* rl_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* RLHEAD_H */
