// C ABI of librlhead (declared in include/rlhead.h): host-side argument checks,
// workspace sizing and dispatch to the implementations.  Nothing here allocates device
// memory or synchronises, except rl_status_read.
#include <cmath>
#include <cstring>

#include "internal.h"

using namespace rl;

int64_t rl_launch_counter_value();

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int fail(int code, const char* msg) {
    set_last_error(msg);
    return code;
}

int check_params(const rl_params* p) {
    if (!p) return fail(RL_ERR_ARG, "params is NULL");
    if (p->loss_type < RL_LOSS_IPO || p->loss_type > RL_LOSS_REINFORCE) return fail(RL_ERR_ARG, "bad loss_type");
    if (p->kl_estimator < RL_KL_EXACT || p->kl_estimator > RL_KL_K1) return fail(RL_ERR_ARG, "bad kl_estimator");
    if (p->kl_staleness < RL_STALE_NONE || p->kl_staleness > RL_STALE_INV_SQRT) return fail(RL_ERR_ARG, "bad kl_staleness");
    if (p->bwd_mode < RL_BWD_AUTO || p->bwd_mode > RL_BWD_SPARSE) return fail(RL_ERR_ARG, "bad bwd_mode");
    if (p->grad_precision < RL_GRAD_BF16 || p->grad_precision > RL_GRAD_SPLIT) return fail(RL_ERR_ARG, "bad grad_precision");
    if (!(p->eps >= 0.f) || !(p->max_importance_ratio > 0.f)) return fail(RL_ERR_ARG, "bad eps / max_importance_ratio");
    if (!(p->icepop_low >= 0.f) || !(p->icepop_low <= p->icepop_high)) return fail(RL_ERR_ARG, "bad icepop band");
    if (!(p->temperature > 0.f) || !std::isfinite(p->temperature)) return fail(RL_ERR_ARG, "bad temperature");
    if (!(p->kl_coeff >= 0.f) || !std::isfinite(p->adv_tau)) return fail(RL_ERR_ARG, "bad kl_coeff / adv_tau");
    if (p->token_chunk < 0 || p->token_chunk % 128 != 0) return fail(RL_ERR_ARG, "token_chunk must be a multiple of 128");
    if (!(p->entropy_coeff >= 0.f) || !std::isfinite(p->entropy_coeff)) return fail(RL_ERR_ARG, "bad entropy_coeff");
    if (p->entropy_coeff != 0.f && p->bwd_mode == RL_BWD_SPARSE)
        return fail(RL_ERR_ARG, "the entropy term's gradient is dense: no sparse backward with entropy_coeff > 0");
    if (p->keep_e != 0 && p->keep_e != 1) return fail(RL_ERR_ARG, "keep_e must be 0 or 1");
    return RL_OK;
}

int check_shape(int64_t N, int64_t H, int64_t V, int64_t nnz) {
    if (N < 0 || H <= 0 || V <= 0 || nnz < 0) return fail(RL_ERR_ARG, "negative or zero size");
    if (H % 64 != 0) return fail(RL_ERR_UNSUPPORTED, "H must be a multiple of 64");
    if (V % 8 != 0) return fail(RL_ERR_UNSUPPORTED, "V must be a multiple of 8");
    if (V >= (int64_t(1) << 30) || N >= (int64_t(1) << 31)) return fail(RL_ERR_UNSUPPORTED, "N or V too large");
    return RL_OK;
}

int check_batch(const rl_head_batch* b) {
    if (!b) return fail(RL_ERR_ARG, "batch is NULL");
    int rc = check_shape(b->N, b->H, b->V, b->support.nnz);
    if (rc != RL_OK) return rc;
    if (b->N == 0) return RL_OK;
    if (!b->hidden || !b->weight || !b->labels || !b->label_logq || !b->adv || !b->support.offsets ||
        !b->support.replayed)
        return fail(RL_ERR_ARG, "required batch pointer is NULL");
    if (b->support.nnz > 0 && (!b->support.ids || !b->support.logq))
        return fail(RL_ERR_ARG, "support ids/logq NULL with nnz > 0");
    if (!aligned16(b->hidden) || !aligned16(b->weight)) return fail(RL_ERR_ARG, "hidden/weight not 16-byte aligned");
    return RL_OK;
}

int sm100_family() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    int major = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return 0;
    return major == 10;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

}  // namespace

extern "C" {

size_t rl_head_saved_bytes(int64_t N, int64_t nnz) {
    if (N < 0 || nnz < 0) return 0;
    size_t bytes = 0;
    saved_view(nullptr, N, nnz, &bytes);
    return bytes;
}

int64_t rl_head_token_chunk(int64_t N, int64_t H, const rl_params* params) {
    if (N < 0 || H <= 0 || !params) return 0;
    return bwd_chunk(N, H, params);
}

size_t rl_head_saved_bytes_ex(int64_t N, int64_t nnz, int64_t V, const rl_params* params) {
    if (N < 0 || nnz < 0 || V <= 0 || !params) return 0;
    size_t bytes = 0;
    if (keep_e_active(params))
        kept_view(nullptr, N, nnz, V, params, &bytes);
    else
        saved_view(nullptr, N, nnz, &bytes);
    return bytes;
}

size_t rl_head_fwd_workspace_bytes(int64_t N, int64_t H, int64_t V, int64_t nnz, const rl_params* params) {
    (void)params;
    if (N < 0 || H <= 0 || V <= 0 || nnz < 0) return 0;
    size_t bytes = 0;
    fwd_ws_view(nullptr, N, H, V, nnz, &bytes);
    return bytes;
}

size_t rl_head_bwd_workspace_bytes(int64_t N, int64_t H, int64_t V, int64_t nnz, const rl_params* params) {
    if (N < 0 || H <= 0 || V <= 0 || nnz < 0 || !params) return 0;
    if (keep_e_active(params)) return kept_bwd_ws_bytes(N, H, V, nnz, params);
    size_t bytes = 0;
    bwd_ws_view(nullptr, N, H, V, nnz, params, &bytes);
    return bytes;
}

int rl_validate_support(const rl_head_batch* batch, int32_t* dev_status, void* stream) {
    int rc = check_batch(batch);
    if (rc != RL_OK) return rc;
    if (!dev_status) return fail(RL_ERR_ARG, "dev_status is NULL");
    if (!sm100_family()) return fail(RL_ERR_UNSUPPORTED, "needs an sm_100-family GPU");
    return validate_impl(batch, dev_status, as_stream(stream));
}

int rl_head_loss_fwd(const rl_head_batch* batch, const rl_params* params, const rl_head_outputs* out,
                     void* saved, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
    int rc = check_batch(batch);
    if (rc != RL_OK) return rc;
    if ((rc = check_params(params)) != RL_OK) return rc;
    if (!out || (batch->N > 0 && (!out->loss || !saved)) || !dev_status)
        return fail(RL_ERR_ARG, "out/loss/saved/dev_status NULL");
    if (ws_bytes < rl_head_fwd_workspace_bytes(batch->N, batch->H, batch->V, batch->support.nnz, params))
        return fail(RL_ERR_WORKSPACE, "forward workspace too small");
    if (!ws) return fail(RL_ERR_ARG, "ws is NULL");
    if (!sm100_family()) return fail(RL_ERR_UNSUPPORTED, "needs an sm_100-family GPU");
    return head_fwd_impl(batch, params, out, saved, ws, dev_status, as_stream(stream));
}

int rl_head_loss_bwd(const rl_head_batch* batch, const rl_params* params, const void* saved, const float* dloss,
                     void* dhidden, float* dW, int accumulate_dW, void* ws, size_t ws_bytes, int32_t* dev_status,
                     void* stream) {
    int rc = check_batch(batch);
    if (rc != RL_OK) return rc;
    if ((rc = check_params(params)) != RL_OK) return rc;
    if ((batch->N > 0 && (!saved || !dloss || !dhidden)) || !dW || !dev_status)
        return fail(RL_ERR_ARG, "saved/dloss/dhidden/dW/dev_status NULL");
    if (!aligned16(dW) || !aligned16(dhidden)) return fail(RL_ERR_ARG, "dW/dhidden not 16-byte aligned");
    if (ws_bytes < rl_head_bwd_workspace_bytes(batch->N, batch->H, batch->V, batch->support.nnz, params))
        return fail(RL_ERR_WORKSPACE, "backward workspace too small");
    if (!ws) return fail(RL_ERR_ARG, "ws is NULL");
    if (!sm100_family()) return fail(RL_ERR_UNSUPPORTED, "needs an sm_100-family GPU");
    return head_bwd_impl(batch, params, saved, dloss, dhidden, dW, accumulate_dW, ws, dev_status,
                         as_stream(stream));
}

size_t rl_head_fwd_bwd_workspace_bytes(int64_t N, int64_t H, int64_t V, int64_t nnz, const rl_params* params) {
    if (N < 0 || H <= 0 || V <= 0 || nnz < 0 || !params) return 0;
    return fused_ws_bytes(N, H, V, nnz, params);
}

int rl_head_loss_fwd_bwd(const rl_head_batch* batch, const rl_params* params, const rl_head_outputs* out,
                         const float* dloss, void* dhidden, float* dW, int accumulate_dW, void* saved, void* ws,
                         size_t ws_bytes, int32_t* dev_status, void* stream) {
    int rc = check_batch(batch);
    if (rc != RL_OK) return rc;
    if ((rc = check_params(params)) != RL_OK) return rc;
    const bool any = batch->N > 0;
    if (!out || (any && (!out->loss || !saved || !dloss || !dhidden)) || !dev_status || !dW)
        return fail(RL_ERR_ARG, "out/loss/saved/dev_status/dloss/dhidden/dW NULL");
    if (!aligned16(dW) || !aligned16(dhidden)) return fail(RL_ERR_ARG, "dW/dhidden not 16-byte aligned");
    if (ws_bytes < rl_head_fwd_bwd_workspace_bytes(batch->N, batch->H, batch->V, batch->support.nnz, params))
        return fail(RL_ERR_WORKSPACE, "forward+backward workspace too small");
    if (!ws) return fail(RL_ERR_ARG, "ws is NULL");
    if (!sm100_family()) return fail(RL_ERR_UNSUPPORTED, "needs an sm_100-family GPU");
    return head_fused_impl(batch, params, out, dloss, dhidden, dW, accumulate_dW, saved, ws, dev_status,
                           as_stream(stream));
}

int rl_head_shard_remap(const int32_t* ids, int64_t n, int64_t vocab_begin, int64_t vocab_end, int32_t* ids_local,
                        void* stream) {
    if (n < 0 || vocab_begin < 0 || vocab_end <= vocab_begin || vocab_end >= (int64_t(1) << 30))
        return fail(RL_ERR_ARG, "bad shard range or size");
    if (n > 0 && (!ids || !ids_local)) return fail(RL_ERR_ARG, "ids NULL");
    if (n > 0 && !sm100_family()) return fail(RL_ERR_UNSUPPORTED, "needs an sm_100-family GPU");
    return shard_remap_impl(ids, n, vocab_begin, vocab_end, ids_local, as_stream(stream));
}

int rl_head_shard_stats(const rl_head_batch* shard, const rl_params* params, float* stats, float* zlab, float* zsup,
                        void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
    int rc = check_batch(shard);
    if (rc != RL_OK) return rc;
    if ((rc = check_params(params)) != RL_OK) return rc;
    if (keep_e_active(params)) return fail(RL_ERR_ARG, "keep_e is for the single-GPU forward, not a vocabulary shard");
    if (shard->N > 0 && (!stats || !zlab || (shard->support.nnz > 0 && !zsup))) return fail(RL_ERR_ARG, "output NULL");
    if (!dev_status) return fail(RL_ERR_ARG, "dev_status NULL");
    if (ws_bytes < rl_head_fwd_workspace_bytes(shard->N, shard->H, shard->V, shard->support.nnz, params) || !ws)
        return fail(RL_ERR_WORKSPACE, "shard workspace too small");
    if (!sm100_family()) return fail(RL_ERR_UNSUPPORTED, "needs an sm_100-family GPU");
    return shard_stats_impl(shard, params, stats, zlab, zsup, ws, dev_status, as_stream(stream));
}

int rl_head_loss_from_shard_stats(const rl_head_batch* batch, const rl_params* params, int32_t n_shards,
                                  const float* stats_all, const float* zlab, const float* zsup,
                                  const rl_head_outputs* out, void* saved, void* ws, size_t ws_bytes,
                                  int32_t* dev_status, void* stream) {
    if (!batch) return fail(RL_ERR_ARG, "batch is NULL");
    int rc = check_shape(batch->N, batch->H, batch->V, batch->support.nnz);
    if (rc != RL_OK) return rc;
    if ((rc = check_params(params)) != RL_OK) return rc;
    if (keep_e_active(params))
        return fail(RL_ERR_ARG, "keep_e is for the single-GPU forward: the shard path's saved state holds no numerators");
    if (n_shards < 1 || n_shards > 4096) return fail(RL_ERR_ARG, "n_shards out of [1, 4096]");
    const bool any = batch->N > 0;
    if (any && (!batch->labels || !batch->label_logq || !batch->adv || !batch->support.offsets ||
                !batch->support.replayed || (batch->support.nnz > 0 && (!batch->support.ids || !batch->support.logq))))
        return fail(RL_ERR_ARG, "required batch pointer is NULL");
    if (!out || (any && (!out->loss || !saved || !stats_all || !zlab || (batch->support.nnz > 0 && !zsup))) ||
        !dev_status)
        return fail(RL_ERR_ARG, "out/loss/saved/stats/zlab/zsup/dev_status NULL");
    if (ws_bytes < rl_head_fwd_workspace_bytes(batch->N, batch->H, batch->V, batch->support.nnz, params) || !ws)
        return fail(RL_ERR_WORKSPACE, "forward workspace too small");
    if (!sm100_family()) return fail(RL_ERR_UNSUPPORTED, "needs an sm_100-family GPU");
    return loss_from_shards_impl(batch, params, n_shards, stats_all, zlab, zsup, out, saved, ws, dev_status,
                                 as_stream(stream));
}

int rl_mismatch_metrics(const rl_head_batch* batch, const void* saved, rl_head_metrics* metrics, void* ws,
                        size_t ws_bytes, void* stream) {
    int rc = check_batch(batch);
    if (rc != RL_OK) return rc;
    if (!saved || !metrics || !ws) return fail(RL_ERR_ARG, "saved/metrics/ws NULL");
    if (ws_bytes < rl_head_fwd_workspace_bytes(batch->N, batch->H, batch->V, batch->support.nnz, nullptr))
        return fail(RL_ERR_WORKSPACE, "workspace too small");
    if (!sm100_family()) return fail(RL_ERR_UNSUPPORTED, "needs an sm_100-family GPU");
    return metrics_impl(batch, saved, metrics, ws, as_stream(stream));
}

size_t rl_policy_workspace_bytes(int64_t T) { return T < 0 ? 0 : policy_ws_bytes(T); }

int rl_policy_loss_elementwise(const float* lp_theta, const float* lp_old, const float* lp_samp, const float* adv,
                               const uint8_t* mask, int64_t T, const rl_pg_params* params, float* loss_ppo,
                               float* loss_dec, float* grad_ppo, float* grad_dec, rl_pg_metrics* metrics, void* ws,
                               size_t ws_bytes, void* stream) {
    if (T < 0) return fail(RL_ERR_ARG, "T < 0");
    if (!params) return fail(RL_ERR_ARG, "params NULL");
    if (params->n_curve < 0 || params->n_curve > RL_PG_MAX_CURVE) return fail(RL_ERR_ARG, "bad n_curve");
    if (!(params->clip_ratio_low >= 0.f) || !(params->clip_ratio_high >= 0.f) || !(params->clip_ratio_c > 1.f) ||
        !(params->tis_upper > 0.f) || !(params->icepop_low <= params->icepop_high))
        return fail(RL_ERR_ARG, "bad pg params");
    if (T > 0 && (!lp_theta || !lp_old || !lp_samp || !adv)) return fail(RL_ERR_ARG, "input NULL");
    if (ws_bytes < rl_policy_workspace_bytes(T) || !ws) return fail(RL_ERR_WORKSPACE, "policy workspace too small");
    if (T == 0 && !metrics) return RL_OK;
    if (!sm100_family()) return fail(RL_ERR_UNSUPPORTED, "needs an sm_100-family GPU");
    return policy_impl(lp_theta, lp_old, lp_samp, adv, mask, T, params, loss_ppo, loss_dec, grad_ppo, grad_dec,
                       metrics, ws, ws_bytes, as_stream(stream));
}

size_t rl_rollout_correction_workspace_bytes(int64_t B) { return B < 0 ? 0 : rollout_ws_bytes(B); }

int rl_rollout_correction(const float* lp_train, const float* lp_rollout, const uint8_t* mask,
                          const int64_t* seq_offsets, int64_t B, int64_t T, const rl_rc_params* params,
                          float* weights, uint8_t* keep, rl_rc_metrics* metrics, void* ws, size_t ws_bytes,
                          void* stream) {
    if (T < 0 || B < 0) return fail(RL_ERR_ARG, "T < 0 or B < 0");
    if (B == 0 && T > 0) return fail(RL_ERR_ARG, "T > 0 with no sequence: the offsets must cover [0, T)");
    if (B >= (int64_t(1) << 31)) return fail(RL_ERR_UNSUPPORTED, "B >= 2^31");
    if (!params) return fail(RL_ERR_ARG, "params NULL");
    const rl_rc_params& p = *params;
    auto level_ok = [](int l) { return l == RL_LEVEL_TOKEN || l == RL_LEVEL_SEQUENCE || l == RL_LEVEL_GEOMETRIC; };
    if (p.tis_mode != RL_TIS_TRUNCATE && p.tis_mode != RL_TIS_CLIP && p.tis_mode != RL_TIS_MASK)
        return fail(RL_ERR_ARG, "bad tis_mode");
    if (!level_ok(p.tis_level) || !level_ok(p.rs_level)) return fail(RL_ERR_ARG, "bad level");
    if (!(p.tis_lower_bound >= 0.f) || !(p.tis_upper_bound >= p.tis_lower_bound))
        return fail(RL_ERR_ARG, "tis bounds: need 0 <= lower <= upper");
    const float rl = std::isnan(p.rs_lower_bound) ? p.tis_lower_bound : p.rs_lower_bound;
    const float ru = std::isnan(p.rs_upper_bound) ? p.tis_upper_bound : p.rs_upper_bound;
    if (!(rl >= 0.f) || !(ru >= rl)) return fail(RL_ERR_ARG, "rs bounds: need 0 <= lower <= upper");
    if (B > 0 && !seq_offsets) return fail(RL_ERR_ARG, "seq_offsets NULL");
    if (T > 0 && (!lp_train || !lp_rollout || !mask)) return fail(RL_ERR_ARG, "input NULL");
    if (!ws || ws_bytes < rl_rollout_correction_workspace_bytes(B))
        return fail(RL_ERR_WORKSPACE, "rollout-correction workspace too small");
    if (!sm100_family()) return fail(RL_ERR_UNSUPPORTED, "needs an sm_100-family GPU");
    return rollout_impl(lp_train, lp_rollout, mask, seq_offsets, B, T, params, weights, keep, metrics, ws,
                        ws_bytes, as_stream(stream));
}

int rl_rollout_metrics_named(const rl_rc_metrics* metrics, const rl_rc_params* params, rl_rc_named* named,
                             void* stream) {
    if (!metrics || !params || !named) return fail(RL_ERR_ARG, "NULL pointer");
    if (params->tis_mode != RL_TIS_TRUNCATE && params->tis_mode != RL_TIS_CLIP && params->tis_mode != RL_TIS_MASK)
        return fail(RL_ERR_ARG, "bad tis_mode");
    if (!sm100_family()) return fail(RL_ERR_UNSUPPORTED, "needs an sm_100-family GPU");
    return rollout_named_impl(metrics, params, named, as_stream(stream));
}

int rl_gemm_bf16(const void* A, int a_mn_major, const void* B, int b_mn_major, int64_t M, int64_t N,
                 int64_t K, float* D, int32_t* dev_status, void* stream) {
    if (!A || !B || !D || !dev_status) return fail(RL_ERR_ARG, "NULL pointer");
    if (M <= 0 || N <= 0 || K <= 0) return fail(RL_ERR_ARG, "non-positive size");
    if (N % 4 != 0) return fail(RL_ERR_UNSUPPORTED, "N % 4 != 0");
    if ((a_mn_major ? M : K) % 8 != 0 || (b_mn_major ? N : K) % 8 != 0)
        return fail(RL_ERR_UNSUPPORTED, "contiguous extent of an operand not a multiple of 8");
    if (!aligned16(A) || !aligned16(B) || !aligned16(D)) return fail(RL_ERR_ARG, "not 16-byte aligned");
    if (!sm100_family()) return fail(RL_ERR_UNSUPPORTED, "needs an sm_100-family GPU");
    return gemm_util_impl(A, a_mn_major != 0, B, b_mn_major != 0, M, N, K, D, dev_status, as_stream(stream));
}

int rl_gemm_bf16_tn(const void* A, const void* B, int64_t M, int64_t N, int64_t K, float* D,
                    int32_t* dev_status, void* stream) {
    return rl_gemm_bf16(A, 0, B, 0, M, N, K, D, dev_status, stream);
}

int rl_wait_selftest(int32_t* dev_status, void* stream) {
    if (!dev_status) return fail(RL_ERR_ARG, "dev_status is NULL");
    if (!sm100_family()) return fail(RL_ERR_UNSUPPORTED, "needs an sm_100-family GPU");
    return wait_selftest_impl(dev_status, as_stream(stream));
}

int rl_status_read(const int32_t* dev_status, int32_t* host_out) {
    if (!dev_status || !host_out) return fail(RL_ERR_ARG, "NULL pointer");
    return cudaMemcpy(host_out, dev_status, sizeof(int32_t), cudaMemcpyDeviceToHost) == cudaSuccess ? RL_OK
                                                                                                     : RL_ERR_CUDA;
}

int64_t rl_kernel_launch_count(void) {
    return rl_launch_counter_value();
}

const char* rl_error_string(int code) {
    switch (code) {
        case RL_OK: return "ok";
        case RL_ERR_ARG: return "invalid argument";
        case RL_ERR_WORKSPACE: return "workspace too small";
        case RL_ERR_UNSUPPORTED: return "unsupported shape or device";
        case RL_ERR_CUDA: return "CUDA error";
        default: return "unknown error";
    }
}

}  // extern "C"
