// Host-side declarations shared by the translation units of librlhead.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/rlhead.h"

namespace rl {

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Bump allocator over a caller-provided buffer (or a null base when only measuring).
struct Carve {
    uint8_t* base;
    size_t off = 0;
    explicit Carve(void* b) : base(static_cast<uint8_t*>(b)) {}
    template <class T>
    T* take(size_t count) {
        off = align_up(off, 256);
        T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
        off += count * sizeof(T);
        return p;
    }
};

// Forward -> backward saved state (caller-owned).
struct SavedView {
    float* lse;       // [N] full-vocab logsumexp of z
    float* lse_s;     // [N] logsumexp over the support on replayed rows (= lse otherwise)
    float* dcoef;     // [N] coefficient of the dense softmax term P_full (0 on replayed rows)
    float* labcoef;   // [N] coefficient of the spike at the label
    float* entcoef;   // [nnz] coefficient of the spike at each support entry
    float* mterm;     // [N, 8] per-token metric terms
    float* zlab;      // [N] label logit z_t,a_t (already / T), as the forward GEMM produced it
    float* zsup;      // [nnz] support logits, same
};
SavedView saved_view(void* base, int64_t N, int64_t nnz, size_t* bytes);

struct FwdWs {
    int splits;
    float* part_m;    // [splits, N]
    float* part_s;
    float* part_u;
    double* mpart;    // metric partials
};
FwdWs fwd_ws_view(void* base, int64_t N, int64_t H, int64_t V, int64_t nnz, size_t* bytes);
constexpr int kMetricBlocks = 128;
constexpr int kMetricFields = 16;

struct BwdWs {
    int64_t chunk;        // tokens per chunk (multiple of 128)
    bool dense;
    bool split;
    void* Wt;             // [H, V] bf16 (dense)
    void* Xt;             // [H, chunk] bf16 (dense)
    void* G;              // [chunk, V] bf16 (dense)       (hi)
    void* Gt;             // [V, chunk] bf16 (dense)       (hi)
    void* G_lo;           // split only
    void* Gt_lo;
    float* dxs;           // [N, H] fp32 sparse part of dX
    float* resid;         // [nnz + N] what bf16 rounding of the dense G drops at each spike
    int32_t* item_tok;    // [nnz + N] token of each gradient item
    int32_t* keys_a;      // radix-sort double buffers (vocab id keys, item payloads)
    int32_t* vals_a;
    int32_t* keys_b;
    int32_t* vals_b;
    int32_t* hist;        // [tiles, 512]
    int64_t* bucket;      // [V + 1] start of each vocab id's items after the sort
};
BwdWs bwd_ws_view(void* base, int64_t N, int64_t H, int64_t V, int64_t nnz,
                  const rl_params* prm, size_t* bytes);
bool bwd_is_dense(const rl_params* prm);

void count_launch(int n = 1);

// Event pair around a launch group when profiling is on (see rl_profile_enable).
struct ProfScope {
    int kind;
    cudaStream_t stream;
    void* begin;
    ProfScope(int kind, cudaStream_t s);
    ~ProfScope();
};
void set_last_error(const char* msg);
int num_sms();
// Limit of the kernels' work-loop waits, ns (RL_OPT_WAIT_LIMIT_US; read at each launch).
uint64_t wait_limit_ns();

int head_fwd_impl(const rl_head_batch* b, const rl_params* prm, const rl_head_outputs* out,
                  void* saved, void* ws, int32_t* status, cudaStream_t stream);
int metrics_impl(const rl_head_batch* b, const void* saved, rl_head_metrics* metrics, void* ws,
                 cudaStream_t stream);
// flags / nflags: the fused path's per-chunk range flags (counted into recomputed_chunks)
int metrics_run(const rl_head_batch* b, const void* saved, rl_head_metrics* metrics, double* mpart,
                cudaStream_t stream, const int* flags = nullptr, int nflags = 0);
// What the forward GEMM of the fused forward + backward leaves for the backward of one
// token chunk (all per-token arrays chunk-relative).
//  bf16 gradient precision:  Eb [n, V] and Ebt [V, ldt] hold e = 2^(z log2(e) - cref) in
//    bf16, one reference cref per row (the label logit, log2 units), so that the dense
//    softmax gradient is G = rs * e with one scale rs = alpha 2^(cref - lse log2(e)) per
//    row (token_loss writes rs).  *flag = 1 when a row's values leave the range where that
//    holds; the chunk's dense backward then recomputes G from the logits instead.
//  hi/lo gradient precision: E32 [n, V] holds e = 2^(z log2(e) - m2) in fp32 with the
//    running max m2 it is relative to per 32-column chunk in M2 [n, ldm].
struct EStore {
    uint16_t* Eb = nullptr;
    uint16_t* Ebt = nullptr;
    int64_t ldt = 0;
    const float* cref = nullptr;
    int* flag = nullptr;
    float* rs = nullptr;
    const float* dloss = nullptr;
    float* E32 = nullptr;
    float* M2 = nullptr;
};
// Largest |log2| distance between a row's logits and its reference that the bf16 store
// accepts; beyond it the chunk takes the recompute path.
constexpr float kRefRangeLog2 = 64.f;
int fwd_rows(const rl_head_batch* b, const rl_params* prm, const rl_head_outputs* out, const SavedView& sv,
             const FwdWs& w, int64_t c0, int64_t n, const EStore* es, int sparse, int32_t* status,
             cudaStream_t stream);
int head_fused_impl(const rl_head_batch* b, const rl_params* prm, const rl_head_outputs* out,
                    const float* dloss, void* dhidden, float* dW, int accumulate, void* saved, void* ws,
                    int32_t* status, cudaStream_t stream);
size_t fused_ws_bytes(int64_t N, int64_t H, int64_t V, int64_t nnz, const rl_params* prm);
int validate_impl(const rl_head_batch* b, int32_t* status, cudaStream_t stream);
int shard_remap_impl(const int32_t* in, int64_t n, int64_t v0, int64_t v1, int32_t* out, cudaStream_t stream);
int shard_stats_impl(const rl_head_batch* b, const rl_params* prm, float* stats, float* zlab, float* zsup, void* ws,
                     int32_t* status, cudaStream_t stream);
int loss_from_shards_impl(const rl_head_batch* b, const rl_params* prm, int32_t R, const float* stats_all,
                          const float* zlab, const float* zsup, const rl_head_outputs* out, void* saved, void* ws,
                          int32_t* status, cudaStream_t stream);
int64_t bwd_chunk(int64_t N, int64_t H, const rl_params* prm);
// rl_params.keep_e in effect: a dense backward with BF16 gradients and no entropy term.
bool keep_e_active(const rl_params* prm);
// The kept numerators in the saved state, after the standard saved data: e [N, V] and
// e^T [V, N] bf16, the reference logit per token, the range flag per token chunk.
struct KeptView {
    uint16_t* Eb;
    uint16_t* Ebt;        // [V, ldt]: ldt = N rounded up to 128 (TMA strides are multiples of 16 bytes)
    int64_t ldt;
    float* cref;
    int* flags;          // one per token chunk: room for the smallest chunk (one row tile)
    int64_t chunks_max;
};
KeptView kept_view(void* saved, int64_t N, int64_t nnz, int64_t V, const rl_params* prm, size_t* bytes);
// The forward with keep_e: per token chunk the reference logits, then the forward GEMM that
// also stores e / e^T into the saved state.
int head_fwd_kept(const rl_head_batch* b, const rl_params* prm, const rl_head_outputs* out, void* saved,
                  void* ws, int32_t* status, cudaStream_t stream);
// Workspace of the backward on kept numerators.
size_t kept_bwd_ws_bytes(int64_t N, int64_t H, int64_t V, int64_t nnz, const rl_params* prm);
int head_bwd_impl(const rl_head_batch* b, const rl_params* prm, const void* saved,
                  const float* dloss, void* dhidden, float* dW, int accumulate, void* ws,
                  int32_t* status, cudaStream_t stream);
int policy_impl(const float* lt, const float* lo, const float* ls, const float* adv,
                const uint8_t* mask, int64_t T, const rl_pg_params* p, float* loss_ppo,
                float* loss_dec, float* grad_ppo, float* grad_dec, rl_pg_metrics* metrics,
                void* ws, size_t ws_bytes, cudaStream_t stream);
size_t policy_ws_bytes(int64_t T);
// The elementwise pass's workspace: counters, flags and the metric accumulators (one
// 128-byte line each).
constexpr size_t kPolicyWorkspaceBytes = 4096;
int rollout_impl(const float* lt, const float* lr, const uint8_t* mask, const int64_t* off, int64_t B, int64_t T,
                 const rl_rc_params* p, float* w, uint8_t* keep, rl_rc_metrics* metrics, void* ws,
                 size_t ws_bytes, cudaStream_t stream);
size_t rollout_ws_bytes(int64_t B);
int rollout_named_impl(const rl_rc_metrics* m, const rl_rc_params* p, rl_rc_named* named, cudaStream_t stream);
int wait_selftest_impl(int32_t* status, cudaStream_t stream);
int gemm_util_impl(const void* A, int a_mn, const void* B, int b_mn, int64_t M, int64_t N, int64_t K,
                   float* D, int32_t* status, cudaStream_t stream);

}  // namespace rl
