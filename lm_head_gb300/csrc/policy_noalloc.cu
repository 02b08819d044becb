// rl_policy_loss_elementwise_noalloc: the elementwise PPO / TIS / mismatch path for callers
// that cannot allocate device memory.  Its scratch (the counters, flags and metric
// accumulators) lives in a file-scope device array instead of a caller workspace.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace rl {

// 4096 bytes: the elementwise pass's workspace.
constexpr size_t kNoAllocScratchBytes = kPolicyWorkspaceBytes;
static __device__ __align__(256) double g_policy_scratch[kNoAllocScratchBytes / sizeof(double)];

// Device address of g_policy_scratch for the current device, looked up once per device
// with that device current.  In host code the array's name is only a host-side stand-in.
static int scratch_address(void** out) {
    static std::mutex mu;
    static void* addr[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return RL_ERR_CUDA;
    std::lock_guard<std::mutex> g(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_policy_scratch) != cudaSuccess || p == nullptr) {
            set_last_error("cudaGetSymbolAddress of the static scratch failed");
            return RL_ERR_CUDA;
        }
        addr[dev] = p;
    }
    *out = addr[dev];
    return RL_OK;
}

}  // namespace rl

extern "C" int rl_policy_loss_elementwise_noalloc(const float* lp_theta, const float* lp_old,
                                                  const float* lp_samp, const float* adv,
                                                  const uint8_t* mask, int64_t T,
                                                  const rl_pg_params* params, float* loss_ppo,
                                                  float* loss_dec, float* grad_ppo, float* grad_dec,
                                                  rl_pg_metrics* metrics, void* stream) {
    using namespace rl;
    if (T < 0 || !params) {
        set_last_error("T < 0 or params NULL");
        return RL_ERR_ARG;
    }
    if (params->n_curve < 0 || params->n_curve > RL_PG_MAX_CURVE || !(params->clip_ratio_low >= 0.f) ||
        !(params->clip_ratio_high >= 0.f) || !(params->clip_ratio_c > 1.f) || !(params->tis_upper > 0.f) ||
        !(params->icepop_low <= params->icepop_high)) {
        set_last_error("bad pg params");
        return RL_ERR_ARG;
    }
    if (T > 0 && (!lp_theta || !lp_old || !lp_samp || !adv)) {
        set_last_error("input NULL");
        return RL_ERR_ARG;
    }
    if (T == 0 && !metrics) return RL_OK;
    int dev = 0, major = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess || major != 10) {
        set_last_error("needs an sm_100-family GPU");
        return RL_ERR_UNSUPPORTED;
    }
    static_assert(kNoAllocScratchBytes >= kPolicyWorkspaceBytes, "the scratch must hold the pass's workspace");
    void* scratch = nullptr;
    int rc = scratch_address(&scratch);
    if (rc != RL_OK) return rc;
    return policy_impl(lp_theta, lp_old, lp_samp, adv, mask, T, params, loss_ppo, loss_dec, grad_ppo,
                       grad_dec, metrics, scratch, kNoAllocScratchBytes, static_cast<cudaStream_t>(stream));
}
