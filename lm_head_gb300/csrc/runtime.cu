// Host runtime of librlhead: TMA descriptor encoding, device queries, GEMM planning,
// launch accounting and error strings.
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include <cudaTypedefs.h>

#include "gemm_tc.cuh"
#include "internal.h"

namespace rl {

static std::atomic<int64_t> g_launches{0};
static std::atomic<int> g_gemm_pair{1};
constexpr int kWaitLimitUsDefault = 1000000;          // 1 s, the device-side kWaitLimitNs
constexpr int kWaitLimitUsMax = 10000000;
static std::atomic<int> g_wait_limit_us{kWaitLimitUsDefault};

int gemm_pair_mode() { return g_gemm_pair.load(std::memory_order_relaxed); }
uint64_t wait_limit_ns() { return 1000ull * static_cast<uint64_t>(g_wait_limit_us.load(std::memory_order_relaxed)); }
static thread_local char g_last_error[256] = "";

void count_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

// ---- per-kind launch timing with recycled CUDA events ------------------------------
namespace {
struct Prof {
    std::mutex mu;
    bool on = false;
    std::vector<cudaEvent_t> pool;
    struct Pending {
        int kind;
        cudaEvent_t a, b;
    };
    std::vector<Pending> pending;
    double ms[RL_PROF_KINDS] = {0};
    int64_t launches[RL_PROF_KINDS] = {0};
    cudaEvent_t get() {
        if (!pool.empty()) {
            cudaEvent_t e = pool.back();
            pool.pop_back();
            return e;
        }
        cudaEvent_t e = nullptr;
        cudaEventCreate(&e);
        return e;
    }
};
Prof& prof() {
    static Prof p;
    return p;
}
}  // namespace

ProfScope::ProfScope(int k, cudaStream_t s) : kind(k), stream(s), begin(nullptr) {
    Prof& p = prof();
    std::lock_guard<std::mutex> g(p.mu);
    if (!p.on) return;
    cudaEvent_t e = p.get();
    if (e && cudaEventRecord(e, s) == cudaSuccess) begin = e;
}
ProfScope::~ProfScope() {
    if (!begin) return;
    Prof& p = prof();
    std::lock_guard<std::mutex> g(p.mu);
    cudaEvent_t e = p.get();
    if (e && cudaEventRecord(e, stream) == cudaSuccess)
        p.pending.push_back({kind, static_cast<cudaEvent_t>(begin), e});
}
void set_last_error(const char* msg) {
    std::strncpy(g_last_error, msg, sizeof(g_last_error) - 1);
    g_last_error[sizeof(g_last_error) - 1] = 0;
}

int num_sms() {
    int dev = 0;
    cudaGetDevice(&dev);
    static std::atomic<int> cached[64];   // zero-initialised (static storage); one per device
    if (dev < 0 || dev >= 64) return 148;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        n = n > 0 ? n : 148;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

int make_tmap_bf16(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld,
                   int box_rows) {
    auto fn = encode_fn();
    if (!fn) {
        set_last_error("cuTensorMapEncodeTiled unavailable");
        return RL_ERR_CUDA;
    }
    if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || (ld * 2) % 16 != 0 || rows <= 0 ||
        cols <= 0 || rows > (int64_t(1) << 31) || cols > (int64_t(1) << 31)) {
        set_last_error("tensor map: misaligned base/stride or bad extent");
        return RL_ERR_UNSUPPORTED;
    }
    cuuint64_t gdim[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t gstride[1] = {static_cast<cuuint64_t>(ld * 2)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim,
                    gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_last_error("cuTensorMapEncodeTiled failed");
        return RL_ERR_CUDA;
    }
    return RL_OK;
}

int make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int elem_bytes, int64_t rows,
                 int64_t cols, int64_t ld, int box_cols, int box_rows, int swizzle_bytes) {
    auto fn = encode_fn();
    if (!fn) {
        set_last_error("cuTensorMapEncodeTiled unavailable");
        return RL_ERR_CUDA;
    }
    if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || (ld * elem_bytes) % 16 != 0 || rows <= 0 || cols <= 0) {
        set_last_error("tensor map: misaligned base/stride or bad extent");
        return RL_ERR_UNSUPPORTED;
    }
    cuuint64_t gdim[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t gstride[1] = {static_cast<cuuint64_t>(ld * elem_bytes)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = fn(map, dtype, 2, const_cast<void*>(base), gdim, gstride, box, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                    : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                          : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_last_error("cuTensorMapEncodeTiled failed");
        return RL_ERR_CUDA;
    }
    return RL_OK;
}

GemmPlan make_plan(int64_t M, int64_t N, int64_t K, int passes, int n_splits, int m_fastest,
                   int32_t* status, int a_mn, int b_mn, int pair) {
    GemmPlan p;
    const int64_t rows = pair ? 2 * kBM : kBM;
    p.m_blocks = static_cast<int>((M + rows - 1) / rows);
    p.n_blocks = static_cast<int>((N + kBN - 1) / kBN);
    if (n_splits < 1) n_splits = 1;
    if (n_splits > p.n_blocks) n_splits = p.n_blocks;
    p.tiles_per_unit = (p.n_blocks + n_splits - 1) / n_splits;
    p.n_splits = (p.n_blocks + p.tiles_per_unit - 1) / p.tiles_per_unit;
    p.num_units = p.m_blocks * p.n_splits;
    p.m_fastest = m_fastest;
    p.kb_per_pass = static_cast<int>((K + kBK - 1) / kBK);
    p.passes = passes;
    p.a_mn = a_mn;
    p.b_mn = b_mn;
    p.status = status;
    p.wait_ns = wait_limit_ns();
    return p;
}

}  // namespace rl

int64_t rl_launch_counter_value() { return rl::g_launches.load(std::memory_order_relaxed); }

extern "C" const char* rl_last_error(void) { return rl::g_last_error; }

extern "C" int rl_set_option(int key, int value) {
    if (key == RL_OPT_GEMM_PAIR) {
        rl::g_gemm_pair.store(value ? 1 : 0, std::memory_order_relaxed);
        return RL_OK;
    }
    if (key == RL_OPT_WAIT_LIMIT_US) {
        if (value < 1 || value > rl::kWaitLimitUsMax) {
            rl::set_last_error("wait limit out of [1, 10000000] us");
            return RL_ERR_ARG;
        }
        rl::g_wait_limit_us.store(value, std::memory_order_relaxed);
        return RL_OK;
    }
    rl::set_last_error("unknown option");
    return RL_ERR_ARG;
}

extern "C" int rl_get_option(int key) {
    if (key == RL_OPT_GEMM_PAIR) return rl::g_gemm_pair.load(std::memory_order_relaxed);
    if (key == RL_OPT_WAIT_LIMIT_US) return rl::g_wait_limit_us.load(std::memory_order_relaxed);
    return -1;
}

extern "C" int rl_profile_enable(int on) {
    rl::Prof& p = rl::prof();
    std::lock_guard<std::mutex> g(p.mu);
    p.on = on != 0;
    for (auto& q : p.pending) {
        p.pool.push_back(q.a);
        p.pool.push_back(q.b);
    }
    p.pending.clear();
    for (int k = 0; k < RL_PROF_KINDS; ++k) {
        p.ms[k] = 0.0;
        p.launches[k] = 0;
    }
    return RL_OK;
}

extern "C" int rl_profile_read(double* ms, int64_t* launches) {
    rl::Prof& p = rl::prof();
    std::lock_guard<std::mutex> g(p.mu);
    int rc = RL_OK;
    for (auto& q : p.pending) {
        float t = 0.f;
        if (cudaEventSynchronize(q.b) != cudaSuccess || cudaEventElapsedTime(&t, q.a, q.b) != cudaSuccess)
            rc = RL_ERR_CUDA;
        if (q.kind >= 0 && q.kind < RL_PROF_KINDS) {
            p.ms[q.kind] += t;
            p.launches[q.kind] += 1;
        }
        p.pool.push_back(q.a);
        p.pool.push_back(q.b);
    }
    p.pending.clear();
    for (int k = 0; k < RL_PROF_KINDS; ++k) {
        if (ms) ms[k] = p.ms[k];
        if (launches) launches[k] = p.launches[k];
    }
    return rc;
}

extern "C" const char* rl_profile_kind_name(int kind) {
    static const char* names[RL_PROF_KINDS] = {
        "validate", "gemm_fwd_stats", "token_loss", "metrics", "transpose", "gemm_bwd_grad",
        "gemm_bwd_dx", "gemm_bwd_dw", "sparse_dx", "sparse_dw", "policy", "gemm_util", "memset", "other",
        "spike_resid", "grad_from_e", "ref_logit", "rollout"};
    return (kind >= 0 && kind < RL_PROF_KINDS) ? names[kind] : "unknown";
}
