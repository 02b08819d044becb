// Host runtime of librlhead: TMA descriptor encoding, device queries, GEMM planning,
// launch accounting and error strings.
#include <atomic>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "gemm_tc.cuh"
#include "internal.h"

namespace rl {

static std::atomic<int64_t> g_launches{0};
static thread_local char g_last_error[256] = "";

void count_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
void set_last_error(const char* msg) {
    std::strncpy(g_last_error, msg, sizeof(g_last_error) - 1);
    g_last_error[sizeof(g_last_error) - 1] = 0;
}

int num_sms() {
    int dev = 0;
    cudaGetDevice(&dev);
    static int cached[64] = {0};
    if (dev < 0 || dev >= 64) return 148;
    if (cached[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 148;
    }
    return cached[dev];
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

GemmPlan make_plan(int64_t M, int64_t N, int64_t K, int passes, int n_splits, int m_fastest,
                   int32_t* status) {
    GemmPlan p;
    p.m_blocks = static_cast<int>((M + kBM - 1) / kBM);
    p.n_blocks = static_cast<int>((N + kBN - 1) / kBN);
    if (n_splits < 1) n_splits = 1;
    if (n_splits > p.n_blocks) n_splits = p.n_blocks;
    p.tiles_per_unit = (p.n_blocks + n_splits - 1) / n_splits;
    p.n_splits = (p.n_blocks + p.tiles_per_unit - 1) / p.tiles_per_unit;
    p.num_units = p.m_blocks * p.n_splits;
    p.m_fastest = m_fastest;
    p.kb_per_pass = static_cast<int>((K + kBK - 1) / kBK);
    p.passes = passes;
    p.status = status;
    return p;
}

}  // namespace rl

int64_t rl_launch_counter_value() { return rl::g_launches.load(std::memory_order_relaxed); }

extern "C" const char* rl_last_error(void) { return rl::g_last_error; }
