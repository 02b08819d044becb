// rl_gemm_bf16_tn: the head contraction alone, D[M, N] (fp32) = A[M, K] B[N, K]^T with
// bf16 K-major operands, through the same tcgen05 pipeline as the fused kernels and a
// plain store epilogue.  Used to unit-test and time the tensor-core path in isolation.
#include "gemm_tc2.cuh"
#include "internal.h"

namespace rl {

struct EpiStore {
    struct Params {
        int64_t M, N;
        float* D;
    };
    int64_t t;
    bool valid;
    RL_DEVINL void begin_unit(const Params& p, int row, int, int m_blk, int, int) {
        t = static_cast<int64_t>(m_blk) * kBM + row;
        valid = t < p.M;
    }
    RL_DEVINL void chunk(const Params& p, const uint32_t (&acc)[32], int col0, uint8_t*, int) {
        if (!valid || col0 >= p.N) return;
        float* d = p.D + t * p.N + col0;
        if (col0 + 32 <= p.N) {
            float4* d4 = reinterpret_cast<float4*>(d);
#pragma unroll
            for (int q = 0; q < 8; ++q)
                d4[q] = make_float4(__uint_as_float(acc[4 * q]), __uint_as_float(acc[4 * q + 1]),
                                    __uint_as_float(acc[4 * q + 2]), __uint_as_float(acc[4 * q + 3]));
        } else {
#pragma unroll
            for (int k = 0; k < 32; ++k)
                if (col0 + k < p.N) d[k] = __uint_as_float(acc[k]);
        }
    }
    RL_DEVINL void end_unit(const Params&, int, int) {}
};

int gemm_util_impl(const void* A, int a_mn, const void* B, int b_mn, int64_t M, int64_t N, int64_t K,
                   float* D, int32_t* status, cudaStream_t stream) {
    CUtensorMap ta, tb;
    const int pair = gemm_pair_mode();
    int rc = a_mn ? make_tmap_bf16(&ta, A, K, M, M, 64) : make_tmap_bf16(&ta, A, M, K, K, kBM);
    if (rc != RL_OK) return rc;
    rc = b_mn ? make_tmap_bf16(&tb, B, K, N, N, 64) : make_tmap_bf16(&tb, B, N, K, K, pair ? kBN / 2 : kBN);
    if (rc != RL_OK) return rc;
    const GemmPlan plan = make_plan(M, N, K, 1, 1 << 30, 1, status, a_mn, b_mn, pair);
    if (pair) {
        EpiStore::Params ep{M, N, D};
        ProfScope ps(RL_PROF_GEMM_UTIL, stream);
        rc = launch_gemm_pair<EpiStore>(ta, ta, tb, plan, ep, stream);
        count_launch();
        return rc;
    }
    EpiStore::Params ep{M, N, D};
    {
        ProfScope ps(RL_PROF_GEMM_UTIL, stream);
        rc = launch_gemm<EpiStore>(ta, ta, tb, plan, ep, stream);
    }
    count_launch();
    return rc;
}

// One thread waits, with the work-loop limit, on an mbarrier of its block that nothing
// arrives on: the wait runs out, ORs RL_STATUS_TIMEOUT into *status and returns false;
// the kernel then ends normally (no copy or MMA is in flight, so nothing to drain).
__global__ void wait_selftest_kernel(int32_t* status, uint64_t wait_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_wait(&bar, 0, status, wait_ns);
}

int wait_selftest_impl(int32_t* status, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(status, wait_limit_ns());
    count_launch();
    return cudaPeekAtLastError() == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}

}  // namespace rl
