// Pair (cta_group::2) variant of the tcgen05 GEMM: a cluster of two CTAs on two SMs
// computes a 256 x 256 tile per MMA step,
//
//   D[256 rows, 256 cols] = A[256, K] * B[256, K]^T,
//
// CTA rank r of the pair holds A rows [128 r, 128 r + 128) and B rows [128 r, 128 r + 128)
// of the tile in its own shared memory, and its 128 output rows in its own TMEM.  Per SM a
// 64-deep K step stages 32 KB (16 KB of A + half of B) instead of 48 KB, so six stages fit
// beside the epilogue staging tiles.
//
// * Both CTAs: warp 0 lane 0 loads its A and B halves with TMA (.cta_group::2), the
//   completion bytes of both CTAs counted on the even CTA's full barrier.  An operand
//   stored M- (or N-) contiguous comes in as two 64 x 64 boxes per CTA (plan.a_mn / b_mn)
//   and is described to the MMA as MN-major.
// * Even CTA only: warp 1 lane 0 issues tcgen05.mma.cta_group::2 (M=256, N=256, K=16) and
//   commits with multicast to both CTAs' "stage empty" and "accumulator full" barriers.
// * Both CTAs: warps 2-9 drain their own TMEM (same epilogue policies as gemm_tc_kernel,
//   with m_blk = 2 * pair_block + rank) and release the accumulator to the even CTA's
//   barrier (16 arrivals).
// * TMEM is allocated / freed collectively (one warp of each CTA, cta_group::2).
// Every mbarrier wait is bounded as in gemm_tc_kernel; cluster barriers at entry (before
// any cross-CTA signal) and before exit (no CTA leaves while its peer may still signal it).
#pragma once

#include "gemm_tc.cuh"

namespace rl {

constexpr int kStages2 = 6;
constexpr int kATileBytes2 = kBM * kBK * 2;          // 16 KB
constexpr int kBTileBytes2 = (kBN / 2) * kBK * 2;    // 16 KB (this CTA's half of B)
constexpr int kStageBytes2 = kATileBytes2 + kBTileBytes2;
constexpr int kGemmSmemBytes2 = kStages2 * kStageBytes2 + kEpiWarps * kEpiStageBytes + 1024 + 256;
constexpr uint32_t kIdesc2 = idesc_bf16_f32(2 * kBM, kBN);

RL_DEVINL uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Address of the same shared variable in CTA `rank` of the cluster.
RL_DEVINL uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
RL_DEVINL void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}
RL_DEVINL void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                     "memory");
}
RL_DEVINL void tma_load_2d_pair(const CUtensorMap* map, uint32_t bar_cluster_addr, void* dst, int32_t x,
                                int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster_addr)
        : "memory");
}
RL_DEVINL void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
RL_DEVINL void umma_commit_pair_multicast(uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_addr(bar)),
        "h"(cta_mask)
        : "memory");
}
RL_DEVINL void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
RL_DEVINL void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
RL_DEVINL void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// plan.m_blocks counts 256-row pair blocks here.
template <class Epi>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tc2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                    const __grid_constant__ CUtensorMap tmB, const GemmPlan plan,
                    const __grid_constant__ typename Epi::Params ep) {
    if (!epi_gate_open(ep, 0)) return;   // uniform over the grid: both CTAs of a pair leave
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* epi_stage = smem + kStages2 * kStageBytes2;
    uint64_t* full = reinterpret_cast<uint64_t*>(epi_stage + kEpiWarps * kEpiStageBytes);
    uint64_t* empty = full + kStages2;
    uint64_t* accf = empty + kStages2;
    uint64_t* acce = accf + 2;
    uint64_t* done_bar = acce + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages2; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf + b, 1);
            mbar_init(acce + b, 2 * kEpiWarps);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (plan.passes > 1) tma_prefetch_desc(&tmA2);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();   // barriers of both CTAs initialised, TMEM allocated in both
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int kb_total = plan.kb_per_pass * plan.passes;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs) ----------------
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            bool issued = false;
            for (int u = pair; u < plan.num_units && ok; u += npairs) {
                const UnitCoords c = decode_unit(plan, u);
                for (int nb = c.nb_begin; nb < c.nb_end && ok; ++nb) {
                    for (int kb = 0; kb < kb_total; ++kb) {
                        if (!mbar_wait(empty + stage, phase ^ 1u, plan.status, plan.wait_ns) || *abort_flag) {
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                        uint8_t* sa = smem + stage * kStageBytes2;
                        uint8_t* sb = sa + kATileBytes2;
                        const uint32_t bar = mapa_shared(smem_addr(full + stage), 0);
                        if (leader) mbar_arrive_expect_tx(full + stage, 2 * kStageBytes2);
                        const int pass = kb / plan.kb_per_pass;
                        const int kx = (kb - pass * plan.kb_per_pass) * kBK;
                        const int m0 = (c.m_blk * 2 + static_cast<int>(rank)) * kBM;
                        const int n0 = nb * kBN + static_cast<int>(rank) * (kBN / 2);
                        const CUtensorMap* ma = pass ? &tmA2 : &tmA;
                        if (plan.a_mn) {   // [K, M] storage: two 64 x 64 boxes, M contiguous
                            tma_load_2d_pair(ma, bar, sa, m0, kx);
                            tma_load_2d_pair(ma, bar, sa + 8192, m0 + 64, kx);
                        } else {
                            tma_load_2d_pair(ma, bar, sa, kx, m0);
                        }
                        if (plan.b_mn) {
                            tma_load_2d_pair(&tmB, bar, sb, n0, kx);
                            tma_load_2d_pair(&tmB, bar, sb + 8192, n0 + 64, kx);
                        } else {
                            tma_load_2d_pair(&tmB, bar, sb, kx, n0);
                        }
                        issued = true;
                        if (++stage == kStages2) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            if (!ok && issued) {
                // copies in flight signal the even CTA; give them time to land
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 200000ull) {
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------- MMA issuer (even CTA) ----------------
            uint32_t stage = 0, phase = 0, abuf = 0, aphase = 0;
            bool ok = true;
            bool any = false;
            const uint32_t idesc = kIdesc2 | (plan.a_mn ? (1u << 15) : 0u) | (plan.b_mn ? (1u << 16) : 0u);
            for (int u = pair; u < plan.num_units && ok; u += npairs) {
                const UnitCoords c = decode_unit(plan, u);
                for (int nb = c.nb_begin; nb < c.nb_end && ok; ++nb) {
                    if (!mbar_wait(acce + abuf, aphase ^ 1u, plan.status, plan.wait_ns) || *abort_flag) {
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + abuf * kBN;
                    for (int kb = 0; kb < kb_total; ++kb) {
                        if (!mbar_wait(full + stage, phase, plan.status, plan.wait_ns) || *abort_flag) {
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sa = smem_addr(smem + stage * kStageBytes2);
                        const uint32_t sb = sa + kATileBytes2;
#pragma unroll
                        for (int k = 0; k < kBK / 16; ++k) {
                            const uint64_t da = plan.a_mn ? sdesc_mnmajor_sw128(sa + k * 2048, 8192)
                                                          : sdesc_kmajor_sw128(sa + k * 32);
                            const uint64_t db = plan.b_mn ? sdesc_mnmajor_sw128(sb + k * 2048, 8192)
                                                          : sdesc_kmajor_sw128(sb + k * 32);
                            umma_bf16_pair(d_tmem, da, db, idesc, (kb | k) != 0 ? 1u : 0u);
                        }
                        any = true;
                        umma_commit_pair_multicast(empty + stage, 0x3);
                        if (++stage == kStages2) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    umma_commit_pair_multicast(accf + abuf, 0x3);
                    abuf ^= 1u;
                    if (abuf == 0) aphase ^= 1u;
                }
            }
            if (any) {
                // the MMAs must be done before either CTA releases TMEM or its stages, also
                // after a normal end of the loop (an epilogue may have given up its waits)
                umma_commit_pair_multicast(done_bar, 0x1);
                mbar_wait(done_bar, 0, plan.status);
            }
        }
    } else {
        // ---------------- epilogue (warps 2..9, both CTAs) ----------------
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int row = quarter * 32 + lane;
        uint8_t* my_stage = epi_stage + (warp - 2) * kEpiStageBytes;
        uint32_t abuf = 0, aphase = 0;
        bool ok = true;
        for (int u = pair; u < plan.num_units && ok; u += npairs) {
            const UnitCoords c = decode_unit(plan, u);
            Epi epi;
            const int m_blk = c.m_blk * 2 + static_cast<int>(rank);
            epi.begin_unit(ep, row, half, m_blk, c.split, c.nb_begin * kBN + half * (kBN / 2));
            for (int nb = c.nb_begin; nb < c.nb_end; ++nb) {
                if (!mbar_wait(accf + abuf, aphase, plan.status, plan.wait_ns) || *abort_flag) {
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + abuf * kBN;
#pragma unroll 1
                for (int ch = half * (kBN / 64); ch < (half + 1) * (kBN / 64); ++ch) {
                    uint32_t acc[32];
                    __syncwarp();
                    tmem_load_row32(taddr + ch * 32, acc);
                    epi.chunk(ep, acc, nb * kBN + ch * 32, my_stage, lane);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_addr(acce + abuf), 0));
                abuf ^= 1u;
                if (abuf == 0) aphase ^= 1u;
            }
            if (ok) epi.end_unit(ep, c.split, half);
        }
        if (lane == 0) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();   // no CTA leaves while its peer may still signal or read it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

// Launch gemm_tc2_kernel<Epi> as clusters of two CTAs.  tmB must have 128-row boxes.
template <class Epi>
int launch_gemm_pair(const CUtensorMap& tmA, const CUtensorMap& tmA2, const CUtensorMap& tmB,
                     const GemmPlan& plan, const typename Epi::Params& ep, cudaStream_t stream) {
    if (cudaFuncSetAttribute(gemm_tc2_kernel<Epi>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kGemmSmemBytes2) != cudaSuccess)
        return RL_ERR_CUDA;
    if (plan.num_units <= 0) return RL_OK;
    const int max_pairs = num_sms() / 2;
    const int pairs = plan.num_units < max_pairs ? plan.num_units : max_pairs;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = kGemmSmemBytes2;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, gemm_tc2_kernel<Epi>, tmA, tmA2, tmB, plan, ep) != cudaSuccess)
        return RL_ERR_CUDA;
    return cudaPeekAtLastError() == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}

// The B operand's tensor map for the kernel the current mode runs (128-row boxes for the
// pair kernel, 256-row boxes otherwise), and the matching dispatch.
inline int make_tmap_b(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld) {
    return make_tmap_bf16(map, base, rows, cols, ld, gemm_pair_mode() ? kBN / 2 : kBN);
}
inline GemmPlan make_plan_auto(int64_t M, int64_t N, int64_t K, int passes, int n_splits, int m_fastest,
                               int32_t* status, int a_mn = 0) {
    return make_plan(M, N, K, passes, n_splits, m_fastest, status, a_mn, 0, gemm_pair_mode());
}
template <class Epi>
int launch_gemm_auto(const CUtensorMap& tmA, const CUtensorMap& tmA2, const CUtensorMap& tmB,
                     const GemmPlan& plan, const typename Epi::Params& ep, cudaStream_t stream) {
    return gemm_pair_mode() ? launch_gemm_pair<Epi>(tmA, tmA2, tmB, plan, ep, stream)
                            : launch_gemm<Epi>(tmA, tmA2, tmB, plan, ep, stream);
}

}  // namespace rl
