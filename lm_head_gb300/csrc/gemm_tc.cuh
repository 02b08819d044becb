// Persistent warp-specialised tcgen05 GEMM for sm_100-family GPUs:
//
//   D[M, N] = A[M, K] * B[N, K]^T        (bf16 x bf16 -> fp32)
//
// Each operand is K-major (stored [M, K] / [N, K], K contiguous) or MN-major (stored
// [K, M] / [K, N], M or N contiguous): the transpose bits of the instruction descriptor
// and the shared-memory descriptors follow the layout, so no operand is ever transposed
// in memory.
//
// * warp 0, one lane: TMA producer.  Stages A (128 x 64) and B (256 x 64) tiles with the
//   128-byte swizzle into a 4-deep shared-memory ring; completion on per-stage mbarriers.
// * warp 1, one lane: MMA issuer.  Four tcgen05.mma (M=128, N=256, K=16) per stage into a
//   TMEM accumulator; tcgen05.commit frees the stage and, after the last K block of a
//   tile, hands the accumulator to the epilogue.  Two 256-column accumulators (all 512
//   TMEM columns) let the epilogue of tile i overlap the MMAs of tile i+1.
// * warps 2-9: epilogue.  Warp w reads TMEM lanes 32*(w%4) .. +31 and one half of the
//   tile's columns (warps 2-5 the first 128, warps 6-9 the last 128), so each row of the
//   tile is owned by two threads that see 128 columns each, in four 32-column chunks.
//   Two epilogue warps per scheduler keep the epilogue off the MMA's critical path.  The
//   epilogue policy (template parameter) decides what a row does with its columns.
//
// Work is split into "units": one 128-row block of A times a contiguous range of 256-col
// tiles of B.  CTAs take units round-robin (grid = min(units, SMs)).  A unit's tiles are
// processed in order by one CTA, so a policy can carry per-row state across the range
// (the online logsumexp of the LM-head forward does).
//
// Every mbarrier wait is bounded (plan.wait_ns); a wait that runs out sets
// RL_STATUS_TIMEOUT, raises a CTA-wide abort flag, and all roles unwind, wait for their
// own copies / MMAs in flight (bounded again, by the fixed kWaitLimitNs), and release
// TMEM.  The MMA issuer waits for its last MMAs before TMEM is released whether or not it
// aborted itself: an epilogue that gave up no longer proves the accumulators are done.
#pragma once

#include "common.cuh"

namespace rl {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kATileBytes = kBM * kBK * 2;   // 16 KB
constexpr int kBTileBytes = kBN * kBK * 2;   // 32 KB
constexpr int kStageBytes = kATileBytes + kBTileBytes;
constexpr int kEpiWarps = 8;
constexpr int kGemmThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t kTmemCols = 512;
// Per epilogue warp: 4 KB of shared memory to stage tiles for TMA stores.
constexpr int kEpiStageBytes = 4096;
constexpr int kGemmSmemBytes = kStages * kStageBytes + kEpiWarps * kEpiStageBytes + 1024 + 256;
constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBN);

struct GemmPlan {
    int m_blocks;        // ceil(M / 128)
    int n_blocks;        // ceil(N / 256)
    int tiles_per_unit;  // B tiles per unit
    int n_splits;        // ceil(n_blocks / tiles_per_unit)
    int num_units;       // m_blocks * n_splits
    int m_fastest;       // 1: u -> (m = u % m_blocks, s = u / m_blocks); 0: (m = u / n_splits, s = u % n_splits)
    int kb_per_pass;     // ceil(K / 64)
    int passes;          // 1; 2 when A comes as a hi/lo pair (tmA then tmA2, same B)
    int a_mn;            // A stored [K, M] (MN-major): tensor map over [K, M], 64 x 64 boxes
    int b_mn;            // B stored [K, N]
    int32_t* status;
    uint64_t wait_ns;    // limit of the work loops' waits (RL_OPT_WAIT_LIMIT_US)
};

struct UnitCoords {
    int m_blk, split, nb_begin, nb_end;
};

RL_DEVINL UnitCoords decode_unit(const GemmPlan& p, int u) {
    UnitCoords c;
    if (p.m_fastest) {
        c.m_blk = u % p.m_blocks;
        c.split = u / p.m_blocks;
    } else {
        c.m_blk = u / p.n_splits;
        c.split = u % p.n_splits;
    }
    c.nb_begin = c.split * p.tiles_per_unit;
    c.nb_end = min(p.n_blocks, c.nb_begin + p.tiles_per_unit);
    return c;
}

// tcgen05.ld of 32 columns followed by the wait, with the registers threaded through the
// wait so no use can be scheduled before the data has landed.
RL_DEVINL void tmem_load_row32(uint32_t taddr, uint32_t (&r)[32]) {
    tmem_ld_32x32(taddr, r);
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// An epilogue policy may carry `const int* gate` in its Params: the launch then does no work
// unless *gate != 0, a decision an earlier kernel of the stream wrote to device memory.
template <class P>
RL_DEVINL auto epi_gate_open(const P& p, int) -> decltype(p.gate, bool()) {
    return p.gate == nullptr || *p.gate != 0;
}
template <class P>
RL_DEVINL bool epi_gate_open(const P&, long) {
    return true;
}

// Epilogue policy interface (all device, per thread; `row` in [0, 128), `half` 0/1 says
// which 128 columns of every 256-column tile this thread sees; `col_begin` is the first
// column it will see in the unit; `stage` is the warp's kEpiStageBytes of shared memory
// for TMA stores, `lane` the thread's lane; chunk() is entered by all 32 lanes together):
//   struct Epi {
//     struct Params { ... };
//     __device__ void begin_unit(const Params&, int row, int half, int m_blk, int split, int col_begin);
//     __device__ void chunk(const Params&, const uint32_t (&acc)[32], int col0, uint8_t* stage, int lane);
//     __device__ void end_unit(const Params&, int split, int half);
//   };
template <class Epi>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                   const __grid_constant__ CUtensorMap tmB, const GemmPlan plan,
                   const __grid_constant__ typename Epi::Params ep) {
    if (!epi_gate_open(ep, 0)) return;   // uniform over the grid
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* epi_stage = smem + kStages * kStageBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(epi_stage + kEpiWarps * kEpiStageBytes);
    uint64_t* empty = full + kStages;
    uint64_t* accf = empty + kStages;
    uint64_t* acce = accf + 2;
    uint64_t* done_bar = acce + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf + b, 1);
            mbar_init(acce + b, kEpiWarps);
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
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int kb_total = plan.kb_per_pass * plan.passes;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            uint32_t stage = 0, phase = 0;
            uint32_t armed_parity[kStages];
            bool armed[kStages];
#pragma unroll
            for (int s = 0; s < kStages; ++s) {
                armed[s] = false;
                armed_parity[s] = 0;
            }
            bool ok = true;
            for (int u = blockIdx.x; u < plan.num_units && ok; u += gridDim.x) {
                const UnitCoords c = decode_unit(plan, u);
                for (int nb = c.nb_begin; nb < c.nb_end && ok; ++nb) {
                    for (int kb = 0; kb < kb_total; ++kb) {
                        if (!mbar_wait(empty + stage, phase ^ 1u, plan.status, plan.wait_ns) || *abort_flag) {
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                        uint8_t* sa = smem + stage * kStageBytes;
                        uint8_t* sb = sa + kATileBytes;
                        mbar_arrive_expect_tx(full + stage, kStageBytes);
                        armed[stage] = true;
                        armed_parity[stage] = phase;
                        const int pass = kb / plan.kb_per_pass;
                        const int kx = (kb - pass * plan.kb_per_pass) * kBK;
                        const CUtensorMap* ma = pass ? &tmA2 : &tmA;
                        if (plan.a_mn) {
#pragma unroll
                            for (int i = 0; i < kBM / 64; ++i)
                                tma_load_2d(ma, full + stage, sa + i * 8192, c.m_blk * kBM + 64 * i, kx);
                        } else {
                            tma_load_2d(ma, full + stage, sa, kx, c.m_blk * kBM);
                        }
                        if (plan.b_mn) {
#pragma unroll
                            for (int i = 0; i < kBN / 64; ++i)
                                tma_load_2d(&tmB, full + stage, sb + i * 8192, nb * kBN + 64 * i, kx);
                        } else {
                            tma_load_2d(&tmB, full + stage, sb, kx, nb * kBN);
                        }
                        if (++stage == kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            if (!ok) {
                // Let every copy this thread issued land before the CTA can exit.
                for (int s = 0; s < kStages; ++s)
                    if (armed[s]) mbar_wait(full + s, armed_parity[s], plan.status);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            uint32_t stage = 0, phase = 0, abuf = 0, aphase = 0;
            bool ok = true;
            bool issued = false;
            const uint32_t idesc = kIdesc | (plan.a_mn ? (1u << 15) : 0u) | (plan.b_mn ? (1u << 16) : 0u);
            for (int u = blockIdx.x; u < plan.num_units && ok; u += gridDim.x) {
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
                        const uint32_t sa = smem_addr(smem + stage * kStageBytes);
                        const uint32_t sb = sa + kATileBytes;
#pragma unroll
                        for (int k = 0; k < kBK / 16; ++k) {
                            const uint64_t da = plan.a_mn ? sdesc_mnmajor_sw128(sa + k * 2048, 8192)
                                                          : sdesc_kmajor_sw128(sa + k * 32);
                            const uint64_t db = plan.b_mn ? sdesc_mnmajor_sw128(sb + k * 2048, 8192)
                                                          : sdesc_kmajor_sw128(sb + k * 32);
                            umma_bf16(d_tmem, da, db, idesc, (kb | k) != 0 ? 1u : 0u);
                        }
                        issued = true;
                        umma_commit(empty + stage);
                        if (++stage == kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    umma_commit(accf + abuf);
                    abuf ^= 1u;
                    if (abuf == 0) aphase ^= 1u;
                }
            }
            if (issued) {
                // Every MMA issued so far must finish before TMEM is released (also after a
                // normal end of the loop: the epilogue may have given up on its waits).
                umma_commit(done_bar);
                mbar_wait(done_bar, 0, plan.status);
            }
        }
    } else {
        // ---------------- epilogue (warps 2..9) ----------------
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int row = quarter * 32 + lane;
        uint8_t* my_stage = epi_stage + (warp - 2) * kEpiStageBytes;
        uint32_t abuf = 0, aphase = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < plan.num_units && ok; u += gridDim.x) {
            const UnitCoords c = decode_unit(plan, u);
            Epi epi;
            epi.begin_unit(ep, row, half, c.m_blk, c.split, c.nb_begin * kBN + half * (kBN / 2));
            for (int nb = c.nb_begin; nb < c.nb_end; ++nb) {
                if (!mbar_wait(accf + abuf, aphase, plan.status, plan.wait_ns) || *abort_flag) {
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                       abuf * kBN;
#pragma unroll 1
                for (int ch = half * (kBN / 64); ch < (half + 1) * (kBN / 64); ++ch) {
                    uint32_t acc[32];
                    __syncwarp();
                    tmem_load_row32(taddr + ch * 32, acc);
                    epi.chunk(ep, acc, nb * kBN + ch * 32, my_stage, lane);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acce + abuf);
                abuf ^= 1u;
                if (abuf == 0) aphase ^= 1u;
            }
            if (ok) epi.end_unit(ep, c.split, half);
        }
        if (lane == 0) bulk_wait_all();   // every TMA store of this warp has landed
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------
// 2-D bf16 tensor map over a row-major [rows, cols] matrix with row stride `ld` elements,
// box = box_rows x 64 columns, 128-byte swizzle, zero fill out of bounds.
int make_tmap_bf16(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld,
                   int box_rows);

// General 2-D tensor map: [rows, cols] with row stride `ld` elements, box box_rows x box_cols,
// swizzle_bytes 0 (none), 64 or 128.
int make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int elem_bytes, int64_t rows,
                 int64_t cols, int64_t ld, int box_cols, int box_rows, int swizzle_bytes);

int num_sms();
uint64_t wait_limit_ns();

// pair = 1: m_blocks counts 256-row blocks of the two-CTA kernel.
GemmPlan make_plan(int64_t M, int64_t N, int64_t K, int passes, int n_splits, int m_fastest,
                   int32_t* status, int a_mn = 0, int b_mn = 0, int pair = 0);
int gemm_pair_mode();

// Launch `gemm_tc_kernel<Epi>`; A2 may equal A when passes == 1.
template <class Epi>
int launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmA2, const CUtensorMap& tmB,
                const GemmPlan& plan, const typename Epi::Params& ep, cudaStream_t stream) {
    if (cudaFuncSetAttribute(gemm_tc_kernel<Epi>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kGemmSmemBytes) != cudaSuccess)
        return RL_ERR_CUDA;
    if (plan.num_units <= 0) return RL_OK;
    const int grid = plan.num_units < num_sms() ? plan.num_units : num_sms();
    gemm_tc_kernel<Epi><<<grid, kGemmThreads, kGemmSmemBytes, stream>>>(tmA, tmA2, tmB, plan, ep);
    return cudaPeekAtLastError() == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}

}  // namespace rl
