// attn_bwd_sm103.cu — bf16 attention backward on the sm_103a tensor cores.
//
// The backward pass recomputes the score and probability tiles from Q, K, V,
// the saved per-row log-sum-exp and D = rowsum(dO * O), instead of storing
// the N x N probabilities ("What is FlashAttention?", Step 4; "FlashAttention",
// "What it does not do"). Per (b, h) the gradients are the textbook ones:
//     P = exp(scale * Q K^T + mask - LSE),   dV = P^T dO,   dP = dO V^T,
//     dS = P * (dP - D),   dK = scale * dS^T Q,   dQ = scale * dS K.
//
// One CTA owns a 128-key tile of one (b, h) and keeps K, V and the fp32 dK,
// dV accumulators on chip while 128-query tiles stream past (query tiles that
// lie entirely above the causal diagonal are never visited). Per query tile:
//   S^T = K Q^T and dP^T = V dO^T      (tcgen05, both operands in shared memory)
//   P^T, dS^T (one thread per key row)  bf16 into tensor memory, dS also into
//                                      shared memory (swizzled, query-contiguous)
//   dV += P^T dO, dK += dS^T Q         (tcgen05, A operand in tensor memory)
//   dQ_tile = dS K                     (tcgen05, A = dS read query-major)
// and the warpgroups stage scale * dQ_tile in shared memory, from where a TMA
// reduce-add puts it into the fp32 dQ accumulator in global memory (other key
// tiles add to the same rows).
//
// Warp roles (12 warps):
//   warps 0-7   two warpgroups; warpgroup g builds P^T / dS^T for query
//               columns [64 g, 64 g + 64) of each tile (thread = key row),
//               then stages its half of the dQ tile's columns (thread = query
//               row); at the end warpgroup 0 writes dV and warpgroup 1 dK
//   warp  8     TMA producer: K and V once, then per query tile Q_i, dO_i, the
//               mask tile and the tile's -LSE*log2(e) and -D statistics (1 KB,
//               written tile-padded by the pre-pass)
//   warp  9     TMEM allocator and MMA issuer
//   warp 10     issues the TMA reduce-add of each staged dQ tile
//   warp 11     idle
//
// Tensor memory (512 columns, lane = key row for S^T/dP^T/dK/dV, query row for dQ):
//   [0,128)    S^T fp32; P^T bf16 pairs in [0,32) and [64,96) (see packed_col)
//   [128,256)  dP^T fp32; dS^T bf16 pairs in [128,160) and [192,224);
//              then the dQ tile
//   [256,256+D)      dV accumulator
//   [256+D,256+2D)   dK accumulator
// The dQ MMAs overwrite packed dS^T columns, and the next tile's S^T MMAs packed P^T
// columns, only after the dV / dK MMAs that read them: tcgen05 MMAs issued by one thread
// execute in order. So the next tile's S^T runs while the warpgroups read the dQ tile out
// of tensor memory; only its dP^T waits for them.
//
// S^T and dP^T complete separately, so the warpgroups compute the first chunk's P^T while
// the dP^T product runs. They hand over P^T / dS^T in two steps, one per 32-query chunk each
// of them has packed, and the dV / dK products of the first chunks run while the second ones
// are computed.
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

using namespace ptx;

constexpr int BQ = 128;  // query rows per tile
constexpr int BK = 128;  // key rows per CTA

template <int D, bool MASK>
struct BwdCfg {
    static constexpr int kBoxes = D / 64;
    static constexpr int kTileBytes = 128 * D * 2;
    static constexpr int kMaskBytes = BQ * BK * 2;
    static constexpr int kStages = (D == 128 && MASK) ? 1 : 2;
    static constexpr int kVecOffInStage = 2 * kTileBytes + (MASK ? kMaskBytes : 0);
    static constexpr int kStageBytes = kVecOffInStage + 1024;  // + [-LSE*log2e | D] x 128
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kKOff + kTileBytes;
    static constexpr int kDSOff = kVOff + kTileBytes;
    static constexpr int kStageOff = kDSOff + BQ * BK * 2;
    // one stage: a separate area that holds half a dQ tile (one warpgroup's columns) at a time
    static constexpr int kStgOff = kStageOff + kStages * kStageBytes;
    static constexpr int kStgBytes = kStages == 1 ? BQ * (D / 2) * 4 : 0;
    static constexpr int kBarOff = kStgOff + kStgBytes;
    static constexpr int kSmemBytes = kBarOff + 256;
};

struct BwdParamsDev {
    int B, H, N;
    int causal;
    float c;      // scale * log2(e)
    float scale;
    const float* stats;  // [B*H][nq][2][128]: -LSE*log2e, then -D
    float* dq_acc;
    __nv_bfloat16 *dk, *dv;
    long long dk_sb, dk_sh, dk_sn, dv_sb, dv_sh, dv_sn;
    int mask_hb, mask_bb;
    int n_ktiles;
    int num_units;  // persistent d = 64 kernel: key tiles x heads
    int* err;
    unsigned long long timeout_ns;
};

struct __align__(8) BwdBarriers {
    uint64_t kv_full;
    uint64_t st_full[2], st_empty[2];  // per stage: Q, the statistics (and the mask tile)
    uint64_t do_full[2], do_empty[2];  // per stage: dO
    uint64_t s_full, dp_full, dq_full, dq_empty, kv_done;  // s_full: S^T done; dp_full: dP^T done
    uint64_t dv_done;  // the tile's last dV products (the last readers of its dO) done
    uint64_t ds_ready[2];   // P^T / dS^T of chunk step cc (query chunks cc and 2 + cc) packed
    uint64_t dq_staged[2][2];  // two stages: per stage and warpgroup, its half of the dQ tile staged in
                               // the stage's Q (warpgroup 0) or dO (warpgroup 1) area for the TMA
                               // reduction; one stage: [0][0] a warpgroup's half in the separate area
    uint64_t stg_free;      // one stage: the separate area read by the last reduction
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk) {
    return sdesc_sw128(tile + (kk >> 2) * (128 * 128) + (kk & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t tile, int kk) {
    return sdesc_sw128(tile + kk * (16 * 128), 128 * 128, 1024);
}
// TMEM column (relative to the S^T or dP^T region) of the bf16 pairs for
// query chunk c (32 queries): each warpgroup packs its results into the
// first half of the 64 fp32 columns it has itself already read, never into
// columns the other warpgroup may still be reading.
__host__ __device__ constexpr int packed_col(int c) { return 64 * (c >> 1) + 16 * (c & 1); }
// ... and of the 16 queries of MMA k-step kk.
__host__ __device__ constexpr int packed_col_k(int kk) { return packed_col(kk >> 1) + 8 * (kk & 1); }

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(a, parity))
        if (globaltimer() - t0 > timeout_ns) break;
}

template <int D, bool MASK, bool F16>
__global__ void __launch_bounds__(384, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_mask, const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
                  const __grid_constant__ CUtensorMap tm_dv,
                  const BwdParamsDev p) {
    using Cfg = BwdCfg<D, MASK>;
    // 16-bit element type of the operands and of P^T, dS^T: bf16, or IEEE half when F16
    constexpr uint32_t kIdescS = idesc_h16(BK, BQ, false, false, F16);  // S^T, dP^T
    constexpr uint32_t kIdescKV = idesc_h16(BK, D, false, true, F16);   // dV, dK (A in TMEM)
    constexpr uint32_t kIdescQ = idesc_h16(BQ, D, true, true, F16);     // dQ (A = dS query-major)
    // dQ leaves through shared memory and TMA reductions. With two stages the current
    // stage's Q/dO area holds the whole tile (the next tile's operands sit in the other
    // stage); with one stage, staging there would hold up the next tile's load, so the
    // two warpgroups take turns with a separate half-tile area.
    constexpr bool kStageDq = Cfg::kStages > 1;
    static_assert(!kStageDq || 2 * Cfg::kTileBytes >= BQ * D * 4, "dQ staging fits in a stage");
    extern __shared__ __align__(1024) uint8_t smem[];
    BwdBarriers& bar = *reinterpret_cast<BwdBarriers*>(smem + Cfg::kBarOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    WaitCtl wc{p.err, &bar.abort_flag, p.timeout_ns};

    // work unit: key tile kt of (b, h). Heads outermost, so the CTAs resident at any time
    // work on one or two heads and their dQ reductions and Q / dO reads stay in L2; within a
    // head early key tiles first (under causal masking they see the most query tiles).
    const int kt = blockIdx.x % p.n_ktiles;
    const int bh_i = blockIdx.x / p.n_ktiles;
    const int b = bh_i / p.H, h = bh_i % p.H;
    const int k0 = kt * BK;
    const int nq_all = (p.N + BQ - 1) / BQ;
    const int i_begin = p.causal ? kt : 0;  // first query tile on or below the diagonal
    const int n_it = nq_all - i_begin;

    if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled tiles need a 1024-byte aligned base
        if (threadIdx.x == 0) atomicExch(p.err, -7);
        return;
    }
    if (threadIdx.x == 0) {
        bar.abort_flag = 0;
        mbar_init(&bar.kv_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar.st_full[s], 1);
            mbar_init(&bar.do_full[s], 1);
            // with two stages a stage is also the dQ staging area: its Q and dO areas are free
            // after the tile's MMAs and after the TMA reduction has read the half staged there
            mbar_init(&bar.st_empty[s], kStageDq ? 2 : 1);
            mbar_init(&bar.do_empty[s], kStageDq ? 2 : 1);
            mbar_init(&bar.dq_staged[s][0], 128);
            mbar_init(&bar.dq_staged[s][1], 128);
        }
        mbar_init(&bar.stg_free, 1);
        mbar_init(&bar.s_full, 1);
        mbar_init(&bar.dp_full, 1);
        mbar_init(&bar.dv_done, 1);
        mbar_init(&bar.ds_ready[0], 256);
        mbar_init(&bar.ds_ready[1], 256);
        mbar_init(&bar.dq_full, 1);
        mbar_init(&bar.dq_empty, 256);
        mbar_init(&bar.kv_done, 1);
        mbar_init(&bar.drain, 1);
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(&bar.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // No global memory is touched above: from here on the pre-pass must be complete.
    grid_dep_launch();
    grid_dep_wait();
    const uint32_t tmem = bar.tmem_base;
    const uint32_t sK = smem_u32(smem + Cfg::kKOff), sV = smem_u32(smem + Cfg::kVOff);
    const uint32_t sDS = smem_u32(smem + Cfg::kDSOff);

    if (warp == 8) {
        // ------------------------------------------------ producer
        // The whole warp walks the schedule and waits; one elected lane issues the copies.
        if (elect_one()) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_do);
            mbar_arrive_expect_tx(&bar.kv_full, 2 * Cfg::kTileBytes);
            for (int bx = 0; bx < Cfg::kBoxes; ++bx) {
                tma_load_4d(smem + Cfg::kKOff + bx * 128 * 128, &tm_k, &bar.kv_full, bx * 64, k0, h, b);
                tma_load_4d(smem + Cfg::kVOff + bx * 128 * 128, &tm_v, &bar.kv_full, bx * 64, k0, h, b);
            }
        }
        __syncwarp();
        const int hm = p.mask_hb ? h : 0, bm = p.mask_bb ? b : 0;
        bool ok = true;
        int it = 0;
        for (; it < n_it && ok; ++it) {
            const int s = it % Cfg::kStages;
            ok = mbar_wait_warp(&bar.st_empty[s], ((it / Cfg::kStages) & 1) ^ 1, wc);
            if (!ok) break;
            const int q0 = (i_begin + it) * BQ;
            uint8_t* st = smem + Cfg::kStageOff + s * Cfg::kStageBytes;
            if (elect_one()) {
                mbar_arrive_expect_tx(&bar.st_full[s], Cfg::kStageBytes - Cfg::kTileBytes);
                for (int bx = 0; bx < Cfg::kBoxes; ++bx)
                    tma_load_4d(st + bx * 128 * 128, &tm_q, &bar.st_full[s], bx * 64, q0, h, b);
                if (MASK)
                    for (int bx = 0; bx < 2; ++bx)
                        tma_load_4d(st + 2 * Cfg::kTileBytes + bx * 128 * 128, &tm_mask, &bar.st_full[s],
                                    k0 + bx * 64, q0, hm, bm);
                bulk_load(st + Cfg::kVecOffInStage,
                          p.stats + ((long long)(b * p.H + h) * nq_all + (i_begin + it)) * 256, 1024,
                          &bar.st_full[s]);
            }
            __syncwarp();
            // dO: its area may be freed later than Q's (the dQ half staged there is reduced second)
            ok = mbar_wait_warp(&bar.do_empty[s], ((it / Cfg::kStages) & 1) ^ 1, wc);
            if (!ok) break;
            if (elect_one()) {
                mbar_arrive_expect_tx(&bar.do_full[s], Cfg::kTileBytes);
                for (int bx = 0; bx < Cfg::kBoxes; ++bx)
                    tma_load_4d(st + Cfg::kTileBytes + bx * 128 * 128, &tm_do, &bar.do_full[s], bx * 64, q0, h, b);
            }
            __syncwarp();
        }
        if (lane == 0) {
            const int last = it < Cfg::kStages ? it : Cfg::kStages;
            for (int i = it - last; i < it; ++i) {
                drain_wait(&bar.st_full[i % Cfg::kStages], (i / Cfg::kStages) & 1, p.timeout_ns);
                drain_wait(&bar.do_full[i % Cfg::kStages], (i / Cfg::kStages) & 1, p.timeout_ns);
            }
            drain_wait(&bar.kv_full, 0, p.timeout_ns);
        }
    } else if (warp == 9) {
        // ------------------------------------------------ MMA issuer
        // Converged warp; one elected lane (always the same one) issues MMAs and commits.
        bool ok = mbar_wait_warp(&bar.kv_full, 0, wc);
        tc_fence_after();
        for (int it = 0; it < n_it && ok; ++it) {
            const int s = it % Cfg::kStages;
            ok = mbar_wait_warp(&bar.st_full[s], (it / Cfg::kStages) & 1, wc);
            if (!ok) break;
            tc_fence_after();
            const uint32_t sQ = smem_u32(smem + Cfg::kStageOff + s * Cfg::kStageBytes);
            const uint32_t sdO = sQ + Cfg::kTileBytes;
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + 0, kmajor_desc(sK, kk), kmajor_desc(sQ, kk), kIdescS, kk > 0 ? 1u : 0u);
                mma_commit(&bar.s_full);
            }
            __syncwarp();
            if (it > 0) {  // dP^T overwrites the previous dQ tile
                ok = mbar_wait_warp(&bar.dq_empty, (it - 1) & 1, wc);
                if (!ok) break;
            }
            ok = mbar_wait_warp(&bar.do_full[s], (it / Cfg::kStages) & 1, wc);
            if (!ok) break;
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + 128, kmajor_desc(sV, kk), kmajor_desc(sdO, kk), kIdescS, kk > 0 ? 1u : 0u);
                mma_commit(&bar.dp_full);
            }
            __syncwarp();
            // dV += P^T dO and dK += dS^T Q, 16 queries per k-step: chunk step cc brings the
            // k-steps of query chunks cc and 2 + cc (2 k-steps each)
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                ok = mbar_wait_warp(&bar.ds_ready[cc], it & 1, wc);
                if (!ok) break;
                tc_fence_after();
                if (elect_one()) {
                    // the second chunks' dV products run after dQ (below), so that the dQ
                    // tile's drain overlaps products that read only one operand from shared memory
                    if (cc == 0) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int kk = 4 * (j >> 1) + (j & 1);
                            mma_ts(tmem + 256, tmem + packed_col_k(kk), mnmajor_desc(sdO, kk), kIdescKV,
                                   (it > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int kk = 4 * (j >> 1) + 2 * cc + (j & 1);
                        mma_ts(tmem + 256 + D, tmem + 128 + packed_col_k(kk), mnmajor_desc(sQ, kk), kIdescKV,
                               (it > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                __syncwarp();
            }
            if (!ok) break;
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)  // N = D: K read head-dim-major across its 64-column boxes
                    mma_ss(tmem + 128, mnmajor_desc(sDS, kk), mnmajor_desc(sK, kk), kIdescQ, kk > 0 ? 1u : 0u);
                mma_commit(&bar.dq_full);
                mma_commit(&bar.st_empty[s]);
                // dV of the second chunks (P^T stays in the S^T columns, which dQ does not touch)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int kk = 4 * (j >> 1) + 2 + (j & 1);
                    mma_ts(tmem + 256, tmem + packed_col_k(kk), mnmajor_desc(sdO, kk), kIdescKV, 1u);
                }
                mma_commit(&bar.dv_done);
                mma_commit(&bar.do_empty[s]);
            }
            __syncwarp();
        }
        if (elect_one()) {
            if (ok) mma_commit(&bar.kv_done);
            mma_commit(&bar.drain);
            drain_wait(&bar.drain, 0, p.timeout_ns);
        }
        __syncwarp();
    } else if (warp == 10) {
        // ------------------------------------------------ dQ reductions
        // Once a dQ tile (two stages) or one warpgroup's half of it (one stage) is
        // staged (fp32, in the accumulator map's 32-column boxes with the 128-byte
        // swizzle), one lane adds the boxes into the accumulator with TMA and frees
        // the staging area: the tile's stage, or the separate area. Rows beyond N
        // are clipped by the tensor map.
        if (lane == 0) {
            prefetch_tmap(&tm_dq);
            bool ok = true;
            for (int it = 0; it < n_it && ok; ++it) {
                const int q0 = (i_begin + it) * BQ;
                if constexpr (kStageDq) {
                    // warpgroup 0's half (Q area) first: the next load into the stage is Q's
                    const int s = it % Cfg::kStages;
                    const uint8_t* stg = smem + Cfg::kStageOff + s * Cfg::kStageBytes;
                    for (int g = 0; g < 2 && ok; ++g) {
                        ok = mbar_wait(&bar.dq_staged[s][g], (it / Cfg::kStages) & 1, wc);
                        if (!ok) break;
#pragma unroll
                        for (int bx = 0; bx < D / 64; ++bx)
                            tma_reduce_add_4d(&tm_dq, stg + (g * (D / 64) + bx) * (BQ * 128), g * (D / 2) + 32 * bx,
                                              q0, h, b);
                        bulk_commit();
                        bulk_wait_read0();
                        mbar_arrive(g == 0 ? &bar.st_empty[s] : &bar.do_empty[s]);
                    }
                } else {
                    for (int g = 0; g < 2 && ok; ++g) {  // staging use k = 2 it + g
                        ok = mbar_wait(&bar.dq_staged[0][0], g, wc);
                        if (!ok) break;
                        const uint8_t* stg = smem + Cfg::kStgOff;
#pragma unroll
                        for (int bx = 0; bx < D / 64; ++bx)
                            tma_reduce_add_4d(&tm_dq, stg + bx * (BQ * 128), g * (D / 2) + 32 * bx, q0, h, b);
                        bulk_commit();
                        bulk_wait_read0();
                        mbar_arrive(&bar.stg_free);
                    }
                }
            }
            bulk_wait0();  // reductions complete before the CTA exits
        }
    } else if (warp < 8) {
        // ------------------------------------------------ P^T, dS^T, then the dQ drain
        // Two warpgroups share each query tile: warpgroup g takes query columns
        // [64 g, 64 g + 64) of P^T / dS^T (thread = key row), then drains its half
        // of the dQ tile's columns (thread = query row).
        const int g = warp >> 2;
        const int kr = (warp & 3) * 32 + lane;
        const int kg = k0 + kr;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tRow = tmem + lane_off;
        uint8_t* ds_row = smem + Cfg::kDSOff + kr * 128;
        constexpr int kDqCols = D / 2;                                      // dQ columns per warpgroup
        const uint32_t tDq = tRow + 128 + kDqCols * g;                       // their TMEM columns
        const float2 c2 = make_float2(p.c, p.c);
        bool ok = true;
        for (int it = 0; it < n_it && ok; ++it) {
            const int q0 = (i_begin + it) * BQ;
            const int s = it % Cfg::kStages;
            ok = mbar_wait(&bar.s_full, it & 1, wc);
            // the stage's statistics (and mask tile) are visible once its copies completed
            ok = ok && mbar_wait(&bar.st_full[s], (it / Cfg::kStages) & 1, wc);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const uint8_t* stage = smem + Cfg::kStageOff + s * Cfg::kStageBytes;
            const float* nlv = reinterpret_cast<const float*>(stage + Cfg::kVecOffInStage);  // -LSE*log2e
            const float* ndv = nlv + 128;                                                   // -D
            tc_fence_after();
            const bool diag = p.causal && (q0 == k0);
            const bool key_ok = kg < p.N;
            const uint8_t* mt = stage + 2 * Cfg::kTileBytes;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int c = 2 * g + cc;  // 32-column chunk of the tile
                uint32_t sv[32];
                tmem_ld32(tRow + 32 * c, sv);
                tmem_wait_ld();
                float pr[32];
                uint32_t pk[16], dk[16];
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const int q = 32 * c + i;
                    const float2 nl = *reinterpret_cast<const float2*>(nlv + q);
                    float2 x = ffma2(make_float2(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])), c2, nl);
                    if (MASK) {
                        const int kb = kr >> 6, kc = (kr & 63) >> 3;
                        const float m0 = h16_to_float<F16>(*reinterpret_cast<const uint16_t*>(
                            mt + kb * 128 * 128 + q * 128 + ((kc ^ (q & 7)) << 4) + (kr & 7) * 2));
                        const float m1 = h16_to_float<F16>(*reinterpret_cast<const uint16_t*>(
                            mt + kb * 128 * 128 + (q + 1) * 128 + ((kc ^ ((q + 1) & 7)) << 4) + (kr & 7) * 2));
                        x = ffma2(make_float2(m0, m1), make_float2(kLog2e, kLog2e), x);
                    }
                    if (!key_ok || (diag && q < kr)) x.x = -INFINITY;
                    if (!key_ok || (diag && q + 1 < kr)) x.y = -INFINITY;
                    pr[i] = ex2(x.x);
                    pr[i + 1] = ex2(x.y);
                    pk[i / 2] = pack_h16<F16>(pr[i], pr[i + 1]);
                }
                tmem_st16(tRow + packed_col(c), pk);
                if (cc == 0) {  // the dP^T product runs while the first chunk's P^T is computed
                    ok = mbar_wait(&bar.dp_full, it & 1, wc);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    tc_fence_after();
                }
                uint32_t pv[32];
                tmem_ld32(tRow + 128 + 32 * c, pv);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const float2 nd = *reinterpret_cast<const float2*>(ndv + 32 * c + i);
                    const float2 ds = fmul2(make_float2(pr[i], pr[i + 1]),
                                            fadd2(make_float2(__uint_as_float(pv[i]), __uint_as_float(pv[i + 1])), nd));
                    dk[i / 2] = pack_h16<F16>(ds.x, ds.y);
                }
                tmem_st16(tRow + 128 + packed_col(c), dk);
                // dS row kr, queries 32c .. 32c+31 -> box (32c / 64), chunks ((32c % 64) / 8) .. +3
                uint8_t* box = ds_row + ((32 * c) >> 6) * (128 * 128);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int ch = ((32 * c) & 63) / 8 + j;
                    *reinterpret_cast<uint4*>(box + ((ch ^ (kr & 7)) << 4)) =
                        make_uint4(dk[4 * j], dk[4 * j + 1], dk[4 * j + 2], dk[4 * j + 3]);
                }
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&bar.ds_ready[cc]);
            }
            if (!ok) break;

            // dQ drain: this warpgroup's half of the columns of the dQ tile (thread = query row)
            ok = mbar_wait(&bar.dq_full, it & 1, wc);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            uint32_t v[kDqCols];
            tmem_ld32_at<0>(tDq, v);
            if constexpr (kDqCols == 64) tmem_ld32_at<32>(tDq + 32, v);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(&bar.dq_empty);
            // scale * dQ into the staging area: box bx (32 columns, 128 bytes per query row)
            // of this warpgroup's half. Two stages: this tile's stage holds both halves;
            // one stage: the separate area holds one half, warpgroup 0's first.
            uint8_t* stg;
            if constexpr (kStageDq) {
                stg = smem + Cfg::kStageOff + s * Cfg::kStageBytes + g * (kDqCols / 32) * (BQ * 128);
                if (g == 1) {  // the dO area: its last products (dV of the second chunks) follow dQ
                    ok = mbar_wait(&bar.dv_done, it & 1, wc);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                }
            } else {
                stg = smem + Cfg::kStgOff;
                const int k = 2 * it + g;  // staging use; wait for use k-1 to have been read
                if (k > 0) {
                    ok = mbar_wait(&bar.stg_free, (k - 1) & 1, wc);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                }
            }
#pragma unroll
            for (int bx = 0; bx < kDqCols / 32; ++bx) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const int col = 32 * bx + 4 * c;
                    const float2 a0 = fmul2(make_float2(__uint_as_float(v[col]), __uint_as_float(v[col + 1])),
                                            make_float2(p.scale, p.scale));
                    const float2 a1 = fmul2(make_float2(__uint_as_float(v[col + 2]), __uint_as_float(v[col + 3])),
                                            make_float2(p.scale, p.scale));
                    *reinterpret_cast<float4*>(stg + bx * (BQ * 128) + kr * 128 + ((c ^ (kr & 7)) << 4)) =
                        make_float4(a0.x, a0.y, a1.x, a1.y);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(kStageDq ? &bar.dq_staged[s][g] : &bar.dq_staged[0][0]);
        }
        // epilogue: warpgroup 0 writes the dV rows, warpgroup 1 the scale * dK rows of this key tile
        if (ok) ok = mbar_wait(&bar.kv_done, 0, wc);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            tc_fence_after();
            __nv_bfloat16* dst_row = g == 0 ? p.dv + b * p.dv_sb + h * p.dv_sh + (long long)kg * p.dv_sn
                                            : p.dk + b * p.dk_sb + h * p.dk_sh + (long long)kg * p.dk_sn;
            const float mul = g == 0 ? 1.f : p.scale;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(tRow + 256 + g * D + c0, v);
                tmem_wait_ld();
                if (kg < p.N) {
                    uint4* dst = reinterpret_cast<uint4*>(dst_row + c0);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        dst[q] = make_uint4(
                            pack_h16<F16>(__uint_as_float(v[8 * q + 0]) * mul, __uint_as_float(v[8 * q + 1]) * mul),
                            pack_h16<F16>(__uint_as_float(v[8 * q + 2]) * mul, __uint_as_float(v[8 * q + 3]) * mul),
                            pack_h16<F16>(__uint_as_float(v[8 * q + 4]) * mul, __uint_as_float(v[8 * q + 5]) * mul),
                            pack_h16<F16>(__uint_as_float(v[8 * q + 6]) * mul, __uint_as_float(v[8 * q + 7]) * mul));
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tmem, 512);
}


// ============================================================================
// d = 64: half-tile pipelined variant.
//
// At d = 64 tensor memory has room to overlap the phases the d = 128 kernel
// runs one after another. Each 128-query tile is processed as two halves of
// 64 queries. The tensor core computes the scores S^T, dP^T of half u+2 while
// the warpgroups turn half u+1 into P^T / dS^T and while it runs dV / dK of
// half u. dQ of a whole tile has its own TMEM columns and the dS tile two
// shared-memory buffers, so the dQ drain is off the critical path too.
//
// Tensor memory (512 columns, lane = key row), in 64-column slots:
//   S slots   [0,64) [64,128) [128,192)  S^T of half u in slot u % 3 (fp32, 64 queries);
//             the warpgroups overwrite it with P^T and dS^T bf16 pairs (warpgroup g:
//             P^T at 32g + [0,16), dS^T at 32g + [16,32)), which dV / dK read
//   dP slots  [192,256) [448,512)         dP^T of half u in slot u % 2, free once loaded
//   [256,320) dV   [320,384) dK   [384,448) dQ (query rows = lanes)
// A half holds its dP slot only until the warpgroups have loaded it and its S
// slot until dV / dK have read P^T and dS^T, so three halves are in flight.
//
// Persistent: one CTA per SM walks units (b, h, key tile) in snake order. K
// and V are double-buffered across units, so the next unit's K/V load and its
// first scores overlap the previous unit's last gradients, dQ drain and dV/dK
// stores.
//
// Warps (16): 0-7 P^T / dS^T (two warpgroups, 32 queries of each half each),
// 8 TMA producer, 9 and 10 MMA issuers, 11 the TMA reductions of dQ and the
// stores of dV / dK, 12-15 dQ drain and the units' dV / dK epilogues. The drain
// and the epilogues have their own warpgroup so the P^T / dS^T warps move on to
// the next half, and the next unit, at once.
// ============================================================================
template <bool MASK>
struct Bwd64Cfg {
    static constexpr int D = 64;
    static constexpr int kTileBytes = 128 * D * 2;  // 16 KB: Q, K, V or dO tile (one 64-column box)
    static constexpr int kMaskBytes = BQ * BK * 2;
    static constexpr int kStages = MASK ? 1 : 2;
    static constexpr int kVecOffInStage = 2 * kTileBytes + (MASK ? kMaskBytes : 0);
    static constexpr int kStageBytes = kVecOffInStage + 1024;
    static constexpr int kDSBytes = BQ * BK * 2;  // one dS tile (two 64-query boxes)
    static constexpr int kKOff = 0;             // K, V of unit n in buffer n & 1: K at kKOff + 2 tiles x buffer
    static constexpr int kDSOff = 4 * kTileBytes;  // two dS buffers
    static constexpr int kStageOff = kDSOff + 2 * kDSBytes;
    static constexpr int kStgOff = kStageOff + kStages * kStageBytes;  // dQ staging: 2 boxes of 32 fp32 x 128 rows
    static constexpr int kBarOff = kStgOff + BQ * D * 4;
    static constexpr int kSmemBytes = kBarOff + 256;
};

struct __align__(8) Bwd64Barriers {
    uint64_t kv_full[2];              // per K/V buffer
    uint64_t kv_free[2];              // per K/V buffer: both issuers done with its unit's K and V
    uint64_t dkv_empty;               // the drain warpgroup has read this unit's dV and dK
    uint64_t st_full[2], st_empty[2];
    uint64_t s_full[3], ds_ready[3];  // per S slot
    uint64_t dp_loaded[2];            // per dP slot: the warpgroups have loaded dP^T
    uint64_t dq_full, dq_empty, kv_done, drain[2];
    uint64_t dq_staged, dq_free;      // staging area filled (a dQ tile, or a unit's dV / dK) / free again
    uint64_t buf_free[3];             // per S slot: dV / dK of its half done reading it
    uint64_t dq_done[2];              // dQ of the tile in a dS buffer done reading it
    uint32_t tmem_base;
    int abort_flag;
};

// TMEM column, within an S slot, of the P^T bf16 pairs for MMA k-step kk (16 queries) of a
// half; dS^T pairs are 16 columns further.
__host__ __device__ constexpr int half_packed_col(int kk) { return 32 * (kk >> 1) + 8 * (kk & 1); }
__host__ __device__ constexpr uint32_t s_slot_col(int u) { return 64u * (uint32_t)(u % 3); }
__host__ __device__ constexpr uint32_t dp_slot_col(int u) { return (u & 1) ? 448u : 192u; }
static_assert(sizeof(Bwd64Barriers) <= 256, "barrier block");

// A unit of the d = 64 backward: key tile kt of head (b, h) against all its query tiles.
struct Unit64 {
    int b, h, k0, i_begin, n_it;
};
// Units are numbered key tile major, so the first units (early key tiles) are the heaviest
// under causal masking.
__device__ __forceinline__ Unit64 unit64(const BwdParamsDev& p, int u) {
    const int bh = p.B * p.H;
    const int kt = u / bh, r = u % bh;
    Unit64 w;
    w.b = r / p.H;
    w.h = r % p.H;
    w.k0 = kt * BK;
    w.i_begin = p.causal ? kt : 0;
    w.n_it = (p.N + BQ - 1) / BQ - w.i_begin;
    return w;
}
// The k-th unit of this CTA: rows of gridDim.x units dealt left to right on even rows and
// right to left on odd rows, which evens the per-CTA work when units get lighter.
__device__ __forceinline__ int bwd_unit_at(int k) {
    const int g = gridDim.x, i = blockIdx.x;
    return k * g + ((k & 1) ? g - 1 - i : i);
}

template <bool MASK, bool F16>
__global__ void __launch_bounds__(512, 1)
    bwd_tc64_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_mask, const __grid_constant__ CUtensorMap tm_dq,
                    const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                    const BwdParamsDev p) {
    using Cfg = Bwd64Cfg<MASK>;
    constexpr int D = 64;
    // 16-bit element type of the operands and of P^T, dS^T: bf16, or IEEE half when F16
    constexpr uint32_t kIdescS = idesc_h16(BK, 64, false, false, F16);  // S^T / dP^T of a half
    constexpr uint32_t kIdescKV = idesc_h16(BK, D, false, true, F16);   // dV, dK (A in TMEM)
    constexpr uint32_t kIdescQ = idesc_h16(BQ, D, true, true, F16);     // dQ (A = dS query-major)
    extern __shared__ __align__(1024) uint8_t smem[];
    Bwd64Barriers& bar = *reinterpret_cast<Bwd64Barriers*>(smem + Cfg::kBarOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    WaitCtl wc{p.err, &bar.abort_flag, p.timeout_ns};
    const int nq_all = (p.N + BQ - 1) / BQ;

    if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled tiles need a 1024-byte aligned base
        if (threadIdx.x == 0) atomicExch(p.err, -7);
        return;
    }
    if (threadIdx.x == 0) {
        bar.abort_flag = 0;
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar.kv_full[i], 1);
            mbar_init(&bar.kv_free[i], 2);
        }
        mbar_init(&bar.dkv_empty, 128);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar.st_full[i], 1);
            mbar_init(&bar.st_empty[i], 1);
            mbar_init(&bar.dp_loaded[i], 256);
        }
        for (int i = 0; i < 3; ++i) {
            mbar_init(&bar.s_full[i], 1);
            mbar_init(&bar.ds_ready[i], 256);
            mbar_init(&bar.buf_free[i], 1);
        }
        mbar_init(&bar.dq_full, 1);
        mbar_init(&bar.dq_empty, 128);
        mbar_init(&bar.kv_done, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar.drain[i], 1);
            mbar_init(&bar.dq_done[i], 1);
        }
        mbar_init(&bar.dq_staged, 128);
        mbar_init(&bar.dq_free, 1);
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(&bar.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // No global memory is touched above: from here on the pre-pass must be complete.
    grid_dep_launch();
    grid_dep_wait();
    const uint32_t tmem = bar.tmem_base;

    if (warp == 8) {
        // ------------------------------------------------ producer
        // The whole warp walks the schedule and waits; one elected lane issues the copies.
        if (elect_one()) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_do);
        }
        __syncwarp();
        bool ok = true;
        int n = 0, gt = 0;
        for (int ku = 0, u = bwd_unit_at(0); u < p.num_units && ok; u = bwd_unit_at(++ku), ++n) {
            const Unit64 w = unit64(p, u);
            const int kb = n & 1;
            if (n >= 2) {  // every MMA of unit n-2 that reads this K/V buffer has completed
                ok = mbar_wait_warp(&bar.kv_free[kb], ((n - 2) >> 1) & 1, wc);
                if (!ok) break;
            }
            if (elect_one()) {
                uint8_t* kvb = smem + Cfg::kKOff + kb * 2 * Cfg::kTileBytes;
                mbar_arrive_expect_tx(&bar.kv_full[kb], 2 * Cfg::kTileBytes);
                tma_load_4d(kvb, &tm_k, &bar.kv_full[kb], 0, w.k0, w.h, w.b);
                tma_load_4d(kvb + Cfg::kTileBytes, &tm_v, &bar.kv_full[kb], 0, w.k0, w.h, w.b);
            }
            __syncwarp();
            const int hm = p.mask_hb ? w.h : 0, bm = p.mask_bb ? w.b : 0;
            for (int it = 0; it < w.n_it && ok; ++it, ++gt) {
                const int s = gt % Cfg::kStages;
                ok = mbar_wait_warp(&bar.st_empty[s], ((gt / Cfg::kStages) & 1) ^ 1, wc);
                if (!ok) break;
                const int q0 = (w.i_begin + it) * BQ;
                uint8_t* st = smem + Cfg::kStageOff + s * Cfg::kStageBytes;
                if (elect_one()) {
                    mbar_arrive_expect_tx(&bar.st_full[s], Cfg::kStageBytes);
                    tma_load_4d(st, &tm_q, &bar.st_full[s], 0, q0, w.h, w.b);
                    tma_load_4d(st + Cfg::kTileBytes, &tm_do, &bar.st_full[s], 0, q0, w.h, w.b);
                    if (MASK)
                        for (int bx = 0; bx < 2; ++bx)
                            tma_load_4d(st + 2 * Cfg::kTileBytes + bx * 128 * 128, &tm_mask, &bar.st_full[s],
                                        w.k0 + bx * 64, q0, hm, bm);
                    bulk_load(st + Cfg::kVecOffInStage,
                              p.stats + ((long long)(w.b * p.H + w.h) * nq_all + (w.i_begin + it)) * 256, 1024,
                              &bar.st_full[s]);
                }
                __syncwarp();
            }
        }
        // every copy issued lands before the CTA exits
        if (lane == 0) {
            const int last = gt < Cfg::kStages ? gt : Cfg::kStages;
            for (int i = gt - last; i < gt; ++i)
                drain_wait(&bar.st_full[i % Cfg::kStages], (i / Cfg::kStages) & 1, p.timeout_ns);
            for (int i = n > 2 ? n - 2 : 0; i < n; ++i) drain_wait(&bar.kv_full[i & 1], (i >> 1) & 1, p.timeout_ns);
        }
    } else if (warp == 9 || warp == 10) {
        // ------------------------------------------------ MMA issuers
        // A tcgen05.mma issue returns only once the tensor core has taken it in,
        // so an issuer that waits on a barrier leaves the tensor core idle. Two
        // converged issuer warps, each with one elected lane (always the same
        // one) issuing its MMAs and commits, keep one issuing while the other
        // waits: warp 9 the scores S^T, dP^T of every half, warp 10 the
        // gradients dV, dK of every half and dQ of every tile. Their MMAs do not
        // run in a common order, so the scores of half u wait until the
        // gradients of half u-3 have read its S slot (buf_free) and the warpgroups
        // have loaded dP^T of half u-2 from its dP slot (dp_loaded), and the
        // P^T / dS^T warps wait until dQ of tile i has read the dS buffer before
        // they fill it for tile i+2 (dq_done). Halves and tiles are counted over
        // all units of the CTA.
        bool ok = true;
        int n = 0, gu = 0;
        for (int ku = 0, u = bwd_unit_at(0); u < p.num_units && ok; u = bwd_unit_at(++ku), ++n) {
            const Unit64 w = unit64(p, u);
            ok = mbar_wait_warp(&bar.kv_full[n & 1], (n >> 1) & 1, wc);
            if (!ok) break;
            const uint32_t sK = smem_u32(smem + Cfg::kKOff + (n & 1) * 2 * Cfg::kTileBytes);
            const uint32_t sV = sK + Cfg::kTileBytes;
            if (warp == 10 && n > 0) {  // the warpgroups have read dV / dK of the previous unit
                ok = mbar_wait_warp(&bar.dkv_empty, (n - 1) & 1, wc);
                if (!ok) break;
            }
            tc_fence_after();
            const int n_half = 2 * w.n_it;
            if (warp == 9) {
                for (int hl = 0; hl < n_half && ok; ++hl, ++gu) {
                    // S^T of half gu into S slot gu % 3, dP^T into dP slot gu % 2
                    const int gt = gu >> 1, hf = gu & 1, s = gt % Cfg::kStages;
                    if (hf == 0) {
                        ok = mbar_wait_warp(&bar.st_full[s], (gt / Cfg::kStages) & 1, wc);
                        if (!ok) break;
                    }
                    if (gu >= 3) {  // dV / dK of half gu-3 have read the S slot
                        ok = mbar_wait_warp(&bar.buf_free[gu % 3], ((gu - 3) / 3) & 1, wc);
                        if (!ok) break;
                    }
                    if (gu >= 2) {  // dP^T of half gu-2 has been loaded out of the dP slot
                        ok = mbar_wait_warp(&bar.dp_loaded[gu & 1], ((gu - 2) >> 1) & 1, wc);
                        if (!ok) break;
                    }
                    tc_fence_after();
                    const uint32_t sQ = smem_u32(smem + Cfg::kStageOff + s * Cfg::kStageBytes) + hf * 64 * 128;
                    const uint32_t sdO = sQ + Cfg::kTileBytes;
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk)
                            mma_ss(tmem + s_slot_col(gu), kmajor_desc(sK, kk), kmajor_desc(sQ, kk), kIdescS,
                                   kk > 0 ? 1u : 0u);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk)
                            mma_ss(tmem + dp_slot_col(gu), kmajor_desc(sV, kk), kmajor_desc(sdO, kk), kIdescS,
                                   kk > 0 ? 1u : 0u);
                        mma_commit(&bar.s_full[gu % 3]);
                    }
                    __syncwarp();
                }
                if (elect_one() && ok) mma_commit(&bar.kv_free[n & 1]);  // this unit's reads of K and V
                __syncwarp();
            } else {
                for (int vl = 0; vl < n_half && ok; ++vl, ++gu) {
                    // dV += P^T dO and dK += dS^T Q of half gu
                    const int gt = gu >> 1, hv = gu & 1, sv = gt % Cfg::kStages;
                    ok = mbar_wait_warp(&bar.ds_ready[gu % 3], (gu / 3) & 1, wc);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t sQ = smem_u32(smem + Cfg::kStageOff + sv * Cfg::kStageBytes) + hv * 64 * 128;
                    const uint32_t sdO = sQ + Cfg::kTileBytes;
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_ts(tmem + 256, tmem + s_slot_col(gu) + half_packed_col(kk), mnmajor_desc(sdO, kk),
                                   kIdescKV, (vl > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_ts(tmem + 320, tmem + s_slot_col(gu) + 16 + half_packed_col(kk),
                                   mnmajor_desc(sQ, kk), kIdescKV, (vl > 0 || kk > 0) ? 1u : 0u);
                        mma_commit(&bar.buf_free[gu % 3]);
                        // the tile's last reads of Q and dO (its scores completed before ds_ready)
                        if (hv == 1) mma_commit(&bar.st_empty[sv]);
                        // dV and dK of this unit are complete: the drain reads them out before the
                        // unit's last dQ, so the next unit's gradients need not wait for that dQ
                        if (vl == n_half - 1) mma_commit(&bar.kv_done);
                    }
                    __syncwarp();
                    if (hv == 1) {
                        // dQ = dS K of the tile, once the drain has read the previous one out of TMEM
                        if (gt > 0) {
                            ok = mbar_wait_warp(&bar.dq_empty, (gt - 1) & 1, wc);
                            if (!ok) break;
                            tc_fence_after();
                        }
                        const uint32_t sDS = smem_u32(smem + Cfg::kDSOff + (gt & 1) * Cfg::kDSBytes);
                        if (elect_one()) {
#pragma unroll
                            for (int kk = 0; kk < BK / 16; ++kk)
                                mma_ss(tmem + 384, mnmajor_desc(sDS, kk), mnmajor_desc(sK, kk), kIdescQ,
                                       kk > 0 ? 1u : 0u);
                            mma_commit(&bar.dq_full);
                            mma_commit(&bar.dq_done[gt & 1]);
                        }
                        __syncwarp();
                    }
                }
                if (elect_one() && ok) mma_commit(&bar.kv_free[n & 1]);  // its dQ products have read K
                __syncwarp();
            }
        }
        if (elect_one()) {
            mma_commit(&bar.drain[warp - 9]);
            drain_wait(&bar.drain[warp - 9], 0, p.timeout_ns);
        }
        __syncwarp();
    } else if (warp < 8) {
        // ------------------------------------------------ P^T, dS^T (thread = key row)
        const int g = warp >> 2;  // this warpgroup's 32 queries of each half
        const int kr = (warp & 3) * 32 + lane;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tRow = tmem + lane_off;
        const float2 c2 = make_float2(p.c, p.c);
        bool ok = true;
        int n = 0, gu = 0;
        for (int ku = 0, uu = bwd_unit_at(0); uu < p.num_units && ok; uu = bwd_unit_at(++ku), ++n) {
            const Unit64 w = unit64(p, uu);
            const int kg = w.k0 + kr;
            const bool key_ok = kg < p.N;
            const int n_half = 2 * w.n_it;
            for (int hl = 0; hl < n_half && ok; ++hl, ++gu) {
                const int gt = gu >> 1, hf = gu & 1, s = gt % Cfg::kStages;
                const int q0 = (w.i_begin + (hl >> 1)) * BQ;
                ok = mbar_wait(&bar.s_full[gu % 3], (gu / 3) & 1, wc);
                ok = ok && mbar_wait(&bar.st_full[s], (gt / Cfg::kStages) & 1, wc);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                const uint8_t* stage = smem + Cfg::kStageOff + s * Cfg::kStageBytes;
                const int ql0 = 64 * hf + 32 * g;  // first query (within the tile) of this warpgroup's chunk
                const float* nlv = reinterpret_cast<const float*>(stage + Cfg::kVecOffInStage) + ql0;  // -LSE*log2e
                const float* ndv = nlv + 128;                                                            // -D
                const bool diag = p.causal && (q0 == w.k0);
                const uint8_t* mt = stage + 2 * Cfg::kTileBytes;
                uint32_t sv[32], pv[32];
                const uint32_t tS = tRow + s_slot_col(gu) + 32 * g;
                tmem_ld32(tS, sv);
                tmem_ld32(tRow + dp_slot_col(gu) + 32 * g, pv);
                // before the first half of tile gt >= 2 writes the dS buffer, dQ of tile gt-2 must
                // have read it: test now, wait (if still needed) just before the writes
                const bool need_dq_done = hf == 0 && gt >= 2;
                bool dq_done_seen = !need_dq_done || mbar_test(&bar.dq_done[gt & 1], ((gt - 2) >> 1) & 1);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(&bar.dp_loaded[gu & 1]);  // the dP slot may take the half after next
                uint32_t pk[16], dk[16];
                if (!MASK && !diag && key_ok) {
                    // interior tile: no masking
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        const float4 nl = *reinterpret_cast<const float4*>(nlv + i);
                        const float4 nd = *reinterpret_cast<const float4*>(ndv + i);
                        const float2 x0 = ffma2(make_float2(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])), c2,
                                                make_float2(nl.x, nl.y));
                        const float2 x1 = ffma2(make_float2(__uint_as_float(sv[i + 2]), __uint_as_float(sv[i + 3])),
                                                c2, make_float2(nl.z, nl.w));
                        const float2 p0 = make_float2(ex2(x0.x), ex2(x0.y));
                        const float2 p1 = make_float2(ex2(x1.x), ex2(x1.y));
                        const float2 d0 = fmul2(p0, fadd2(make_float2(__uint_as_float(pv[i]), __uint_as_float(pv[i + 1])),
                                                          make_float2(nd.x, nd.y)));
                        const float2 d1 = fmul2(
                            p1, fadd2(make_float2(__uint_as_float(pv[i + 2]), __uint_as_float(pv[i + 3])),
                                      make_float2(nd.z, nd.w)));
                        pk[i / 2] = pack_h16<F16>(p0.x, p0.y);
                        pk[i / 2 + 1] = pack_h16<F16>(p1.x, p1.y);
                        dk[i / 2] = pack_h16<F16>(d0.x, d0.y);
                        dk[i / 2 + 1] = pack_h16<F16>(d1.x, d1.y);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const int q = ql0 + i;
                        const float2 nl = *reinterpret_cast<const float2*>(nlv + i);
                        const float2 nd = *reinterpret_cast<const float2*>(ndv + i);
                        float2 x = ffma2(make_float2(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])), c2, nl);
                        if (MASK) {
                            const int kb = kr >> 6, kc = (kr & 63) >> 3;
                            const float m0 = h16_to_float<F16>(*reinterpret_cast<const uint16_t*>(
                                mt + kb * 128 * 128 + q * 128 + ((kc ^ (q & 7)) << 4) + (kr & 7) * 2));
                            const float m1 = h16_to_float<F16>(*reinterpret_cast<const uint16_t*>(
                                mt + kb * 128 * 128 + (q + 1) * 128 + ((kc ^ ((q + 1) & 7)) << 4) + (kr & 7) * 2));
                            x = ffma2(make_float2(m0, m1), make_float2(kLog2e, kLog2e), x);
                        }
                        if (!key_ok || (diag && q < kr)) x.x = -INFINITY;
                        if (!key_ok || (diag && q + 1 < kr)) x.y = -INFINITY;
                        const float2 pr = make_float2(ex2(x.x), ex2(x.y));
                        const float2 ds =
                            fmul2(pr, fadd2(make_float2(__uint_as_float(pv[i]), __uint_as_float(pv[i + 1])), nd));
                        pk[i / 2] = pack_h16<F16>(pr.x, pr.y);
                        dk[i / 2] = pack_h16<F16>(ds.x, ds.y);
                    }
                }
                // P^T and dS^T pairs go into the 32 S^T columns this thread just read
                tmem_st16(tS, pk);
                tmem_st16(tS + 16, dk);
                if (!__all_sync(0xffffffffu, dq_done_seen)) {
                    ok = mbar_wait(&bar.dq_done[gt & 1], ((gt - 2) >> 1) & 1, wc);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                }
                // dS row kr, queries ql0 .. ql0+31 of tile buffer (gt & 1): box hf, chunks 4g .. 4g+3
                uint8_t* box = smem + Cfg::kDSOff + (gt & 1) * Cfg::kDSBytes + hf * (128 * 128) + kr * 128;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int ch = 4 * g + j;
                    *reinterpret_cast<uint4*>(box + ((ch ^ (kr & 7)) << 4)) =
                        make_uint4(dk[4 * j], dk[4 * j + 1], dk[4 * j + 2], dk[4 * j + 3]);
                }
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&bar.ds_ready[gu % 3]);
            }
        }
    }

    else if (warp >= 12) {
        // ------------------------------------------------ dQ drain (thread = query row of the tile),
        // and each unit's dV / dK epilogue
        // Both leave through one shared-memory staging area, in the 128-byte-swizzled layout
        // of the TMA maps, and warp 11 copies them out: scale * dQ (box bx = columns 32 bx ..
        // 32 bx + 31) is added into the fp32 accumulator, dV and scale * dK are stored. The
        // area is used in a fixed order, the same for both sides: each dQ tile, with a unit's
        // epilogue just before its last one. Use k waits until use k-1 has been read.
        const int qr = (warp & 3) * 32 + lane;
        const uint32_t tRow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        uint8_t* stg = smem + Cfg::kStgOff;
        bool ok = true;
        int gt = 0, n = 0, use = 0;
        for (int ku = 0, u = bwd_unit_at(0); u < p.num_units && ok; u = bwd_unit_at(++ku), ++n) {
            const Unit64 w = unit64(p, u);
            for (int it = 0; it < w.n_it && ok; ++it, ++gt) {
                if (it == w.n_it - 1) {
                    // unit epilogue (thread = key row), before the unit's last dQ: dV and dK are
                    // complete once their last products are (kv_done), and reading them out
                    // here lets the next unit's gradients start while that dQ is still in the
                    // tensor core. The P^T / dS^T warps go straight on to the next unit.
                    ok = mbar_wait(&bar.kv_done, n & 1, wc);
                    if (use > 0) ok = ok && mbar_wait(&bar.dq_free, (use - 1) & 1, wc);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    tc_fence_after();
                    uint32_t kv[64];
                    tmem_ld32_at<0>(tRow + 256, kv);   // dV
                    tmem_ld32_at<32>(tRow + 288, kv);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4*>(stg + qr * 128 + ((c ^ (qr & 7)) << 4)) =
                            make_uint4(pack_h16<F16>(__uint_as_float(kv[8 * c + 0]), __uint_as_float(kv[8 * c + 1])),
                                       pack_h16<F16>(__uint_as_float(kv[8 * c + 2]), __uint_as_float(kv[8 * c + 3])),
                                       pack_h16<F16>(__uint_as_float(kv[8 * c + 4]), __uint_as_float(kv[8 * c + 5])),
                                       pack_h16<F16>(__uint_as_float(kv[8 * c + 6]), __uint_as_float(kv[8 * c + 7])));
                    tmem_ld32_at<0>(tRow + 320, kv);   // dK
                    tmem_ld32_at<32>(tRow + 352, kv);
                    tmem_wait_ld();
                    tc_fence_before();
                    mbar_arrive(&bar.dkv_empty);  // the accumulators may take the next unit
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4*>(stg + 128 * 128 + qr * 128 + ((c ^ (qr & 7)) << 4)) = make_uint4(
                            pack_h16<F16>(__uint_as_float(kv[8 * c + 0]) * p.scale,
                                          __uint_as_float(kv[8 * c + 1]) * p.scale),
                            pack_h16<F16>(__uint_as_float(kv[8 * c + 2]) * p.scale,
                                          __uint_as_float(kv[8 * c + 3]) * p.scale),
                            pack_h16<F16>(__uint_as_float(kv[8 * c + 4]) * p.scale,
                                          __uint_as_float(kv[8 * c + 5]) * p.scale),
                            pack_h16<F16>(__uint_as_float(kv[8 * c + 6]) * p.scale,
                                          __uint_as_float(kv[8 * c + 7]) * p.scale));
                    fence_proxy_async_smem();
                    mbar_arrive(&bar.dq_staged);  // warp 11 stores them
                    ++use;
                }
                ok = mbar_wait(&bar.dq_full, gt & 1, wc);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                uint32_t v[64];
                tmem_ld32_at<0>(tRow + 384, v);
                tmem_ld32_at<32>(tRow + 416, v);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(&bar.dq_empty);
                if (use > 0) {  // the previous use of the staging area has been read
                    ok = mbar_wait(&bar.dq_free, (use - 1) & 1, wc);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                }
#pragma unroll
                for (int bx = 0; bx < 2; ++bx) {
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const int col = 32 * bx + 4 * c;
                        const float2 a0 = fmul2(make_float2(__uint_as_float(v[col]), __uint_as_float(v[col + 1])),
                                                make_float2(p.scale, p.scale));
                        const float2 a1 = fmul2(make_float2(__uint_as_float(v[col + 2]), __uint_as_float(v[col + 3])),
                                                make_float2(p.scale, p.scale));
                        *reinterpret_cast<float4*>(stg + bx * (BQ * 128) + qr * 128 + ((c ^ (qr & 7)) << 4)) =
                            make_float4(a0.x, a0.y, a1.x, a1.y);
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(&bar.dq_staged);
                ++use;
            }
        }
    } else if (warp == 11) {
        // ------------------------------------------------ bulk copies out of the staging area
        // One elected lane (always the same one: the warp is converged) copies each use of
        // the staging area out, in the drain's order, and waits for the copy to read shared
        // memory before handing the area back. Keeping those waits here keeps them off the
        // drain warpgroup. Rows beyond N are clipped by the tensor maps.
        uint8_t* stg = smem + Cfg::kStgOff;
        if (elect_one()) {
            prefetch_tmap(&tm_dq);
            prefetch_tmap(&tm_dk);
            prefetch_tmap(&tm_dv);
        }
        __syncwarp();
        bool ok = true;
        int use = 0;
        for (int ku = 0, u = bwd_unit_at(0); u < p.num_units && ok; u = bwd_unit_at(++ku)) {
            const Unit64 w = unit64(p, u);
            for (int it = 0; it < w.n_it && ok; ++it) {
                if (it == w.n_it - 1) {  // the unit's dV and dK
                    ok = mbar_wait_warp(&bar.dq_staged, use & 1, wc);
                    if (!ok) break;
                    if (elect_one()) {
                        tma_store_4d(&tm_dv, stg, 0, w.k0, w.h, w.b);
                        tma_store_4d(&tm_dk, stg + 128 * 128, 0, w.k0, w.h, w.b);
                        bulk_commit();
                        bulk_wait_read0();
                        mbar_arrive(&bar.dq_free);
                    }
                    __syncwarp();
                    ++use;
                }
                ok = mbar_wait_warp(&bar.dq_staged, use & 1, wc);
                if (!ok) break;
                if (elect_one()) {
                    const int q0 = (w.i_begin + it) * BQ;
                    tma_reduce_add_4d(&tm_dq, stg, 0, q0, w.h, w.b);
                    tma_reduce_add_4d(&tm_dq, stg + BQ * 128, 32, q0, w.h, w.b);
                    bulk_commit();
                    bulk_wait_read0();
                    mbar_arrive(&bar.dq_free);
                }
                __syncwarp();
                ++use;
            }
        }
        if (elect_one()) bulk_wait0();  // reductions and stores complete before the CTA exits
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tmem, 512);
}

template <int D, bool MASK, bool F16>
cudaError_t launch_bwd_tc_t(const attn_bwd_params& prm, const BwdMaps& maps, const BwdWorkspace& ws,
                            const LaunchCommon& lc, cudaStream_t s) {
    constexpr int kSmem = [] {
        if constexpr (D == 64)
            return Bwd64Cfg<MASK>::kSmemBytes;
        else
            return BwdCfg<D, MASK>::kSmemBytes;
    }();
    static_assert(kSmem <= 232448, "shared memory budget");
    auto kernel = [] {
        if constexpr (D == 64)
            return bwd_tc64_kernel<MASK, F16>;
        else
            return bwd_tc_kernel<D, MASK, F16>;
    }();
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    const attn_fwd_params& f = prm.fwd;
    BwdParamsDev p{};
    p.B = f.B;
    p.H = f.H;
    p.N = f.N;
    p.causal = f.causal;
    p.c = f.scale * kLog2e;
    p.scale = f.scale;
    p.stats = ws.stats;
    p.dq_acc = ws.dq_acc;
    p.dk = static_cast<__nv_bfloat16*>(prm.dk);
    p.dv = static_cast<__nv_bfloat16*>(prm.dv);
    p.dk_sb = prm.dk_stride[0];
    p.dk_sh = prm.dk_stride[1];
    p.dk_sn = prm.dk_stride[2];
    p.dv_sb = prm.dv_stride[0];
    p.dv_sh = prm.dv_stride[1];
    p.dv_sn = prm.dv_stride[2];
    p.mask_hb = f.mask ? (f.mask_stride[1] != 0) : 0;
    p.mask_bb = f.mask ? (f.mask_stride[0] != 0) : 0;
    p.n_ktiles = (f.N + BK - 1) / BK;
    p.err = lc.err;
    p.timeout_ns = lc.timeout_ns;
    p.num_units = p.n_ktiles * f.B * f.H;
    // d = 64: persistent, one CTA per SM walking the units; d = 128: one CTA per unit
    const unsigned grid = D == 64 ? (unsigned)(p.num_units < lc.num_sms ? p.num_units : lc.num_sms)
                                  : (unsigned)p.num_units;
    e = launch_pdl(kernel, dim3(grid), dim3(D == 64 ? 512 : 384), kSmem, s, maps.q, maps.k, maps.v, maps.dout,
                   maps.mask, maps.dq_acc, maps.dk, maps.dv, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}


template <bool F16>
cudaError_t launch_bwd_tc_dt(const attn_bwd_params& p, const BwdMaps& maps, const BwdWorkspace& ws,
                             const LaunchCommon& lc, cudaStream_t s) {
    const bool mask = p.fwd.mask != nullptr;
    if (p.fwd.d == 64)
        return mask ? launch_bwd_tc_t<64, true, F16>(p, maps, ws, lc, s)
                    : launch_bwd_tc_t<64, false, F16>(p, maps, ws, lc, s);
    return mask ? launch_bwd_tc_t<128, true, F16>(p, maps, ws, lc, s)
                : launch_bwd_tc_t<128, false, F16>(p, maps, ws, lc, s);
}

}  // namespace

cudaError_t launch_bwd_tc(const attn_bwd_params& p, const BwdMaps& maps, const BwdWorkspace& ws,
                          const LaunchCommon& lc, cudaStream_t s) {
    return p.fwd.dtype == ATTN_F16 ? launch_bwd_tc_dt<true>(p, maps, ws, lc, s)
                                   : launch_bwd_tc_dt<false>(p, maps, ws, lc, s);
}

}  // namespace attn
