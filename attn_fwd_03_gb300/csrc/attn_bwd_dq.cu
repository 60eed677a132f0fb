// attn_bwd_dq.cu — dQ of the attention backward with a fixed order of additions.
//
// The main backward kernel keeps a key tile on chip and adds every query
// tile's share of dQ into an fp32 accumulator with TMA reduce-add: the order
// in which the key tiles' additions reach a dQ row changes from run to run,
// so dQ is reproducible only to rounding. This kernel computes dQ the other
// way round, query-stationary like the forward ("What is FlashAttention?",
// Step 3 loop order): one 128-row query tile stays on chip with its dO rows
// while the key and value tiles stream past, and
//     S = Q K_j^T,  dP = dO V_j^T              (tcgen05, operands in shared memory)
//     P = exp(scale * S + mask - LSE),  dS = P * (dP - D)   (one warpgroup per 64 keys)
//     dQ += dS K_j                             (tcgen05, dS from tensor memory)
// accumulate in tensor memory in key-tile order, so every bit of dQ is a
// function of the inputs alone. P is recomputed from the saved log-sum-exp and
// D = rowsum(dO * O) as the rest of the backward does ("What is
// FlashAttention?", Step 4), so no running max is needed. dQ leaves the chip
// once, already scaled, in the dtype of Q: there is no fp32 accumulator and no
// finalize pass.
//
// One persistent CTA per SM walks work units (b, h, 128-row query tile),
// heaviest causal tiles first, dealt in a snake order like the forward's.
//
// Warp roles (12 warps):
//   warps 0-3  keys [0, 64) of every key tile, and dQ columns [0, d/2) at the end of a unit
//   warps 4-7  keys [64, 128), and dQ columns [d/2, d)   (thread = query row in both)
//   warp  8    TMA producer: Q and dO once per unit, then K_j, V_j into a ring
//   warp  9    TMEM allocator and MMA issuer
//   warp 10    TMA producer of the additive mask tiles (mask variant only)
//   warp 11    idle
// The launch gives every thread 168 registers; the dS warpgroups raise theirs
// to 176 (64 scores and 64 dP values per thread) and warps 8-11 drop to 152.
//
// Tensor memory (512 columns, lane = query row):
//   [0,128), [128,256)  S of key tiles j even / odd (fp32); the warpgroups write
//                       dS (16-bit pairs) over the first half of the 64 columns
//                       each of them read: [0,32) and [64,96) of the buffer
//   [256,384)           dP (fp32)
//   [384,384+d)         dQ accumulator (fp32)
// Per key tile the issuer runs S_j, dP_j, then dQ += dS_{j-1} K_{j-1}, so the
// tensor core computes the scores of tile j while the warpgroups build dS of
// tile j-1. S_{j+2} overwrites dS_j only after the dQ product that reads it:
// tcgen05 MMAs issued by one thread execute in order.
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

using namespace ptx;

constexpr int BM = 128;  // query rows per tile
constexpr int BN = 128;  // keys per tile

template <int D, bool MASK>
struct DqCfg {
    static constexpr int kBoxes = D / 64;          // 64-column (128-byte) TMA boxes per row
    static constexpr int kTileBytes = 128 * D * 2;  // one Q, dO, K or V tile
    // K_j stays in the ring until dQ += dS_j K_j is issued, after K_{j+1} and V_{j+1} have
    // been used: the ring needs at least 4 slots or the producer would wait on the issuer
    static constexpr int kStages = D == 128 ? 4 : (MASK ? 6 : 8);
    static_assert(kStages >= 4, "K/V ring too short");
    static constexpr int kMaskBytes = BM * BN * 2;
    static constexpr int kMaskBufs = (D == 128 && MASK) ? 1 : 2;  // d = 128: one fits beside the ring
    static constexpr int kThreads = 12 * 32;
    // per-thread registers after the rebalance: 256 x dS warpgroups + 128 x the rest <= 384 x 168
    static constexpr int kDsRegs = 176;
    static constexpr int kOtherRegs = 152;
    static_assert(256 * kDsRegs + 128 * kOtherRegs <= kThreads * 168, "register split");
    static constexpr int kQOff = 0;  // Q tile, then the dO tile
    static constexpr int kKVOff = kQOff + 2 * kTileBytes;
    static constexpr int kMaskOff = kKVOff + kStages * kTileBytes;
    static constexpr int kBarOff = kMaskOff + (MASK ? kMaskBufs * kMaskBytes : 0);
    static constexpr int kSmemBytes = kBarOff + 256 + 1024;  // barriers + alignment slack
};

struct DqParamsDev {
    int B, H, N;
    int causal;
    float c;      // scale * log2(e)
    float scale;
    const float* stats;  // [B*H][n_qt][2][128]: -LSE*log2e, then -D
    __nv_bfloat16* dq;   // 16-bit output (bf16 or half bits)
    long long dq_sb, dq_sh, dq_sn;
    int mask_hb, mask_bb;
    int n_qt;       // query tiles per (b, h)
    int num_units;  // n_qt * B * H
    int head_major;
    int* err;
    unsigned long long timeout_ns;
};

struct __align__(8) DqBarriers {
    uint64_t q_full, q_empty;
    uint64_t kv_full[8], kv_empty[8];
    uint64_t s_full[2];   // S of the key tile in buffer 0 / 1
    uint64_t dp_full, dp_free;
    uint64_t ds_full[2];  // dS written over S buffer 0 / 1
    uint64_t dq_full, dq_empty;
    uint64_t m_full[2], m_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(DqBarriers) <= 256, "barrier area");

struct DqUnit {
    int b, h, qt, nkv;
};

__device__ __forceinline__ DqUnit dq_unit(const DqParamsDev& p, int u) {
    DqUnit w;
    const int bh = p.B * p.H;
    int r;
    if (p.head_major) {  // all units weigh the same: heads outermost, K/V of a few heads stay in L2
        r = u / p.n_qt;
        w.qt = u % p.n_qt;
    } else {  // heaviest (causal) tiles first, heads innermost
        w.qt = p.n_qt - 1 - u / bh;
        r = u % bh;
    }
    w.b = r / p.H;
    w.h = r % p.H;
    const int nk_all = (p.N + BN - 1) / BN;
    w.nkv = p.causal ? min(nk_all, w.qt + 1) : nk_all;  // BM == BN: tile qt ends on the diagonal
    return w;
}

// The k-th unit of this CTA: rows of gridDim.x units, left to right on even rows and
// right to left on odd ones, which evens the per-CTA work when units get lighter.
__device__ __forceinline__ int unit_at(int k) {
    const int g = gridDim.x, i = blockIdx.x;
    return k * g + ((k & 1) ? g - 1 - i : i);
}

// Shared-memory descriptor of a K-major tile (rows x 64-column boxes) at k-step kk.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk) {
    return sdesc_sw128(tile + (kk >> 2) * (128 * 128) + (kk & 3) * 32, 16, 1024);
}
// Shared-memory descriptor of K (keys x D) read MN-major, as the B operand of dS K, at k-step kk.
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t tile, int kk) {
    return sdesc_sw128(tile + kk * (16 * 128), BN * 128, 1024);
}
// TMEM column (from the S buffer) of the dS pairs of keys [16 kk, 16 kk + 16).
__host__ __device__ constexpr int ds_col(int kk) { return 64 * (kk >> 2) + 8 * (kk & 3); }

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(a, parity))
        if (globaltimer() - t0 > timeout_ns) break;
}

template <int D, bool MASK, bool F16>
__global__ void __launch_bounds__(DqCfg<D, MASK>::kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_mask, const DqParamsDev p) {
    using Cfg = DqCfg<D, MASK>;
    constexpr uint32_t kIdescS = idesc_h16(BM, BN, false, false, F16);  // S and dP: both operands K-major
    constexpr uint32_t kIdescQ = idesc_h16(BM, D, false, true, F16);    // dQ: K read MN-major
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    DqBarriers& bar = *reinterpret_cast<DqBarriers*>(smem + Cfg::kBarOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    WaitCtl wc{p.err, &bar.abort_flag, p.timeout_ns};

    if (threadIdx.x == 0) {
        bar.abort_flag = 0;
        mbar_init(&bar.q_full, 1);
        mbar_init(&bar.q_empty, 1);
        for (int s = 0; s < Cfg::kStages; ++s) {
            mbar_init(&bar.kv_full[s], 1);
            mbar_init(&bar.kv_empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&bar.s_full[t], 1);
            mbar_init(&bar.ds_full[t], 256);
            mbar_init(&bar.m_full[t], 1);
            mbar_init(&bar.m_empty[t], 256);
        }
        mbar_init(&bar.dp_full, 1);
        mbar_init(&bar.dp_free, 256);
        mbar_init(&bar.dq_full, 1);
        mbar_init(&bar.dq_empty, 256);
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
    // No global memory is touched above: from here on the previous kernel must be complete.
    grid_dep_launch();
    grid_dep_wait();
    const uint32_t tmem = bar.tmem_base;
    const uint32_t sQ = smem_u32(smem + Cfg::kQOff);
    const uint32_t sDO = sQ + Cfg::kTileBytes;
    const uint32_t sKV = smem_u32(smem + Cfg::kKVOff);

    if (warp >= 8) {
      regs_decrease<Cfg::kOtherRegs>();
      if (warp == 8) {
        // ------------------------------------------------ Q / dO / K / V producer
        if (elect_one()) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_do);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
        }
        __syncwarp();
        uint32_t it = 0, n_units = 0;
        bool ok = true;
        for (int ku = 0, u = unit_at(0); u < p.num_units && ok; u = unit_at(++ku), ++n_units) {
            const DqUnit w = dq_unit(p, u);
            ok = mbar_wait_warp(&bar.q_empty, (n_units & 1) ^ 1, wc);
            if (!ok) break;
            if (elect_one()) {
                mbar_arrive_expect_tx(&bar.q_full, 2 * Cfg::kTileBytes);
                for (int bx = 0; bx < Cfg::kBoxes; ++bx) {
                    tma_load_4d(smem + Cfg::kQOff + bx * BM * 128, &tm_q, &bar.q_full, bx * 64, w.qt * BM, w.h, w.b);
                    tma_load_4d(smem + Cfg::kQOff + Cfg::kTileBytes + bx * BM * 128, &tm_do, &bar.q_full, bx * 64,
                                w.qt * BM, w.h, w.b);
                }
            }
            __syncwarp();
            for (int j = 0; j < w.nkv && ok; ++j) {
                for (int kv = 0; kv < 2; ++kv, ++it) {
                    const uint32_t s = it % Cfg::kStages;
                    ok = mbar_wait_warp(&bar.kv_empty[s], ((it / Cfg::kStages) & 1) ^ 1, wc);
                    if (!ok) break;
                    if (elect_one()) {
                        mbar_arrive_expect_tx(&bar.kv_full[s], Cfg::kTileBytes);
                        uint8_t* dst = smem + Cfg::kKVOff + s * Cfg::kTileBytes;
                        for (int bx = 0; bx < Cfg::kBoxes; ++bx)
                            tma_load_4d(dst + bx * BN * 128, kv == 0 ? &tm_k : &tm_v, &bar.kv_full[s], bx * 64,
                                        j * BN, w.h, w.b);
                    }
                    __syncwarp();
                }
            }
        }
        // every copy issued must land before the CTA exits
        if (lane == 0) {
            const uint32_t last = it < (uint32_t)Cfg::kStages ? it : (uint32_t)Cfg::kStages;
            for (uint32_t i = it - last; i < it; ++i)
                drain_wait(&bar.kv_full[i % Cfg::kStages], (i / Cfg::kStages) & 1, p.timeout_ns);
            if (n_units > 0) drain_wait(&bar.q_full, (n_units - 1) & 1, p.timeout_ns);
        }
    } else if (MASK && warp == 10) {
        // ------------------------------------------------ mask producer
        if (lane == 0) {
            prefetch_tmap(&tm_mask);
            uint32_t cnt = 0;
            bool ok = true;
            for (int ku = 0, u = unit_at(0); u < p.num_units && ok; u = unit_at(++ku)) {
                const DqUnit w = dq_unit(p, u);
                const int hm = p.mask_hb ? w.h : 0, bm = p.mask_bb ? w.b : 0;
                for (int j = 0; j < w.nkv && ok; ++j, ++cnt) {
                    const int mb = cnt % Cfg::kMaskBufs;
                    ok = mbar_wait(&bar.m_empty[mb], ((cnt / Cfg::kMaskBufs) & 1) ^ 1, wc);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&bar.m_full[mb], Cfg::kMaskBytes);
                    uint8_t* dst = smem + Cfg::kMaskOff + mb * Cfg::kMaskBytes;
                    for (int bx = 0; bx < 2; ++bx)
                        tma_load_4d(dst + bx * BM * 128, &tm_mask, &bar.m_full[mb], j * BN + bx * 64, w.qt * BM, hm,
                                    bm);
                }
            }
            const uint32_t last = cnt < (uint32_t)Cfg::kMaskBufs ? cnt : (uint32_t)Cfg::kMaskBufs;
            for (uint32_t i = cnt - last; i < cnt; ++i)
                drain_wait(&bar.m_full[i % Cfg::kMaskBufs], (i / Cfg::kMaskBufs) & 1, p.timeout_ns);
        }
    } else if (warp == 9) {
        // ------------------------------------------------ MMA issuer
        // Converged warp; one elected lane issues every MMA and commit.
        const uint32_t tDP = tmem + 256, tDQ = tmem + 384;
        uint32_t it = 0, g = 0, n_units = 0;
        bool ok = true;
        for (int ku = 0, u = unit_at(0); u < p.num_units && ok; u = unit_at(++ku), ++n_units) {
            const DqUnit w = dq_unit(p, u);
            ok = mbar_wait_warp(&bar.q_full, n_units & 1, wc);
            if (!ok) break;
            tc_fence_after();
            // step j issues S_j and dP_j (j < nkv), then dQ += dS_{j-1} K_{j-1} (j > 0);
            // g is the CTA-wide index of key tile j, it its K slot in the ring (V_j follows)
            for (int j = 0; j <= w.nkv && ok; ++j) {
                if (j < w.nkv) {
                    const uint32_t sK = it % Cfg::kStages, sV = (it + 1) % Cfg::kStages;
                    ok = mbar_wait_warp(&bar.kv_full[sK], (it / Cfg::kStages) & 1, wc);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t tS = tmem + (g & 1) * 128;
                    const uint32_t kt = sKV + sK * Cfg::kTileBytes, vt = sKV + sV * Cfg::kTileBytes;
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk)
                            mma_ss(tS, kmajor_desc(sQ, kk), kmajor_desc(kt, kk), kIdescS, kk > 0 ? 1u : 0u);
                        mma_commit(&bar.s_full[g & 1]);
                    }
                    __syncwarp();
                    ok = mbar_wait_warp(&bar.kv_full[sV], ((it + 1) / Cfg::kStages) & 1, wc);
                    if (!ok) break;
                    if (g > 0) {  // the warpgroups have read dP of the previous key tile
                        ok = mbar_wait_warp(&bar.dp_free, (g - 1) & 1, wc);
                        if (!ok) break;
                    }
                    tc_fence_after();
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk)
                            mma_ss(tDP, kmajor_desc(sDO, kk), kmajor_desc(vt, kk), kIdescS, kk > 0 ? 1u : 0u);
                        mma_commit(&bar.dp_full);
                        mma_commit(&bar.kv_empty[sV]);  // V_j has no other reader
                        if (j == w.nkv - 1) mma_commit(&bar.q_empty);  // last read of Q and dO
                    }
                    __syncwarp();
                }
                if (j > 0) {
                    // dQ += dS_{j-1} K_{j-1}
                    const uint32_t gp = g - 1, itp = it - 2;
                    const uint32_t sKp = itp % Cfg::kStages;
                    ok = mbar_wait_warp(&bar.ds_full[gp & 1], (gp >> 1) & 1, wc);
                    if (!ok) break;
                    if (j == 1) {  // first dQ product of the unit: the last unit's dQ has been read out
                        ok = mbar_wait_warp(&bar.dq_empty, (n_units & 1) ^ 1, wc);
                        if (!ok) break;
                    }
                    tc_fence_after();
                    const uint32_t tDS = tmem + (gp & 1) * 128;
                    const uint32_t kt = sKV + sKp * Cfg::kTileBytes;
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk)
                            mma_ts(tDQ, tDS + ds_col(kk), mnmajor_desc(kt, kk), kIdescQ, (j > 1 || kk > 0) ? 1u : 0u);
                        mma_commit(&bar.kv_empty[sKp]);
                        if (j == w.nkv) mma_commit(&bar.dq_full);
                    }
                    __syncwarp();
                }
                if (j < w.nkv) {
                    it += 2;
                    ++g;
                }
            }
        }
        // every MMA this warp issued completes before TMEM is released
        if (elect_one()) {
            mma_commit(&bar.drain);
            drain_wait(&bar.drain, 0, p.timeout_ns);
        }
        __syncwarp();
      }
    } else {
        regs_increase<Cfg::kDsRegs>();
        // ------------------------------------------------ dS warpgroups
        const int wg = warp >> 2;             // keys [64 wg, 64 wg + 64) of each tile
        const int r = (warp & 3) * 32 + lane;  // query row within the tile
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tDP = tmem + lane_off + 256 + wg * 64;
        const uint32_t tDQ = tmem + lane_off + 384 + wg * (D / 2);
        const float ninf = -INFINITY;
        uint32_t g = 0, n_units = 0, mcnt = 0;
        bool ok = true;
        for (int ku = 0, u = unit_at(0); u < p.num_units && ok; u = unit_at(++ku), ++n_units) {
            const DqUnit w = dq_unit(p, u);
            const int row = w.qt * BM + r;
            const float* st = p.stats + ((long long)(w.b * p.H + w.h) * p.n_qt + w.qt) * 256;
            const float nlse = st[r];   // -LSE * log2(e); -inf for empty and padding rows
            const float nd = st[128 + r];  // -D
            for (int j = 0; j < w.nkv; ++j, ++g) {
                const uint32_t tS = tmem + lane_off + (g & 1) * 128 + wg * 64;
                ok = mbar_wait(&bar.s_full[g & 1], (g >> 1) & 1, wc);
                if (ok) ok = mbar_wait(&bar.dp_full, g & 1, wc);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                uint32_t su[64], dp[64];
                tmem_ld32_at<0>(tS, su);
                tmem_ld32_at<32>(tS + 32, su);
                tmem_ld32_at<0>(tDP, dp);
                tmem_ld32_at<32>(tDP + 32, dp);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(&bar.dp_free);  // dP is in registers: the next dP may overwrite it
                const int key0 = j * BN + wg * 64;
                const bool diag = p.causal && (j == w.nkv - 1);
                const bool tail = key0 + 64 > p.N;
                float cc = p.c;
                if (MASK || diag || tail) {
                    // fold scale, mask, causal and tail into s (log2 domain)
                    const int lim_causal = diag ? row - key0 + 1 : 64;  // keys <= row survive
                    const int lim = min(lim_causal, p.N - key0);        // first masked column
                    if (MASK) {
                        const int mb = mcnt % Cfg::kMaskBufs;
                        ok = mbar_wait(&bar.m_full[mb], (mcnt / Cfg::kMaskBufs) & 1, wc);
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok) break;
                        ++mcnt;
                        const uint8_t* mrow = smem + Cfg::kMaskOff + mb * Cfg::kMaskBytes + wg * BM * 128 + r * 128;
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch) {
                            const uint4 mv = *reinterpret_cast<const uint4*>(mrow + ((ch ^ (r & 7)) << 4));
                            const uint32_t mw[4] = {mv.x, mv.y, mv.z, mv.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 f = unpack_h16<F16>(mw[e]);
                                const int col = ch * 8 + 2 * e;
                                su[col] = __float_as_uint(fmaf(__uint_as_float(su[col]), p.c, f.x * kLog2e));
                                su[col + 1] = __float_as_uint(fmaf(__uint_as_float(su[col + 1]), p.c, f.y * kLog2e));
                            }
                        }
                        mbar_arrive(&bar.m_empty[mb]);
                    } else {
#pragma unroll
                        for (int col = 0; col < 64; ++col) su[col] = __float_as_uint(__uint_as_float(su[col]) * p.c);
                    }
#pragma unroll
                    for (int col = 0; col < 64; ++col)
                        if (col >= lim) su[col] = __float_as_uint(ninf);
                    cc = 1.f;
                }
                // p = 2^(s cc - LSE log2 e), dS = p (dP - D), packed in pairs over the scores read
                const float2 cc2 = make_float2(cc, cc), nl2 = make_float2(nlse, nlse), nd2 = make_float2(nd, nd);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float2 x =
                        ffma2(make_float2(__uint_as_float(su[2 * i]), __uint_as_float(su[2 * i + 1])), cc2, nl2);
                    const float2 pr = make_float2(ex2(x.x), ex2(x.y));
                    const float2 dd =
                        fmul2(pr, fadd2(make_float2(__uint_as_float(dp[2 * i]), __uint_as_float(dp[2 * i + 1])), nd2));
                    su[i] = pack_h16<F16>(dd.x, dd.y);
                }
                tmem_st32_at<0>(tS, su);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bar.ds_full[g & 1]);
            }
            if (!ok) break;
            // epilogue: this warpgroup's half of the dQ row, scaled, in the dtype of Q
            ok = mbar_wait(&bar.dq_full, n_units & 1, wc);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            __nv_bfloat16* qrow = p.dq + w.b * p.dq_sb + w.h * p.dq_sh + (long long)row * p.dq_sn + wg * (D / 2);
#pragma unroll
            for (int c0 = 0; c0 < D / 2; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(tDQ + c0, v);
                tmem_wait_ld();
                if (row < p.N) {
                    uint4* dst = reinterpret_cast<uint4*>(qrow + c0);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 o;
                        o.x = pack_h16<F16>(__uint_as_float(v[8 * q + 0]) * p.scale, __uint_as_float(v[8 * q + 1]) * p.scale);
                        o.y = pack_h16<F16>(__uint_as_float(v[8 * q + 2]) * p.scale, __uint_as_float(v[8 * q + 3]) * p.scale);
                        o.z = pack_h16<F16>(__uint_as_float(v[8 * q + 4]) * p.scale, __uint_as_float(v[8 * q + 5]) * p.scale);
                        o.w = pack_h16<F16>(__uint_as_float(v[8 * q + 6]) * p.scale, __uint_as_float(v[8 * q + 7]) * p.scale);
                        dst[q] = o;
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&bar.dq_empty);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tmem, 512);
}

template <int D, bool MASK, bool F16>
cudaError_t launch_dq(const attn_bwd_params& prm, const BwdMaps& maps, const BwdWorkspace& ws, const LaunchCommon& lc,
                      cudaStream_t s) {
    using Cfg = DqCfg<D, MASK>;
    static_assert(Cfg::kSmemBytes <= 232448, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(bwd_dq_kernel<D, MASK, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    const attn_fwd_params& f = prm.fwd;
    DqParamsDev p{};
    p.B = f.B;
    p.H = f.H;
    p.N = f.N;
    p.causal = f.causal;
    p.c = f.scale * kLog2e;
    p.scale = f.scale;
    p.stats = ws.stats;
    p.dq = static_cast<__nv_bfloat16*>(prm.dq);
    p.dq_sb = prm.dq_stride[0];
    p.dq_sh = prm.dq_stride[1];
    p.dq_sn = prm.dq_stride[2];
    p.mask_hb = f.mask ? (f.mask_stride[1] != 0) : 0;
    p.mask_bb = f.mask ? (f.mask_stride[0] != 0) : 0;
    p.n_qt = (f.N + BM - 1) / BM;
    p.num_units = p.n_qt * f.B * f.H;
    p.head_major = !f.causal && !MASK;
    p.err = lc.err;
    p.timeout_ns = lc.timeout_ns;
    const int grid = p.num_units < lc.num_sms ? p.num_units : lc.num_sms;
    e = launch_pdl(bwd_dq_kernel<D, MASK, F16>, dim3(grid), dim3(Cfg::kThreads), Cfg::kSmemBytes, s, maps.q, maps.k,
                   maps.v, maps.dout, maps.mask, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <bool F16>
cudaError_t launch_dq_t(const attn_bwd_params& p, const BwdMaps& maps, const BwdWorkspace& ws, const LaunchCommon& lc,
                        cudaStream_t s) {
    const bool mask = p.fwd.mask != nullptr;
    if (p.fwd.d == 64)
        return mask ? launch_dq<64, true, F16>(p, maps, ws, lc, s) : launch_dq<64, false, F16>(p, maps, ws, lc, s);
    return mask ? launch_dq<128, true, F16>(p, maps, ws, lc, s) : launch_dq<128, false, F16>(p, maps, ws, lc, s);
}

}  // namespace

cudaError_t launch_bwd_dq(const attn_bwd_params& p, const BwdMaps& maps, const BwdWorkspace& ws,
                          const LaunchCommon& lc, cudaStream_t s) {
    return p.fwd.dtype == ATTN_F16 ? launch_dq_t<true>(p, maps, ws, lc, s) : launch_dq_t<false>(p, maps, ws, lc, s);
}

}  // namespace attn
