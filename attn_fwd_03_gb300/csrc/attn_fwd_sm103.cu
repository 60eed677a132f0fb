// attn_fwd_sm103.cu — bf16 attention forward on the sm_103a tensor cores.
//
// FlashAttention-2 loop order ("What is FlashAttention?", Step 3): the query
// tile stays resident and key/value tiles stream through shared memory, the
// per-row running max m, sum l and unnormalised output o stay on chip, and
// only O and the per-row log-sum-exp are written back ("What is
// FlashAttention?", step list: "O, m and l are written back, never the
// scores"). The N x N scores exist only one 128 x 128 tile at a time, in
// tensor memory.
//
// One persistent CTA per SM walks work units (b, h, 256 query rows). A unit
// holds two 128-row query tiles that take turns on the tensor core, so the
// softmax of one tile overlaps the matrix products of the other.
//
// Warp roles (12 warps = 3 warpgroups):
//   warps 0-3  softmax for query tile 0 (one thread per query row)
//   warps 4-7  softmax for query tile 1
//   warp  8    TMA producer: Q tiles, then K_j, V_j into a ring of stages
//   warp  9    TMEM allocator; MMA issuer (d = 128: both tiles; d = 64: tile 0)
//   warp 10    TMA producer for the additive mask tiles (mask variant only)
//   warp 11    MMA issuer for tile 1 (d = 64), else idle
// The producer and MMA warps run their loops converged, waits included, and
// one elected lane issues each batch of copies or MMAs.
// The launch gives every thread 168 registers (384 x 168 = 64512); the
// softmax warpgroups then raise theirs (216 for d = 128, 208 for d = 64) and
// the third warpgroup drops to the rest (72 or 88), so a thread can hold a
// whole 128-column score row in registers.
//
// Tensor memory (512 columns x 128 lanes, lane = query row), d = 128:
//   [0,128)        S_0 (fp32 scores of tile 0); P_0 (bf16 pairs) in its first 64 columns
//   [128,256)      S_1 / P_1
//   [256,384)      O_0 (fp32 accumulator)
//   [384,512)      O_1
// Per key tile j and query tile t the MMA warp issues O_t += P_t^{j-1} V_{j-1}
// and then S_t^j = Q_t K_j^T; tcgen05 MMAs from one thread run in issue order,
// so S_t^j overwriting P_t^{j-1} is safe, and the commit that signals S_t^j
// also covers the previous PV, which lets the softmax warps rescale O_t.
//
// d = 64 ("split P"): S_0 [0,128), S_1 [128,256), O_0 [256,320), O_1 [320,384),
// P_0 [384,448), P_1 [448,512). The softmax warps release S_t (s_free) as soon
// as they have loaded it, so S_t^{j+1} is computed while they still work on
// S_t^j; the PV product signals its own completion (pv_done), which the
// softmax warps wait for before they rescale O_t or overwrite P_t. At d = 64
// the matrix products are short next to the softmax, and this keeps the
// softmax warps from waiting on them.
//
// Online softmax in the log2 domain ("Explain FlashAttention and why it is
// IO-aware", "Keep only the state needed for the final weighted average";
// "FlashAttention", "Why it is allowed to be exact"): scores are multiplied
// by c = scale * log2(e); the row keeps a reference max m_ref and
// l = sum 2^(s - m_ref). The reference moves only when a tile's max exceeds
// it by more than kRescaleThreshold (= 8, i.e. a factor of 256), and only
// then are l and O multiplied by alpha = 2^(m_ref_old - m_ref_new). l and O
// always share the same reference, so O / l is exact: the final division
// cancels the common factor. Probabilities stay <= 2^8 in fp32 and bf16.
// Rows whose scores are all -inf keep m_ref = -inf, l = 0, O = 0 and return
// O = 0, LSE = -inf ("Explain FlashAttention and why it is IO-aware",
// "Executable recurrence, with an empty-state policy").
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
constexpr float kRescaleThreshold = 8.0f;

template <int D, bool MASK>
struct FwdCfg {
    static constexpr int kBoxes = D / 64;                  // 64-column (128-byte) TMA boxes per row
    static constexpr int kTileBytes = BM * D * 2;          // one Q, K or V tile
    static constexpr int kStages = (D == 128) ? (MASK ? 3 : 4) : (MASK ? 6 : 8);
    // d = 64: P gets its own TMEM columns and each query tile its own MMA issuer
    static constexpr bool kSplit = D == 64;
    static constexpr int kIssuers = kSplit ? 2 : 1;
    static constexpr int kMaskBytes = BM * BN * 2;
    static constexpr int kWarps = 12;
    // per-thread registers after the rebalance: 2 x 128 x softmax + 128 x other = 384 x 168
    static constexpr int kSoftmaxRegs = D == 64 ? 208 : 216;
    static constexpr int kOtherRegs = D == 64 ? 88 : 72;
    static_assert(2 * 128 * kSoftmaxRegs + 128 * kOtherRegs <= 384 * 168, "register split");
    static constexpr int kThreads = kWarps * 32;
    // shared memory layout (offsets from a 1024-aligned base)
    static constexpr int kQOff = 0;
    static constexpr int kKVOff = kQOff + 2 * kTileBytes;
    static constexpr int kMaskOff = kKVOff + kStages * kTileBytes;
    static constexpr int kBarOff = kMaskOff + (MASK ? 2 * kMaskBytes : 0);
    static constexpr int kSmemBytes = kBarOff + 512 + 1024;  // barriers + alignment slack
};

struct FwdParamsDev {
    int B, H, N;
    int causal;
    float c;          // scale * log2(e)
    float inv_scale;  // 1 / scale: the additive mask in units of the raw scores
    float* lse;
    __nv_bfloat16* o;
    long long o_sb, o_sh, o_sn;
    int mask_hb, mask_bb;  // 1 if the mask varies along h / b
    int num_units, n_qblk;
    int head_major;        // unit order: heads outermost (see decode_unit)
    int* err;
    unsigned long long timeout_ns;
    int stall_after;
};

struct __align__(8) Barriers {
    uint64_t q_full, q_empty;
    uint64_t kv_full[8], kv_empty[8];
    uint64_t s_full[2], p_full[2], o_full[2], o_empty[2];
    uint64_t s_free[2], pv_done[2];  // split-P layout only
    uint64_t m_full[2], m_empty[2];
    uint64_t drain[2];
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(Barriers) <= 512, "barrier area");

struct Unit {
    int b, h, qblk;
    int row0[2];
    int nkv[2];  // key tiles tile t needs (0 if the tile starts beyond N)
    int nkv_max;
};

__device__ __forceinline__ Unit decode_unit(const FwdParamsDev& p, int u) {
    Unit w;
    const int bh = p.B * p.H;
    int r;
    if (p.head_major) {
        // all units weigh the same (no causal mask): heads outermost, so the CTAs running
        // at one time share the K/V of a few heads, which stay in L2
        r = u / p.n_qblk;
        w.qblk = u % p.n_qblk;
    } else {
        // heaviest query blocks first (causal), heads innermost so neighbouring CTAs
        // share the mask rows of the same block
        w.qblk = p.n_qblk - 1 - u / bh;
        r = u % bh;
    }
    w.b = r / p.H;
    w.h = r % p.H;
    const int nk_all = (p.N + BN - 1) / BN;
    for (int t = 0; t < 2; ++t) {
        w.row0[t] = w.qblk * 2 * BM + t * BM;
        if (w.row0[t] >= p.N)
            w.nkv[t] = 0;
        else
            w.nkv[t] = p.causal ? min(nk_all, w.row0[t] / BN + 1) : nk_all;
    }
    w.nkv_max = max(w.nkv[0], w.nkv[1]);
    return w;
}

// The k-th work unit of this CTA. Units are numbered heaviest first and dealt to the CTAs
// in rows of gridDim.x, left to right on even rows and right to left on odd rows, so a
// CTA that drew a heavy unit in one row draws a light one in the next. With causal
// masking this evens the per-CTA work (at B=4 H=16 N=2048 the busiest CTA has 61 tile
// pairs against 72 for a plain round robin, the mean being 57.3).
__device__ __forceinline__ int unit_at(int k) {
    const int g = gridDim.x, i = blockIdx.x;
    return k * g + ((k & 1) ? g - 1 - i : i);
}

// Shared-memory descriptor of a K-major tile (rows x 64-column boxes) at k-step kk.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk) {
    return sdesc_sw128(tile + (kk >> 2) * (BM * 128) + (kk & 3) * 32, 16, 1024);
}
// Shared-memory descriptor of V (keys x D, MN-major for the PV product) at k-step kk.
__device__ __forceinline__ uint64_t vmajor_desc(uint32_t tile, int kk) {
    return sdesc_sw128(tile + kk * (16 * 128), BN * 128, 1024);
}

// Wait that ignores the abort flag (used only to drain in-flight copies at exit).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(a, parity))
        if (globaltimer() - t0 > timeout_ns) break;
}

template <int D, bool MASK, bool F16>
__global__ void __launch_bounds__(FwdCfg<D, MASK>::kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_mask,
                  const FwdParamsDev p) {
    using Cfg = FwdCfg<D, MASK>;
    // 16-bit element type of Q, K, V, P and O: bf16, or IEEE half when F16
    constexpr uint32_t kIdescS = idesc_h16(BM, BN, false, false, F16);
    constexpr uint32_t kIdescO = idesc_h16(BM, D, false, true, F16);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Barriers& bar = *reinterpret_cast<Barriers*>(smem + Cfg::kBarOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    WaitCtl wc{p.err, &bar.abort_flag, p.timeout_ns};

    if (threadIdx.x == 0) {
        bar.abort_flag = 0;
        mbar_init(&bar.q_full, 1);
        mbar_init(&bar.q_empty, Cfg::kIssuers);
        for (int s = 0; s < Cfg::kStages; ++s) {
            mbar_init(&bar.kv_full[s], 1);
            mbar_init(&bar.kv_empty[s], Cfg::kIssuers);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&bar.s_full[t], 1);
            mbar_init(&bar.p_full[t], BM);
            mbar_init(&bar.o_full[t], 1);
            mbar_init(&bar.o_empty[t], BM);
            mbar_init(&bar.m_full[t], 1);
            mbar_init(&bar.m_empty[t], BM);
            mbar_init(&bar.s_free[t], BM);
            mbar_init(&bar.pv_done[t], 1);
            mbar_init(&bar.drain[t], 1);
        }
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
    const uint32_t sKV = smem_u32(smem + Cfg::kKVOff);

    if (warp >= 8) {
      regs_decrease<Cfg::kOtherRegs>();
      if (warp == 8) {
        // ------------------------------------------------ K/V producer
        // The whole warp walks the schedule and waits; one elected lane issues the copies.
        if (elect_one()) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
        }
        __syncwarp();
        uint32_t it = 0, n_units = 0;
        int tiles_issued = 0;
        bool ok = true;
        for (int ku = 0, u = unit_at(0); u < p.num_units && ok; u = unit_at(++ku), ++n_units) {
            const Unit w = decode_unit(p, u);
            ok = mbar_wait_warp(&bar.q_empty, (n_units & 1) ^ 1, wc);
            if (!ok) break;
            const int nt = w.nkv[1] > 0 ? 2 : 1;
            if (elect_one()) {
                mbar_arrive_expect_tx(&bar.q_full, nt * Cfg::kTileBytes);
                for (int t = 0; t < nt; ++t)
                    for (int bx = 0; bx < Cfg::kBoxes; ++bx)
                        tma_load_4d(smem + Cfg::kQOff + t * Cfg::kTileBytes + bx * BM * 128, &tm_q, &bar.q_full,
                                    bx * 64, w.row0[t], w.h, w.b);
            }
            __syncwarp();
            for (int j = 0; j < w.nkv_max && ok; ++j) {
                if (p.stall_after > 0 && tiles_issued >= p.stall_after) {
                    ok = false;  // test hook: stop feeding the consumers
                    break;
                }
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
                ++tiles_issued;
            }
        }
        // drain: every copy issued must land before the CTA exits
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
            uint32_t cnt[2] = {0, 0};
            bool ok = true;
            for (int ku = 0, u = unit_at(0); u < p.num_units && ok; u = unit_at(++ku)) {
                const Unit w = decode_unit(p, u);
                const int hm = p.mask_hb ? w.h : 0, bm = p.mask_bb ? w.b : 0;
                for (int j = 0; j < w.nkv_max && ok; ++j) {
                    for (int t = 0; t < 2; ++t) {
                        if (j >= w.nkv[t]) continue;
                        ok = mbar_wait(&bar.m_empty[t], (cnt[t] & 1) ^ 1, wc);
                        if (!ok) break;
                        mbar_arrive_expect_tx(&bar.m_full[t], Cfg::kMaskBytes);
                        uint8_t* dst = smem + Cfg::kMaskOff + t * Cfg::kMaskBytes;
                        for (int bx = 0; bx < 2; ++bx)
                            tma_load_4d(dst + bx * BM * 128, &tm_mask, &bar.m_full[t], j * BN + bx * 64, w.row0[t],
                                        hm, bm);
                        ++cnt[t];
                    }
                }
            }
            for (int t = 0; t < 2; ++t)
                if (cnt[t] > 0) drain_wait(&bar.m_full[t], (cnt[t] - 1) & 1, p.timeout_ns);
        }
    } else if (Cfg::kSplit && (warp == 9 || warp == 11)) {
        // ------------------------------------------------ MMA issuers, one per query tile
        // With P in its own columns S_t^{j+1} can be computed as soon as the
        // softmax warps have read S_t^j, while they still work on it. Warp 9
        // issues every MMA of query tile 0, warp 11 those of tile 1, so one
        // issuer's barrier waits overlap the other's MMAs. Each issuer walks every
        // K/V ring slot (waiting for it to fill) and releases it once, used or not;
        // the slot's empty barrier expects both.
        const int t = warp == 9 ? 0 : 1;
        const uint32_t tS = tmem + t * BN, tO = tmem + 256 + t * D, tP = tmem + 384 + t * 64;
        uint32_t it = 0, n_units = 0, n_s = 0, n_p = 0;
        bool ok = true;
        for (int ku = 0, u = unit_at(0); u < p.num_units && ok; u = unit_at(++ku), ++n_units) {
            const Unit w = decode_unit(p, u);
            const int nkv = w.nkv[t];
            ok = mbar_wait_warp(&bar.q_full, n_units & 1, wc);
            if (!ok) break;
            tc_fence_after();
            if (nkv == 0) {  // this tile lies beyond N: release Q at once
                if (elect_one()) mbar_arrive(&bar.q_empty);
                __syncwarp();
            }
            for (int j = 0; j <= w.nkv_max && ok; ++j) {
                const uint32_t itK = it;  // ring slot of K_j; V_j follows it
                const uint32_t sK = itK % Cfg::kStages, sV_prev = (itK + Cfg::kStages - 1) % Cfg::kStages;
                if (j < w.nkv_max) {
                    ok = mbar_wait_warp(&bar.kv_full[sK], (itK / Cfg::kStages) & 1, wc);
                    if (!ok) break;
                    if (j < nkv) {
                        // S_t^j = Q_t K_j^T, once the softmax warps have read S_t^{j-1}
                        if (n_s > 0) {
                            ok = mbar_wait_warp(&bar.s_free[t], (n_s - 1) & 1, wc);
                            if (!ok) break;
                        }
                        tc_fence_after();
                        const uint32_t qt = sQ + t * Cfg::kTileBytes, kt = sKV + sK * Cfg::kTileBytes;
                        if (elect_one()) {
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk)
                                mma_ss(tS, kmajor_desc(qt, kk), kmajor_desc(kt, kk), kIdescS, kk > 0 ? 1u : 0u);
                            mma_commit(&bar.s_full[t]);
                            if (j == nkv - 1) mma_commit(&bar.q_empty);  // last read of Q_t
                        }
                        __syncwarp();
                        ++n_s;
                    }
                    if (elect_one()) mma_commit(&bar.kv_empty[sK]);
                    __syncwarp();
                }
                if (j > 0) {  // V_{j-1} lives in the slot before K_j
                    ok = mbar_wait_warp(&bar.kv_full[sV_prev], ((itK - 1) / Cfg::kStages) & 1, wc);
                    if (!ok) break;
                    if (j <= nkv) {
                        // O_t += P_t^{j-1} V_{j-1}, once the softmax warps have stored P_t^{j-1}
                        ok = mbar_wait_warp(&bar.p_full[t], n_p & 1, wc);
                        if (!ok) break;
                        ++n_p;
                        tc_fence_after();
                        const uint32_t vt = sKV + sV_prev * Cfg::kTileBytes;
                        if (elect_one()) {
#pragma unroll
                            for (int kk = 0; kk < BN / 16; ++kk)
                                mma_ts(tO, tP + kk * 8, vmajor_desc(vt, kk), kIdescO, (j > 1 || kk > 0) ? 1u : 0u);
                            mma_commit(&bar.pv_done[t]);
                        }
                        __syncwarp();
                    }
                    if (elect_one()) mma_commit(&bar.kv_empty[sV_prev]);
                    __syncwarp();
                }
                if (j < w.nkv_max) it += 2;
            }
        }
        // every MMA this warp issued completes before TMEM is released
        if (elect_one()) {
            mma_commit(&bar.drain[t]);
            drain_wait(&bar.drain[t], 0, p.timeout_ns);
        }
        __syncwarp();
    } else if (warp == 9) {
        // ------------------------------------------------ MMA issuer
        // The whole warp walks the schedule and waits; one elected lane (the same
        // one every time: the warp is converged) issues the MMAs and their commits.
        uint32_t it = 0, n_units = 0, pcnt[2] = {0, 0}, ocnt[2] = {0, 0};
        bool ok = true;
        for (int ku = 0, u = unit_at(0); u < p.num_units && ok; u = unit_at(++ku), ++n_units) {
            const Unit w = decode_unit(p, u);
            ok = mbar_wait_warp(&bar.q_full, n_units & 1, wc);
            if (!ok) break;
            tc_fence_after();
            for (int j = 0; j <= w.nkv_max && ok; ++j) {
                const uint32_t itK = it;  // ring slot of K_j; V_j follows it
                const uint32_t sK = itK % Cfg::kStages, sV_prev = (itK + Cfg::kStages - 1) % Cfg::kStages;
                if (j < w.nkv_max) {
                    ok = mbar_wait_warp(&bar.kv_full[sK], (itK / Cfg::kStages) & 1, wc);
                    if (!ok) break;
                }
                if (j > 0) {  // V_{j-1} lives in the slot before K_j
                    ok = mbar_wait_warp(&bar.kv_full[sV_prev], ((itK - 1) / Cfg::kStages) & 1, wc);
                    if (!ok) break;
                }
                tc_fence_after();
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (!ok || w.nkv[t] == 0 || j > w.nkv[t]) continue;
                    const uint32_t tS = tmem + t * BN, tO = tmem + 256 + t * D;
                    if (j > 0) {
                        // O_t += P_t^{j-1} V_{j-1}
                        if (j == 1) {  // first PV of the unit overwrites O_t: epilogue must be done with it
                            ok = mbar_wait_warp(&bar.o_empty[t], (ocnt[t] & 1) ^ 1, wc);
                            if (!ok) continue;
                        }
                        ok = mbar_wait_warp(&bar.p_full[t], pcnt[t] & 1, wc);
                        if (!ok) continue;
                        ++pcnt[t];
                        tc_fence_after();
                        const uint32_t vt = sKV + sV_prev * Cfg::kTileBytes;
                        if (elect_one()) {
#pragma unroll
                            for (int kk = 0; kk < BN / 16; ++kk)
                                mma_ts(tO, tS + kk * 8, vmajor_desc(vt, kk), kIdescO, (j > 1 || kk > 0) ? 1u : 0u);
                        }
                        __syncwarp();
                    }
                    if (j < w.nkv[t]) {
                        // S_t^j = Q_t K_j^T
                        const uint32_t qt = sQ + t * Cfg::kTileBytes, kt = sKV + sK * Cfg::kTileBytes;
                        if (elect_one()) {
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk)
                                mma_ss(tS, kmajor_desc(qt, kk), kmajor_desc(kt, kk), kIdescS, kk > 0 ? 1u : 0u);
                            mma_commit(&bar.s_full[t]);
                        }
                        __syncwarp();
                    } else {
                        if (elect_one()) mma_commit(&bar.o_full[t]);  // last PV of this tile issued
                        __syncwarp();
                        ++ocnt[t];
                    }
                }
                if (!ok) break;
                if (elect_one()) {
                    if (j == w.nkv_max - 1) mma_commit(&bar.q_empty);  // last S of the unit issued
                    if (j < w.nkv_max) mma_commit(&bar.kv_empty[sK]);
                    if (j > 0) mma_commit(&bar.kv_empty[sV_prev]);
                }
                __syncwarp();
                if (j < w.nkv_max) it += 2;
            }
        }
        // every MMA this warp issued completes before TMEM is released
        if (elect_one()) {
            mma_commit(&bar.drain[0]);
            drain_wait(&bar.drain[0], 0, p.timeout_ns);
        }
        __syncwarp();
      }
    } else {
        regs_increase<Cfg::kSoftmaxRegs>();
        // ------------------------------------------------ softmax warpgroups
        const int t = warp >> 2;
        const int r = (warp & 3) * 32 + lane;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_off + t * BN;
        const uint32_t tO = tmem + lane_off + 256 + t * D;
        const uint32_t tP = Cfg::kSplit ? tmem + lane_off + 384 + t * 64 : tS;
        const uint8_t* mtile = smem + Cfg::kMaskOff + t * Cfg::kMaskBytes;
        uint32_t scnt = 0, mcnt = 0, ocnt = 0, pvcnt = 0;
        bool ok = true;
        for (int ku = 0, u = unit_at(0); u < p.num_units && ok; u = unit_at(++ku)) {
            const Unit w = decode_unit(p, u);
            const int nkv = w.nkv[t];
            if (nkv == 0) continue;
            const int row = w.row0[t] + r;
            float m_ref = -INFINITY, m_row = -INFINITY, l = 0.f;
            for (int j = 0; j < nkv; ++j) {
                ok = mbar_wait(&bar.s_full[t], scnt & 1, wc);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                ++scnt;
                tc_fence_after();
                uint32_t su[BN];
                tmem_ld32_at<0>(tS + 0, su);
                tmem_ld32_at<32>(tS + 32, su);
                tmem_ld32_at<64>(tS + 64, su);
                tmem_ld32_at<96>(tS + 96, su);
                tmem_wait_ld();
                if (Cfg::kSplit) {  // S_t is in registers: the next S_t may overwrite it
                    tc_fence_before();
                    mbar_arrive(&bar.s_free[t]);
                }
                const bool diag = p.causal && (j == nkv - 1);
                const bool tail = (j + 1) * BN > p.N;
                // s stays in raw score units (times cc = scale * log2(e) below); the additive
                // mask enters as mask / scale, one packed FMA per pair of columns
                const float cc = p.c;
                if (MASK) {
                    ok = mbar_wait(&bar.m_full[t], mcnt & 1, wc);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    ++mcnt;
#pragma unroll
                    for (int bx = 0; bx < 2; ++bx) {
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch) {
                            const uint4 mv = *reinterpret_cast<const uint4*>(
                                mtile + bx * BM * 128 + r * 128 + ((ch ^ (r & 7)) << 4));
                            const uint32_t mw[4] = {mv.x, mv.y, mv.z, mv.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int col = bx * 64 + ch * 8 + 2 * e;
                                const float2 x = ffma2(unpack_h16<F16>(mw[e]), make_float2(p.inv_scale, p.inv_scale),
                                                       make_float2(__uint_as_float(su[col]), __uint_as_float(su[col + 1])));
                                su[col] = __float_as_uint(x.x);
                                su[col + 1] = __float_as_uint(x.y);
                            }
                        }
                    }
                    mbar_arrive(&bar.m_empty[t]);
                }
                if (diag || tail) {  // causal on absolute positions, and the key tail
                    const int key0 = j * BN;
                    const int lim_causal = diag ? row - key0 : BN;  // keys with index <= row survive
                    const int lim_tail = p.N - key0;
                    const int lim = min(lim_causal + 1, lim_tail);  // first masked column
#pragma unroll
                    for (int col = 0; col < BN; ++col)
                        if (col >= lim) su[col] = __float_as_uint(-INFINITY);
                }
                // tile max (in the log2 domain after multiplying by cc): 3-input max, eight
                // independent chains of 16 columns each
                float mx[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float m = fmaxf(__uint_as_float(su[16 * c]), __uint_as_float(su[16 * c + 1]));
#pragma unroll
                    for (int e = 2; e < 16; e += 2)
                        m = fmax3(m, __uint_as_float(su[16 * c + e]), __uint_as_float(su[16 * c + e + 1]));
                    mx[c] = m;
                }
                const float m_tile =
                    fmaxf(fmax3(fmax3(mx[0], mx[1], mx[2]), mx[3], mx[4]), fmax3(mx[5], mx[6], mx[7])) * cc;
                m_row = fmaxf(m_row, m_tile);
                float m_new = m_ref;
                if (m_tile > m_ref + kRescaleThreshold) m_new = m_tile;
                const bool moved = m_new != m_ref;
                const float alpha = moved ? ex2(m_ref - m_new) : 1.f;  // 0 when m_ref = -inf
                const bool rescale = j > 0 && __any_sync(0xffffffffu, moved && m_ref != -INFINITY);
                // O_t *= alpha. The PV of key tile j-1 must be complete: here it precedes S_t^j
                // in the MMA stream (the s_full commit covers it); with P in its own columns
                // it is the pv_done commit, taken after the exponentials below.
                auto rescale_o = [&]() {
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t ov[32];
                        tmem_ld32(tO + c0, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const float2 r2 = fmul2(make_float2(__uint_as_float(ov[i]), __uint_as_float(ov[i + 1])),
                                                    make_float2(alpha, alpha));
                            ov[i] = __float_as_uint(r2.x);
                            ov[i + 1] = __float_as_uint(r2.y);
                        }
                        tmem_st32(tO + c0, ov);
                    }
                };
                if (!Cfg::kSplit && rescale) rescale_o();
                m_ref = m_new;
                const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;
                // p = 2^(s * cc - m): one packed FMA per pair, two exp2, one packed add, one convert
                const float2 cc2 = make_float2(cc, cc), nm2 = make_float2(neg_m, neg_m);
                float2 suma = make_float2(0.f, 0.f), sumb = make_float2(0.f, 0.f);
                if (Cfg::kSplit) {
                    // P packed into su[0..63] (pair i lands in su[i], already consumed)
#pragma unroll
                    for (int i = 0; i < BN / 2; ++i) {
                        const float2 x = ffma2(make_float2(__uint_as_float(su[2 * i]), __uint_as_float(su[2 * i + 1])),
                                               cc2, nm2);
                        const float2 pp = make_float2(ex2(x.x), ex2(x.y));
                        if (i & 1)
                            sumb = fadd2(sumb, pp);
                        else
                            suma = fadd2(suma, pp);
                        su[i] = pack_h16<F16>(pp.x, pp.y);
                    }
                    if (j > 0) {  // PV of key tile j-1 has finished reading P_t and writing O_t
                        ok = mbar_wait(&bar.pv_done[t], pvcnt & 1, wc);
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok) break;
                        ++pvcnt;
                        tc_fence_after();
                        if (rescale) rescale_o();
                    }
                    tmem_st32_at<0>(tP + 0, su);
                    tmem_st32_at<32>(tP + 32, su);
                } else {
#pragma unroll
                    for (int c0 = 0; c0 < BN; c0 += 32) {
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float2 x = ffma2(
                                make_float2(__uint_as_float(su[c0 + 2 * i]), __uint_as_float(su[c0 + 2 * i + 1])), cc2,
                                nm2);
                            const float2 pp = make_float2(ex2(x.x), ex2(x.y));
                            if (i & 1)
                                sumb = fadd2(sumb, pp);
                            else
                                suma = fadd2(suma, pp);
                            pk[i] = pack_h16<F16>(pp.x, pp.y);
                        }
                        tmem_st16(tS + c0 / 2, pk);
                    }
                }
                l = l * alpha + ((suma.x + suma.y) + (sumb.x + sumb.y));
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bar.p_full[t]);
            }
            if (!ok) break;
            // epilogue: O = O / l (0 for fully masked rows), LSE in natural log
            if (Cfg::kSplit) {
                ok = mbar_wait(&bar.pv_done[t], pvcnt & 1, wc);  // the unit's last PV
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                ++pvcnt;
            } else {
                ok = mbar_wait(&bar.o_full[t], ocnt & 1, wc);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                ++ocnt;
            }
            tc_fence_after();
            const float den = o_divisor<F16>(l, m_row, m_ref);
            const float inv = den > 0.f ? 1.f / den : 0.f;
            __nv_bfloat16* orow = p.o + w.b * p.o_sb + w.h * p.o_sh + (long long)row * p.o_sn;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t ov[32];
                tmem_ld32(tO + c0, ov);
                tmem_wait_ld();
                if (row < p.N) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 v;
                        v.x = pack_h16<F16>(__uint_as_float(ov[8 * q + 0]) * inv, __uint_as_float(ov[8 * q + 1]) * inv);
                        v.y = pack_h16<F16>(__uint_as_float(ov[8 * q + 2]) * inv, __uint_as_float(ov[8 * q + 3]) * inv);
                        v.z = pack_h16<F16>(__uint_as_float(ov[8 * q + 4]) * inv, __uint_as_float(ov[8 * q + 5]) * inv);
                        v.w = pack_h16<F16>(__uint_as_float(ov[8 * q + 6]) * inv, __uint_as_float(ov[8 * q + 7]) * inv);
                        dst[q] = v;
                    }
                }
            }
            tc_fence_before();
            if (!Cfg::kSplit) mbar_arrive(&bar.o_empty[t]);
            if (row < p.N)
                p.lse[((long long)w.b * p.H + w.h) * p.N + row] =
                    l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tmem, 512);
}

template <int D, bool MASK, bool F16>
cudaError_t launch_tc(const attn_fwd_params& prm, const FwdMaps& maps, const LaunchCommon& lc, cudaStream_t s) {
    using Cfg = FwdCfg<D, MASK>;
    static_assert(Cfg::kSmemBytes <= 232448, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(fwd_tc_kernel<D, MASK, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    FwdParamsDev p{};
    p.B = prm.B;
    p.H = prm.H;
    p.N = prm.N;
    p.causal = prm.causal;
    p.c = prm.scale * kLog2e;
    p.inv_scale = 1.f / prm.scale;
    p.lse = prm.lse;
    p.o = static_cast<__nv_bfloat16*>(prm.o);
    p.o_sb = prm.o_stride[0];
    p.o_sh = prm.o_stride[1];
    p.o_sn = prm.o_stride[2];
    p.mask_hb = prm.mask ? (prm.mask_stride[1] != 0) : 0;
    p.mask_bb = prm.mask ? (prm.mask_stride[0] != 0) : 0;
    p.n_qblk = (prm.N + 2 * BM - 1) / (2 * BM);
    p.head_major = !prm.causal && !MASK;
    p.num_units = p.n_qblk * prm.B * prm.H;
    p.err = lc.err;
    p.timeout_ns = lc.timeout_ns;
    p.stall_after = lc.stall_after;
    const int grid = p.num_units < lc.num_sms ? p.num_units : lc.num_sms;
    e = launch_pdl(fwd_tc_kernel<D, MASK, F16>, dim3(grid), dim3(Cfg::kThreads), Cfg::kSmemBytes, s,
                   maps.q, maps.k, maps.v, maps.mask, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}


template <bool F16>
cudaError_t launch_fwd_tc_t(const attn_fwd_params& p, const FwdMaps& maps, const LaunchCommon& lc, cudaStream_t s) {
    const bool mask = p.mask != nullptr;
    if (p.d == 64) return mask ? launch_tc<64, true, F16>(p, maps, lc, s) : launch_tc<64, false, F16>(p, maps, lc, s);
    return mask ? launch_tc<128, true, F16>(p, maps, lc, s) : launch_tc<128, false, F16>(p, maps, lc, s);
}

}  // namespace

cudaError_t launch_fwd_tc(const attn_fwd_params& p, const FwdMaps& maps, const LaunchCommon& lc, cudaStream_t s) {
    return p.dtype == ATTN_F16 ? launch_fwd_tc_t<true>(p, maps, lc, s) : launch_fwd_tc_t<false>(p, maps, lc, s);
}

}  // namespace attn
