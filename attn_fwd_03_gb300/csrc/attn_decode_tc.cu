// attn_decode_tc.cu — the split-KV decode's per-split pass on the tensor cores,
// for a few to a few dozen query rows.
//
// Decode is bound by reading K and V once ("FlashAttention", "What it does not
// do"). With more than a handful of query rows the CUDA-core split kernel
// runs out of arithmetic before it runs out of bandwidth (nq x d
// multiply-adds per key and row), so this kernel computes each split's scores
// and weighted sum with tcgen05 products. The nq query rows sit in a 128-row
// M tile whose other rows are zero: the products do up to 128 / nq times the
// useful work, which is cheap next to the key/value read (a 128-key tile is
// 32 KB at d = 128, about 2900 cycles of one SM's share of HBM bandwidth,
// against about 1000 tensor cycles for both products).
//
// Work units are (b, h, split); a persistent CTA per SM walks them. Per unit
// the loop is the forward's (FlashAttention-2 order, "What is FlashAttention?",
// Step 3): Q stays on chip, K_j and V_j stream through a ring of whole-tile
// slots, S = Q K_j^T and O += P V_j on the tensor core, with P in its own
// tensor-memory columns so the next S is computed while the softmax works:
//   issue order  S_0, S_1, PV_0, S_2, PV_1, ..., S_{n-1}, PV_{n-2}, PV_{n-1}
// The online softmax keeps a reference max per row that moves only when a
// tile's max exceeds it by more than 8 (log2 units); l and o share it. The
// split's result per row is the partial state (m, l, o) that the combine
// kernel merges (records [b*h][split][nq][d + 4]: m, l, two unused, o).
//
// Causal decode is aligned bottom-right: query row i is position nk - nq + i
// and sees the keys j <= nk - nq + i.
//
// Warp roles: warps 0 .. ceil(nq / 32) - 1 softmax (one thread per query row),
// warp 4 TMA producer, warp 5 TMEM allocator and MMA issuer.
// Tensor memory (lane = query row): S [0,128) fp32, P [128,192) 16-bit pairs,
// O [256, 256 + d) fp32.
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

using namespace ptx;

constexpr int BM = 128;  // M tile (query rows, zero beyond nq)
constexpr int BN = 128;  // keys per tile
constexpr float kRescaleThreshold = 8.0f;
constexpr int kThreads = 192;  // 6 warps

template <int D>
struct DtcCfg {
    static constexpr int kBoxes = D / 64;
    static constexpr int kTileBytes = BN * D * 2;
    static constexpr int kSlots = D == 128 ? 6 : 12;  // 192 KB of K/V tiles in flight
    static constexpr int kQOff = 0;
    static constexpr int kRingOff = kQOff + kTileBytes;
    static constexpr int kBarOff = kRingOff + kSlots * kTileBytes;
    static constexpr int kSmemBytes = kBarOff + 512 + 1024;  // barriers + alignment slack
};

struct DtcParams {
    int B, H, nq, nk, causal;
    int splits, chunk;
    int num_units;
    int n_sm_warps;  // softmax warps: ceil(nq / 32)
    float c;         // scale * log2(e)
    float* part;     // [B*H][splits][nq][D + 4]
    int* err;
    unsigned long long timeout_ns;
};

struct __align__(8) DtcBarriers {
    uint64_t q_full, q_empty;
    uint64_t slot_full[12], slot_empty[12];
    uint64_t s_full, s_free, p_full, pv_done, o_empty;
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(DtcBarriers) <= 512, "barrier area");

struct DtcUnit {
    int b, h, bh, split;
    int key0, key_end;  // keys [key0, key_end) of this split (before the causal limit)
    int ntiles;
};

__device__ __forceinline__ DtcUnit dtc_unit(const DtcParams& p, int u) {
    DtcUnit w;
    // splits outermost: neighbouring CTAs read different heads' key ranges at the same time
    w.split = u / (p.B * p.H);
    w.bh = u % (p.B * p.H);
    w.b = w.bh / p.H;
    w.h = w.bh % p.H;
    w.key0 = w.split * p.chunk;
    w.key_end = min(p.nk, w.key0 + p.chunk);
    w.ntiles = (w.key_end - w.key0 + BN - 1) / BN;
    return w;
}

// Item t of a unit's K/V sequence (t < 2 n): K_0, then K_i, V_{i-1} for i = 1 .. n-1, then V_{n-1}.
__device__ __forceinline__ void kv_item(int t, int n, bool* is_k, int* tile) {
    if (t == 0) {
        *is_k = true;
        *tile = 0;
    } else if (t == 2 * n - 1) {
        *is_k = false;
        *tile = n - 1;
    } else {
        *is_k = (t & 1) != 0;
        *tile = *is_k ? (t + 1) / 2 : t / 2 - 1;
    }
}

__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk) {
    return sdesc_sw128(tile + (kk >> 2) * (BN * 128) + (kk & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t vmajor_desc(uint32_t tile, int kk) {
    return sdesc_sw128(tile + kk * (16 * 128), BN * 128, 1024);
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(a, parity))
        if (globaltimer() - t0 > timeout_ns) break;
}

template <int D, bool F16>
__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const DtcParams p) {
    using Cfg = DtcCfg<D>;
    constexpr uint32_t kIdescS = idesc_h16(BM, BN, false, false, F16);
    constexpr uint32_t kIdescO = idesc_h16(BM, D, false, true, F16);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    DtcBarriers& bar = *reinterpret_cast<DtcBarriers*>(smem + Cfg::kBarOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t n_sm = 32u * (uint32_t)p.n_sm_warps;  // softmax threads
    WaitCtl wc{p.err, &bar.abort_flag, p.timeout_ns};

    if (threadIdx.x == 0) {
        bar.abort_flag = 0;
        mbar_init(&bar.q_full, 1);
        mbar_init(&bar.q_empty, 1);
        for (int s = 0; s < Cfg::kSlots; ++s) {
            mbar_init(&bar.slot_full[s], 1);
            mbar_init(&bar.slot_empty[s], 1);
        }
        mbar_init(&bar.s_full, 1);
        mbar_init(&bar.s_free, n_sm);
        mbar_init(&bar.p_full, n_sm);
        mbar_init(&bar.pv_done, 1);
        mbar_init(&bar.o_empty, n_sm);
        mbar_init(&bar.drain, 1);
        fence_mbar_init();
    }
    if (warp == 5) {
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
    const uint32_t sRing = smem_u32(smem + Cfg::kRingOff);

    if (warp == 4) {
        // ------------------------------------------------ Q / K / V producer
        if (elect_one()) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
        }
        __syncwarp();
        uint32_t n = 0, n_units = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x, ++n_units) {
            const DtcUnit w = dtc_unit(p, u);
            ok = mbar_wait_warp(&bar.q_empty, (n_units & 1) ^ 1, wc);
            if (!ok) break;
            if (elect_one()) {  // rows nq .. 127 of the box lie beyond the tensor: zero-filled
                mbar_arrive_expect_tx(&bar.q_full, Cfg::kTileBytes);
                for (int bx = 0; bx < Cfg::kBoxes; ++bx)
                    tma_load_4d(smem + Cfg::kQOff + bx * BM * 128, &tm_q, &bar.q_full, bx * 64, 0, w.h, w.b);
            }
            __syncwarp();
            for (int t = 0; t < 2 * w.ntiles && ok; ++t, ++n) {
                bool is_k;
                int j;
                kv_item(t, w.ntiles, &is_k, &j);
                const uint32_t s = n % Cfg::kSlots;
                ok = mbar_wait_warp(&bar.slot_empty[s], ((n / Cfg::kSlots) & 1) ^ 1, wc);
                if (!ok) break;
                if (elect_one()) {
                    mbar_arrive_expect_tx(&bar.slot_full[s], Cfg::kTileBytes);
                    uint8_t* dst = smem + Cfg::kRingOff + s * Cfg::kTileBytes;
                    for (int bx = 0; bx < Cfg::kBoxes; ++bx)
                        tma_load_4d(dst + bx * BN * 128, is_k ? &tm_k : &tm_v, &bar.slot_full[s], bx * 64,
                                    w.key0 + j * BN, w.h, w.b);
                }
                __syncwarp();
            }
        }
        if (lane == 0) {
            const uint32_t last = n < (uint32_t)Cfg::kSlots ? n : (uint32_t)Cfg::kSlots;
            for (uint32_t i = n - last; i < n; ++i)
                drain_wait(&bar.slot_full[i % Cfg::kSlots], (i / Cfg::kSlots) & 1, p.timeout_ns);
            if (n_units > 0) drain_wait(&bar.q_full, (n_units - 1) & 1, p.timeout_ns);
        }
    } else if (warp == 5) {
        // ------------------------------------------------ MMA issuer
        const uint32_t tS = tmem, tP = tmem + 128, tO = tmem + 256;
        uint32_t n = 0, n_units = 0, n_s = 0, n_p = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x, ++n_units) {
            const DtcUnit w = dtc_unit(p, u);
            ok = mbar_wait_warp(&bar.q_full, n_units & 1, wc);
            if (!ok) break;
            tc_fence_after();
            for (int t = 0; t < 2 * w.ntiles && ok; ++t, ++n) {
                bool is_k;
                int j;
                kv_item(t, w.ntiles, &is_k, &j);
                const uint32_t s = n % Cfg::kSlots;
                if (is_k) {  // S = Q K_j^T once the softmax warps have read the previous S
                    if (n_s > 0) {
                        ok = mbar_wait_warp(&bar.s_free, (n_s - 1) & 1, wc);
                        if (!ok) break;
                    }
                    ++n_s;
                } else {  // O += P_j V_j once P_j is stored (the unit's first product after the last epilogue)
                    if (j == 0) {
                        ok = mbar_wait_warp(&bar.o_empty, (n_units & 1) ^ 1, wc);
                        if (!ok) break;
                    }
                    ok = mbar_wait_warp(&bar.p_full, n_p & 1, wc);
                    if (!ok) break;
                    ++n_p;
                }
                ok = mbar_wait_warp(&bar.slot_full[s], (n / Cfg::kSlots) & 1, wc);
                if (!ok) break;
                tc_fence_after();
                const uint32_t tile = sRing + s * Cfg::kTileBytes;
                if (elect_one()) {
                    if (is_k) {
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk)
                            mma_ss(tS, kmajor_desc(sQ, kk), kmajor_desc(tile, kk), kIdescS, kk > 0 ? 1u : 0u);
                        mma_commit(&bar.slot_empty[s]);
                        mma_commit(&bar.s_full);
                        if (j == w.ntiles - 1) mma_commit(&bar.q_empty);  // last read of Q
                    } else {
#pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk)
                            mma_ts(tO, tP + kk * 8, vmajor_desc(tile, kk), kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
                        mma_commit(&bar.slot_empty[s]);
                        mma_commit(&bar.pv_done);
                    }
                }
                __syncwarp();
            }
        }
        if (elect_one()) {
            mma_commit(&bar.drain);
            drain_wait(&bar.drain, 0, p.timeout_ns);
        }
        __syncwarp();
    } else if (warp < p.n_sm_warps) {
        // ------------------------------------------------ softmax (thread = query row)
        const int r = warp * 32 + lane;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const uint32_t tS = tmem + lane_off, tP = tmem + lane_off + 128, tO = tmem + lane_off + 256;
        uint32_t scnt = 0, pvcnt = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
            const DtcUnit w = dtc_unit(p, u);
            // keys this row may see: [key0, lim)
            const int lim = p.causal ? min(w.key_end, p.nk - p.nq + r + 1) : w.key_end;
            float m_ref = -INFINITY, m_row = -INFINITY, l = 0.f;
            for (int j = 0; j < w.ntiles; ++j) {
                ok = mbar_wait(&bar.s_full, scnt & 1, wc);
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
                tc_fence_before();
                mbar_arrive(&bar.s_free);
                const int first_out = lim - (w.key0 + j * BN);  // first column this row may not see
#pragma unroll
                for (int col = 0; col < BN; ++col)
                    su[col] = __float_as_uint(col < first_out ? __uint_as_float(su[col]) * p.c : -INFINITY);
                float mx[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float m = fmaxf(__uint_as_float(su[16 * c]), __uint_as_float(su[16 * c + 1]));
#pragma unroll
                    for (int e = 2; e < 16; e += 2)
                        m = fmax3(m, __uint_as_float(su[16 * c + e]), __uint_as_float(su[16 * c + e + 1]));
                    mx[c] = m;
                }
                const float m_tile = fmaxf(fmax3(fmax3(mx[0], mx[1], mx[2]), mx[3], mx[4]), fmax3(mx[5], mx[6], mx[7]));
                m_row = fmaxf(m_row, m_tile);
                float m_new = m_ref;
                if (m_tile > m_ref + kRescaleThreshold) m_new = m_tile;
                const bool moved = m_new != m_ref;
                const float alpha = moved ? ex2(m_ref - m_new) : 1.f;
                const bool rescale = j > 0 && __any_sync(0xffffffffu, moved && m_ref != -INFINITY);
                m_ref = m_new;
                const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;
                float2 suma = make_float2(0.f, 0.f), sumb = make_float2(0.f, 0.f);
#pragma unroll
                for (int i = 0; i < BN / 2; ++i) {
                    const float2 x = fadd2(make_float2(__uint_as_float(su[2 * i]), __uint_as_float(su[2 * i + 1])),
                                           make_float2(neg_m, neg_m));
                    const float2 pp = make_float2(ex2(x.x), ex2(x.y));
                    if (i & 1)
                        sumb = fadd2(sumb, pp);
                    else
                        suma = fadd2(suma, pp);
                    su[i] = pack_h16<F16>(pp.x, pp.y);
                }
                if (j > 0) {  // the product of tile j-1 has read P and written O
                    ok = mbar_wait(&bar.pv_done, pvcnt & 1, wc);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    ++pvcnt;
                    tc_fence_after();
                    if (rescale) {
#pragma unroll 1
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
                    }
                }
                tmem_st32_at<0>(tP + 0, su);
                tmem_st32_at<32>(tP + 32, su);
                l = l * alpha + ((suma.x + suma.y) + (sumb.x + sumb.y));
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bar.p_full);
            }
            if (!ok) break;
            // the split's partial state of this row: m (log2 units), l and the unnormalised o
            ok = mbar_wait(&bar.pv_done, pvcnt & 1, wc);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            ++pvcnt;
            tc_fence_after();
            float* rec = p.part + (((long long)w.bh * p.splits + w.split) * p.nq + r) * (D + 4);
            if (r < p.nq) {
                rec[0] = l > 0.f ? m_ref : -INFINITY;
                rec[1] = l;
                rec[2] = o_divisor<F16>(l, m_row, m_ref);  // divisor of o (see o_divisor)
            }
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t ov[32];
                tmem_ld32(tO + c0, ov);
                tmem_wait_ld();
                if (r < p.nq) {
                    float4* dst = reinterpret_cast<float4*>(rec + 4 + c0);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        dst[q] = make_float4(__uint_as_float(ov[4 * q]), __uint_as_float(ov[4 * q + 1]),
                                             __uint_as_float(ov[4 * q + 2]), __uint_as_float(ov[4 * q + 3]));
                }
            }
            tc_fence_before();
            mbar_arrive(&bar.o_empty);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_decode_tc(const attn_decode_params& prm, const DecodeSplit& plan, const DecodeMaps& maps,
                             const LaunchCommon& lc, cudaStream_t s) {
    DtcParams p{};
    p.B = prm.B;
    p.H = prm.H;
    p.nq = prm.nq;
    p.nk = prm.nk;
    p.causal = prm.causal;
    p.splits = plan.splits;
    p.chunk = plan.chunk;
    p.num_units = prm.B * prm.H * plan.splits;
    p.n_sm_warps = (prm.nq + 31) / 32;
    p.c = prm.scale * kLog2e;
    p.part = static_cast<float*>(prm.workspace);
    p.err = lc.err;
    p.timeout_ns = lc.timeout_ns;
    const int grid = p.num_units < lc.num_sms ? p.num_units : lc.num_sms;
    const bool f16 = prm.dtype == ATTN_F16;
    cudaError_t e;
    if (prm.d == 64) {
        auto k = f16 ? decode_tc_kernel<64, true> : decode_tc_kernel<64, false>;
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, DtcCfg<64>::kSmemBytes)) !=
            cudaSuccess)
            return e;
        e = launch_pdl(k, dim3(grid), dim3(kThreads), DtcCfg<64>::kSmemBytes, s, maps.q, maps.k, maps.v, p);
    } else {
        auto k = f16 ? decode_tc_kernel<128, true> : decode_tc_kernel<128, false>;
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, DtcCfg<128>::kSmemBytes)) !=
            cudaSuccess)
            return e;
        e = launch_pdl(k, dim3(grid), dim3(kThreads), DtcCfg<128>::kSmemBytes, s, maps.q, maps.k, maps.v, p);
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace attn
