// attn_fwd_fp8.cu — attention forward with 8-bit floating-point (E4M3) Q, K, V
// on the sm_103a tensor cores (tcgen05 kind::f8f6f4).
//
// An FP8 forward pass computes the same exact attention at lower input
// precision ("What is FlashAttention?", FAQ on FlashAttention-3: FP16 and
// BF16 forward and backward and an FP8 forward pass). Q, K and V arrive as
// E4M3 codes with one descale factor per tensor: the values they stand for
// are code x descale. The products run at twice the 16-bit rate:
//   S = Q K^T               (E4M3 x E4M3 -> fp32 in tensor memory)
//   s = c S  with c = scale * log2(e) * q_descale * k_descale
//   P = 2^(s - m)  rounded to E4M3 (the A operand of the next product)
//   O += P V                (E4M3 x E4M3 -> fp32)
//   O_out = v_descale * O / l in bf16,  LSE = ln 2 * (m + log2 l)
// l sums the unrounded fp32 probabilities, so O / l is a weighted mean whose
// weights are off by at most the E4M3 rounding of P (3 fraction bits:
// 2^-4 relative for probabilities of 2^-6 and above).
//
// The loop, the warp roles and the online softmax are those of the 16-bit
// d = 128 forward ("What is FlashAttention?", Step 3 loop order;
// "Explain FlashAttention and why it is IO-aware", "Keep only the state needed
// for the final weighted average"): one persistent CTA per SM over units of
// (b, h, 256 query rows), two 128-row query tiles whose softmax warpgroups
// take turns with the tensor core, a reference max that moves only when a
// tile's max exceeds it by more than 8 (so P <= 2^8, inside E4M3's range of
// 448), and all-masked rows giving O = 0 and LSE = -inf.
//
// Warp roles (12 warps):
//   warps 0-3 / 4-7  softmax of query tile 0 / 1 (one thread per row)
//   warp  8          TMA producer: Q tiles, then K_j, V_j into a ring
//   warp  9          TMEM allocator and MMA issuer
//   warp 10          TMA producer of the bf16 additive mask tiles (mask variant)
//   warp 11          idle
//
// Shared memory: a 128 x 128 E4M3 tile is 16 KB, one 128-byte-swizzled box
// (128 rows of 128 bytes), so the K/V ring has 8 stages (6 with the mask).
// V is read MN-major (d contiguous) as the B operand of P V.
// Tensor memory (lane = query row): S_0 [0,128), S_1 [128,256) fp32, with
// P_t as E4M3 quads in the first 32 columns of S_t; O_0 [256,384), O_1 [384,512).
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "ptx_f8.cuh"

namespace attn {
namespace {

using namespace ptx;
using namespace ptx_f8;

constexpr int D = 128;
constexpr int BM = 128;
constexpr int BN = 128;
constexpr float kRescaleThreshold = 8.0f;
constexpr int kTileBytes = BM * D;  // one E4M3 tile
constexpr int kMaskBytes = BM * BN * 2;

template <bool MASK>
struct F8Cfg {
    static constexpr int kStages = MASK ? 6 : 8;
    static constexpr int kWarps = 12;
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kSoftmaxRegs = 216;
    static constexpr int kOtherRegs = 72;
    static_assert(2 * 128 * kSoftmaxRegs + 128 * kOtherRegs <= 384 * 168, "register split");
    static constexpr int kQOff = 0;
    static constexpr int kKVOff = kQOff + 2 * kTileBytes;
    static constexpr int kMaskOff = kKVOff + kStages * kTileBytes;
    static constexpr int kBarOff = kMaskOff + (MASK ? 2 * kMaskBytes : 0);
    static constexpr int kSmemBytes = kBarOff + 256 + 1024;
};

struct F8Params {
    int B, H, N;
    int causal;
    float c;          // scale * log2(e) * q_descale * k_descale
    float v_descale;
    float* lse;
    __nv_bfloat16* o;
    long long o_sb, o_sh, o_sn;
    int mask_hb, mask_bb;
    int num_units, n_qblk;
    int head_major;
    int* err;
    unsigned long long timeout_ns;
};

struct __align__(8) F8Barriers {
    uint64_t q_full, q_empty;
    uint64_t kv_full[8], kv_empty[8];
    uint64_t s_full[2], p_full[2], o_full[2], o_empty[2];
    uint64_t m_full[2], m_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(F8Barriers) <= 256, "barrier area");

struct F8Unit {
    int b, h;
    int row0[2];
    int nkv[2];
    int nkv_max;
};

__device__ __forceinline__ F8Unit f8_unit(const F8Params& p, int u) {
    F8Unit w;
    const int bh = p.B * p.H;
    int r, qblk;
    if (p.head_major) {
        r = u / p.n_qblk;
        qblk = u % p.n_qblk;
    } else {
        qblk = p.n_qblk - 1 - u / bh;
        r = u % bh;
    }
    w.b = r / p.H;
    w.h = r % p.H;
    const int nk_all = (p.N + BN - 1) / BN;
    for (int t = 0; t < 2; ++t) {
        w.row0[t] = qblk * 2 * BM + t * BM;
        w.nkv[t] = w.row0[t] >= p.N ? 0 : (p.causal ? min(nk_all, w.row0[t] / BN + 1) : nk_all);
    }
    w.nkv_max = max(w.nkv[0], w.nkv[1]);
    return w;
}

__device__ __forceinline__ int unit_at(int k) {
    const int g = gridDim.x, i = blockIdx.x;
    return k * g + ((k & 1) ? g - 1 - i : i);
}

// K-major E4M3 tile (128 rows of 128 bytes, 128-byte swizzle) at k-step kk (32 elements).
__device__ __forceinline__ uint64_t kdesc8(uint32_t tile, int kk) { return sdesc_sw128(tile + kk * 32, 16, 1024); }
// V (keys x 128 bytes of d) read MN-major at k-step kk (32 keys). d spans one 128-byte
// swizzle row, so the offset between column blocks is never used.
__device__ __forceinline__ uint64_t vdesc8(uint32_t tile, int kk) {
    return sdesc_sw128(tile + kk * (32 * 128), kTileBytes, 1024);
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(a, parity))
        if (globaltimer() - t0 > timeout_ns) break;
}

template <bool MASK>
__global__ void __launch_bounds__(F8Cfg<MASK>::kThreads, 1)
    fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_mask,
                   const F8Params p) {
    using Cfg = F8Cfg<MASK>;
    constexpr uint32_t kIdescS = idesc_e4m3(BM, BN, false, false);
    constexpr uint32_t kIdescO = idesc_e4m3(BM, D, false, true);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    F8Barriers& bar = *reinterpret_cast<F8Barriers*>(smem + Cfg::kBarOff);
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
            mbar_init(&bar.p_full[t], BM);
            mbar_init(&bar.o_full[t], 1);
            mbar_init(&bar.o_empty[t], BM);
            mbar_init(&bar.m_full[t], 1);
            mbar_init(&bar.m_empty[t], BM);
        }
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
    const uint32_t sKV = smem_u32(smem + Cfg::kKVOff);

    if (warp >= 8) {
      regs_decrease<Cfg::kOtherRegs>();
      if (warp == 8) {
        // ------------------------------------------------ Q / K / V producer
        if (elect_one()) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
        }
        __syncwarp();
        uint32_t it = 0, n_units = 0;
        bool ok = true;
        for (int ku = 0, u = unit_at(0); u < p.num_units && ok; u = unit_at(++ku), ++n_units) {
            const F8Unit w = f8_unit(p, u);
            ok = mbar_wait_warp(&bar.q_empty, (n_units & 1) ^ 1, wc);
            if (!ok) break;
            const int nt = w.nkv[1] > 0 ? 2 : 1;
            if (elect_one()) {
                mbar_arrive_expect_tx(&bar.q_full, nt * kTileBytes);
                for (int t = 0; t < nt; ++t)
                    tma_load_4d(smem + Cfg::kQOff + t * kTileBytes, &tm_q, &bar.q_full, 0, w.row0[t], w.h, w.b);
            }
            __syncwarp();
            for (int j = 0; j < w.nkv_max && ok; ++j) {
                for (int kv = 0; kv < 2; ++kv, ++it) {
                    const uint32_t s = it % Cfg::kStages;
                    ok = mbar_wait_warp(&bar.kv_empty[s], ((it / Cfg::kStages) & 1) ^ 1, wc);
                    if (!ok) break;
                    if (elect_one()) {
                        mbar_arrive_expect_tx(&bar.kv_full[s], kTileBytes);
                        tma_load_4d(smem + Cfg::kKVOff + s * kTileBytes, kv == 0 ? &tm_k : &tm_v, &bar.kv_full[s], 0,
                                    j * BN, w.h, w.b);
                    }
                    __syncwarp();
                }
            }
        }
        if (lane == 0) {
            const uint32_t last = it < (uint32_t)Cfg::kStages ? it : (uint32_t)Cfg::kStages;
            for (uint32_t i = it - last; i < it; ++i)
                drain_wait(&bar.kv_full[i % Cfg::kStages], (i / Cfg::kStages) & 1, p.timeout_ns);
            if (n_units > 0) drain_wait(&bar.q_full, (n_units - 1) & 1, p.timeout_ns);
        }
      } else if (MASK && warp == 10) {
        // ------------------------------------------------ mask producer (bf16 mask tiles)
        if (lane == 0) {
            prefetch_tmap(&tm_mask);
            uint32_t cnt[2] = {0, 0};
            bool ok = true;
            for (int ku = 0, u = unit_at(0); u < p.num_units && ok; u = unit_at(++ku)) {
                const F8Unit w = f8_unit(p, u);
                const int hm = p.mask_hb ? w.h : 0, bm = p.mask_bb ? w.b : 0;
                for (int j = 0; j < w.nkv_max && ok; ++j) {
                    for (int t = 0; t < 2; ++t) {
                        if (j >= w.nkv[t]) continue;
                        ok = mbar_wait(&bar.m_empty[t], (cnt[t] & 1) ^ 1, wc);
                        if (!ok) break;
                        mbar_arrive_expect_tx(&bar.m_full[t], kMaskBytes);
                        uint8_t* dst = smem + Cfg::kMaskOff + t * kMaskBytes;
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
      } else if (warp == 9) {
        // ------------------------------------------------ MMA issuer
        // Per key tile j and query tile t: O_t += P_t^{j-1} V_{j-1}, then S_t^j = Q_t K_j^T. One
        // thread's MMAs run in issue order, so S_t^j overwrites P_t^{j-1} only after the product
        // that reads it, and the commit that signals S_t^j also covers that product.
        uint32_t it = 0, n_units = 0, pcnt[2] = {0, 0}, ocnt[2] = {0, 0};
        bool ok = true;
        for (int ku = 0, u = unit_at(0); u < p.num_units && ok; u = unit_at(++ku), ++n_units) {
            const F8Unit w = f8_unit(p, u);
            ok = mbar_wait_warp(&bar.q_full, n_units & 1, wc);
            if (!ok) break;
            tc_fence_after();
            for (int j = 0; j <= w.nkv_max && ok; ++j) {
                const uint32_t itK = it;
                const uint32_t sK = itK % Cfg::kStages, sV_prev = (itK + Cfg::kStages - 1) % Cfg::kStages;
                if (j < w.nkv_max) {
                    ok = mbar_wait_warp(&bar.kv_full[sK], (itK / Cfg::kStages) & 1, wc);
                    if (!ok) break;
                }
                if (j > 0) {
                    ok = mbar_wait_warp(&bar.kv_full[sV_prev], ((itK - 1) / Cfg::kStages) & 1, wc);
                    if (!ok) break;
                }
                tc_fence_after();
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (!ok || w.nkv[t] == 0 || j > w.nkv[t]) continue;
                    const uint32_t tS = tmem + t * BN, tO = tmem + 256 + t * D;
                    if (j > 0) {
                        if (j == 1) {  // the unit's first product overwrites O_t: its epilogue is done
                            ok = mbar_wait_warp(&bar.o_empty[t], (ocnt[t] & 1) ^ 1, wc);
                            if (!ok) continue;
                        }
                        ok = mbar_wait_warp(&bar.p_full[t], pcnt[t] & 1, wc);
                        if (!ok) continue;
                        ++pcnt[t];
                        tc_fence_after();
                        const uint32_t vt = sKV + sV_prev * kTileBytes;
                        if (elect_one()) {
#pragma unroll
                            for (int kk = 0; kk < BN / 32; ++kk)
                                mma_f8_ts(tO, tS + kk * 8, vdesc8(vt, kk), kIdescO, (j > 1 || kk > 0) ? 1u : 0u);
                        }
                        __syncwarp();
                    }
                    if (j < w.nkv[t]) {
                        const uint32_t qt = sQ + t * kTileBytes, kt = sKV + sK * kTileBytes;
                        if (elect_one()) {
#pragma unroll
                            for (int kk = 0; kk < D / 32; ++kk)
                                mma_f8_ss(tS, kdesc8(qt, kk), kdesc8(kt, kk), kIdescS, kk > 0 ? 1u : 0u);
                            mma_commit(&bar.s_full[t]);
                        }
                        __syncwarp();
                    } else {
                        if (elect_one()) mma_commit(&bar.o_full[t]);  // last product of this tile issued
                        __syncwarp();
                        ++ocnt[t];
                    }
                }
                if (!ok) break;
                if (elect_one()) {
                    if (j == w.nkv_max - 1) mma_commit(&bar.q_empty);
                    if (j < w.nkv_max) mma_commit(&bar.kv_empty[sK]);
                    if (j > 0) mma_commit(&bar.kv_empty[sV_prev]);
                }
                __syncwarp();
                if (j < w.nkv_max) it += 2;
            }
        }
        if (elect_one()) {
            mma_commit(&bar.drain);
            drain_wait(&bar.drain, 0, p.timeout_ns);
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
        const uint8_t* mtile = smem + Cfg::kMaskOff + t * kMaskBytes;
        uint32_t scnt = 0, mcnt = 0, ocnt = 0;
        bool ok = true;
        for (int ku = 0, u = unit_at(0); u < p.num_units && ok; u = unit_at(++ku)) {
            const F8Unit w = f8_unit(p, u);
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
                const bool diag = p.causal && (j == nkv - 1);
                const bool tail = (j + 1) * BN > p.N;
                float cc = p.c;
                if (MASK || diag || tail) {
                    const int key0 = j * BN;
                    const int lim = min(diag ? row - key0 + 1 : BN, p.N - key0);  // first masked column
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
                                    const float2 f = unpack_h16<false>(mw[e]);
                                    const int col = bx * 64 + ch * 8 + 2 * e;
                                    su[col] = __float_as_uint(fmaf(__uint_as_float(su[col]), p.c, f.x * kLog2e));
                                    su[col + 1] =
                                        __float_as_uint(fmaf(__uint_as_float(su[col + 1]), p.c, f.y * kLog2e));
                                }
                            }
                        }
                        mbar_arrive(&bar.m_empty[t]);
                    } else {
#pragma unroll
                        for (int col = 0; col < BN; ++col) su[col] = __float_as_uint(__uint_as_float(su[col]) * p.c);
                    }
#pragma unroll
                    for (int col = 0; col < BN; ++col)
                        if (col >= lim) su[col] = __float_as_uint(-INFINITY);
                    cc = 1.f;
                }
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
                const float alpha = moved ? ex2(m_ref - m_new) : 1.f;
                const bool rescale = j > 0 && __any_sync(0xffffffffu, moved && m_ref != -INFINITY);
                if (rescale) {  // the product of key tile j-1 precedes S_t^j, so O_t is final for it
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
                }
                m_ref = m_new;
                const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;
                const float2 cc2 = make_float2(cc, cc), nm2 = make_float2(neg_m, neg_m);
                float2 suma = make_float2(0.f, 0.f), sumb = make_float2(0.f, 0.f);
                // P as E4M3 quads packed into su[0..31] (quad i from columns 4i..4i+3, already read)
#pragma unroll
                for (int i = 0; i < BN / 4; ++i) {
                    const float2 xa = ffma2(
                        make_float2(__uint_as_float(su[4 * i]), __uint_as_float(su[4 * i + 1])), cc2, nm2);
                    const float2 xb = ffma2(
                        make_float2(__uint_as_float(su[4 * i + 2]), __uint_as_float(su[4 * i + 3])), cc2, nm2);
                    const float2 pa = make_float2(ex2(xa.x), ex2(xa.y));
                    const float2 pb = make_float2(ex2(xb.x), ex2(xb.y));
                    suma = fadd2(suma, pa);
                    sumb = fadd2(sumb, pb);
                    su[i] = pack_e4m3x4(pa.x, pa.y, pb.x, pb.y);
                }
                tmem_st32_at<0>(tS, su);
                l = l * alpha + ((suma.x + suma.y) + (sumb.x + sumb.y));
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bar.p_full[t]);
            }
            if (!ok) break;
            // epilogue: v_descale * O / l in bf16 (0 for fully masked rows), LSE in natural log
            ok = mbar_wait(&bar.o_full[t], ocnt & 1, wc);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            ++ocnt;
            tc_fence_after();
            const float den = o_divisor_e4m3(l, m_row, m_ref);
            const float inv = den > 0.f ? p.v_descale / den : 0.f;
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
                        v.x = pack_bf16(__uint_as_float(ov[8 * q + 0]) * inv, __uint_as_float(ov[8 * q + 1]) * inv);
                        v.y = pack_bf16(__uint_as_float(ov[8 * q + 2]) * inv, __uint_as_float(ov[8 * q + 3]) * inv);
                        v.z = pack_bf16(__uint_as_float(ov[8 * q + 4]) * inv, __uint_as_float(ov[8 * q + 5]) * inv);
                        v.w = pack_bf16(__uint_as_float(ov[8 * q + 6]) * inv, __uint_as_float(ov[8 * q + 7]) * inv);
                        dst[q] = v;
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&bar.o_empty[t]);
            if (row < p.N)
                p.lse[((long long)w.b * p.H + w.h) * p.N + row] = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tmem, 512);
}

template <bool MASK>
cudaError_t launch_f8(const attn_fwd_fp8_params& prm, const Fp8Maps& maps, const LaunchCommon& lc, cudaStream_t s) {
    using Cfg = F8Cfg<MASK>;
    static_assert(Cfg::kSmemBytes <= 232448, "shared memory budget");
    cudaError_t e =
        cudaFuncSetAttribute(fwd_fp8_kernel<MASK>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    const attn_fwd_params& f = prm.f;
    F8Params p{};
    p.B = f.B;
    p.H = f.H;
    p.N = f.N;
    p.causal = f.causal;
    p.c = f.scale * kLog2e * prm.q_descale * prm.k_descale;
    p.v_descale = prm.v_descale;
    p.lse = f.lse;
    p.o = static_cast<__nv_bfloat16*>(f.o);
    p.o_sb = f.o_stride[0];
    p.o_sh = f.o_stride[1];
    p.o_sn = f.o_stride[2];
    p.mask_hb = f.mask ? (f.mask_stride[1] != 0) : 0;
    p.mask_bb = f.mask ? (f.mask_stride[0] != 0) : 0;
    p.n_qblk = (f.N + 2 * BM - 1) / (2 * BM);
    p.head_major = !f.causal && !MASK;
    p.num_units = p.n_qblk * f.B * f.H;
    p.err = lc.err;
    p.timeout_ns = lc.timeout_ns;
    const int grid = p.num_units < lc.num_sms ? p.num_units : lc.num_sms;
    e = launch_pdl(fwd_fp8_kernel<MASK>, dim3(grid), dim3(Cfg::kThreads), Cfg::kSmemBytes, s, maps.q, maps.k, maps.v,
                   maps.mask, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_fp8(const attn_fwd_fp8_params& p, const Fp8Maps& maps, const LaunchCommon& lc,
                           cudaStream_t s) {
    return p.f.mask ? launch_f8<true>(p, maps, lc, s) : launch_f8<false>(p, maps, lc, s);
}

}  // namespace attn
