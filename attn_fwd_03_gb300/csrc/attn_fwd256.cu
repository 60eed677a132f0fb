// attn_fwd256.cu — attention forward with head dim 256 on the sm_103a tensor cores,
// for bf16, IEEE half and E4M3 (8-bit, the FP8 forward) inputs.
//
// The same FlashAttention-2 loop as the d = 64 / 128 forward ("What is
// FlashAttention?", Step 3): a query tile stays on chip, key/value tiles
// stream past, the online softmax keeps a running max and sum per row and the
// N x N scores exist one 128 x 128 tile at a time in tensor memory. What
// changes at d = 256 is the room:
//   - tensor memory: the fp32 O tile alone takes 256 of the 512 columns, so a
//     CTA holds one 128-row query tile (S 128 columns, P 64, O 256);
//   - shared memory: the Q tile is 64 KB and a K or V tile another 64 KB, so
//     K and V stream through a ring of eight 16 KB slots (a 64-column box of a
//     K tile, or 32 keys x 256 columns of a V tile) instead of whole tiles.
//     A slot is refilled as soon as the products that read it are done, so
//     the next tile's loads overlap the current tile's products.
// P has its own tensor-memory columns (as in the d = 64 forward), so S of key
// tile j + 1 is computed while the softmax warps still work on tile j:
//   issue order  S_0, S_1, PV_0, S_2, PV_1, ..., S_{n-1}, PV_{n-2}, PV_{n-1}
// and the ring is filled in the same order (K_0, K_1, V_0, K_2, V_1, ...).
//
// One persistent CTA per SM walks work units (b, h, 128-row query tile),
// heaviest causal tiles first in a snake order, heads outermost when every
// unit weighs the same.
//
// Warp roles (8 warps):
//   warps 0-3  softmax (one thread per query row)
//   warp  4    TMA producer: Q, then the K/V slots
//   warp  5    TMEM allocator and MMA issuer
//   warp  6    TMA producer of the additive mask tiles (mask variant only)
//   warp  7    idle
//
// Tensor memory (512 columns x 128 lanes, lane = query row):
//   [0,128) S (fp32)   [128,192) P (16-bit pairs)   [256,512) O (fp32)
//
// E4M3 inputs (kind::f8f6f4) take half the bytes: the Q tile is 32 KB, a K
// slot holds 128 keys x 128 columns and a V slot 64 keys x 256 columns, and P
// is rounded to E4M3 (32 TMEM columns); the Q and K descales fold into c and
// the V descale into the epilogue, and O is bf16.
//
// Online softmax as in the other forward ("Explain FlashAttention and why it
// is IO-aware", "Keep only the state needed for the final weighted average";
// "FlashAttention", "Why it is allowed to be exact"): log2 domain with
// c = scale * log2(e), a reference max that moves only when a tile's max
// exceeds it by more than 8, and then l and O are scaled by 2^(old - new).
// Fully masked rows return O = 0 and LSE = -inf.
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

constexpr int D = 256;
constexpr int BM = 128;  // query rows per tile
constexpr int BN = 128;  // keys per tile
constexpr float kRescaleThreshold = 8.0f;
constexpr int kSlotBytes = 16384;
constexpr int kSlots = 8;
constexpr int kMaskBytes = BM * BN * 2;  // the additive mask is 16-bit for every input type
constexpr int kThreads = 256;

// Input element types: bf16, IEEE half, or E4M3 (the FP8 forward, whose O is bf16).
enum : int { kBF16 = 0, kF16 = 1, kE4M3 = 2 };

// Layout of one element type. Every shared-memory tile is made of 128-byte-swizzled rows of
// 128 bytes, so the byte offsets of the MMA k-steps (32 bytes) are the same for both sizes.
template <int ET>
struct Elem {
    static constexpr bool kF8 = ET == kE4M3;
    static constexpr int kBytes = kF8 ? 1 : 2;
    static constexpr int kBoxCols = 128 / kBytes;         // elements per 128-byte row: 64 or 128
    static constexpr int kQBoxes = D / kBoxCols;          // 128-row boxes per Q tile: 4 or 2
    static constexpr int kQBytes = BM * D * kBytes;       // 64 or 32 KB
    static constexpr int kKSlots = D / kBoxCols;          // a K tile: one slot per box (4 or 2)
    static constexpr int kVKeys = kSlotBytes / (D * kBytes);  // keys per V slot: 32 or 64
    static constexpr int kVSlots = BN / kVKeys;           // 4 or 2
    static constexpr int kStepK = 32 / kBytes;            // elements per MMA k-step: 16 or 32
    static_assert(kKSlots == kVSlots, "K and V items take the same number of slots");
    static constexpr int kItemSlots = kKSlots;
};

template <bool MASK, int ET>
struct F256Cfg {
    static constexpr int kQOff = 0;
    static constexpr int kRingOff = kQOff + Elem<ET>::kQBytes;
    static constexpr int kMaskOff = kRingOff + kSlots * kSlotBytes;
    static constexpr int kBarOff = kMaskOff + (MASK ? kMaskBytes : 0);
    static constexpr int kSmemBytes = kBarOff + 256 + 1024;  // barriers + alignment slack
};

struct F256Params {
    int B, H, N;
    int causal;
    float c;          // scale * log2(e) (times the Q and K descales for E4M3)
    float o_factor;   // the V descale for E4M3, else 1
    float* lse;
    __nv_bfloat16* o;  // 16-bit output (bf16 or half bits)
    long long o_sb, o_sh, o_sn;
    int mask_hb, mask_bb;
    int n_qt, num_units, head_major;
    int* err;
    unsigned long long timeout_ns;
};

struct __align__(8) F256Barriers {
    uint64_t q_full, q_empty;
    uint64_t slot_full[kSlots], slot_empty[kSlots];
    uint64_t s_full, s_free, p_full, pv_done, o_empty;
    uint64_t m_full, m_empty;
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(F256Barriers) <= 256, "barrier area");

struct F256Unit {
    int b, h, qt, nkv;
};

__device__ __forceinline__ F256Unit f256_unit(const F256Params& p, int u) {
    F256Unit w;
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

__device__ __forceinline__ int unit_at(int k) {
    const int g = gridDim.x, i = blockIdx.x;
    return k * g + ((k & 1) ? g - 1 - i : i);
}

// Item t of a unit's K/V sequence (t < 2 nkv): K_0, then K_i, V_{i-1} for i = 1..nkv-1, then
// V_{nkv-1}. Sets *is_k and *tile.
__device__ __forceinline__ void kv_item(int t, int nkv, bool* is_k, int* tile) {
    if (t == 0) {
        *is_k = true;
        *tile = 0;
    } else if (t == 2 * nkv - 1) {
        *is_k = false;
        *tile = nkv - 1;
    } else {
        *is_k = (t & 1) != 0;
        *tile = *is_k ? (t + 1) / 2 : t / 2 - 1;
    }
}

// Descriptor of a K-major 128-row box (128-byte rows, 128-byte swizzle) at k-step kk within the box.
__device__ __forceinline__ uint64_t kbox_desc(uint32_t box, int kk) { return sdesc_sw128(box + kk * 32, 16, 1024); }
// Descriptor of a V slot (kVKeys keys x d, as 128-byte-wide boxes of kVKeys rows) read MN-major at
// k-step kk (kStepK keys).
template <int ET>
__device__ __forceinline__ uint64_t vslot_desc(uint32_t slot, int kk) {
    using E = Elem<ET>;
    return sdesc_sw128(slot + kk * (E::kStepK * 128), E::kVKeys * 128, 1024);
}
template <int ET>
__device__ __forceinline__ void mma_s(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    if constexpr (Elem<ET>::kF8)
        mma_f8_ss(d, a, b, idesc, acc);
    else
        mma_ss(d, a, b, idesc, acc);
}
template <int ET>
__device__ __forceinline__ void mma_t(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    if constexpr (Elem<ET>::kF8)
        mma_f8_ts(d, a, b, idesc, acc);
    else
        mma_ts(d, a, b, idesc, acc);
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(a, parity))
        if (globaltimer() - t0 > timeout_ns) break;
}

template <bool MASK, int ET>
__global__ void __launch_bounds__(kThreads, 1)
    fwd256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_mask,
                  const F256Params p) {
    using Cfg = F256Cfg<MASK, ET>;
    using E = Elem<ET>;
    constexpr bool F16 = ET == kF16;  // 16-bit storage of the mask (and of O) is half, else bf16
    constexpr uint32_t kIdescS = E::kF8 ? idesc_e4m3(BM, BN, false, false) : idesc_h16(BM, BN, false, false, F16);
    constexpr uint32_t kIdescO = E::kF8 ? idesc_e4m3(BM, D, false, true) : idesc_h16(BM, D, false, true, F16);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    F256Barriers& bar = *reinterpret_cast<F256Barriers*>(smem + Cfg::kBarOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    WaitCtl wc{p.err, &bar.abort_flag, p.timeout_ns};

    if (threadIdx.x == 0) {
        bar.abort_flag = 0;
        mbar_init(&bar.q_full, 1);
        mbar_init(&bar.q_empty, 1);
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&bar.slot_full[s], 1);
            mbar_init(&bar.slot_empty[s], 1);
        }
        mbar_init(&bar.s_full, 1);
        mbar_init(&bar.s_free, BM);
        mbar_init(&bar.p_full, BM);
        mbar_init(&bar.pv_done, 1);
        mbar_init(&bar.o_empty, BM);
        mbar_init(&bar.m_full, 1);
        mbar_init(&bar.m_empty, BM);
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
        uint32_t n = 0, n_units = 0;  // slots filled so far, units started
        bool ok = true;
        for (int ku = 0, u = unit_at(0); u < p.num_units && ok; u = unit_at(++ku), ++n_units) {
            const F256Unit w = f256_unit(p, u);
            ok = mbar_wait_warp(&bar.q_empty, (n_units & 1) ^ 1, wc);
            if (!ok) break;
            if (elect_one()) {
                mbar_arrive_expect_tx(&bar.q_full, E::kQBytes);
                for (int bx = 0; bx < E::kQBoxes; ++bx)
                    tma_load_4d(smem + Cfg::kQOff + bx * BM * 128, &tm_q, &bar.q_full, bx * E::kBoxCols, w.qt * BM,
                                w.h, w.b);
            }
            __syncwarp();
            for (int t = 0; t < 2 * w.nkv && ok; ++t) {
                bool is_k;
                int j;
                kv_item(t, w.nkv, &is_k, &j);
                for (int q4 = 0; q4 < E::kItemSlots; ++q4, ++n) {
                    const uint32_t s = n % kSlots;
                    ok = mbar_wait_warp(&bar.slot_empty[s], ((n / kSlots) & 1) ^ 1, wc);
                    if (!ok) break;
                    if (elect_one()) {
                        mbar_arrive_expect_tx(&bar.slot_full[s], kSlotBytes);
                        uint8_t* dst = smem + Cfg::kRingOff + s * kSlotBytes;
                        if (is_k) {  // box q4 (128-byte-wide columns) of K_j
                            tma_load_4d(dst, &tm_k, &bar.slot_full[s], q4 * E::kBoxCols, j * BN, w.h, w.b);
                        } else {  // keys [kVKeys q4, kVKeys (q4 + 1)) of V_j, as 128-byte-wide boxes
                            for (int bx = 0; bx < E::kQBoxes; ++bx)
                                tma_load_4d(dst + bx * E::kVKeys * 128, &tm_v, &bar.slot_full[s], bx * E::kBoxCols,
                                            j * BN + q4 * E::kVKeys, w.h, w.b);
                        }
                    }
                    __syncwarp();
                }
            }
        }
        // every copy issued must land before the CTA exits
        if (lane == 0) {
            const uint32_t last = n < (uint32_t)kSlots ? n : (uint32_t)kSlots;
            for (uint32_t i = n - last; i < n; ++i) drain_wait(&bar.slot_full[i % kSlots], (i / kSlots) & 1, p.timeout_ns);
            if (n_units > 0) drain_wait(&bar.q_full, (n_units - 1) & 1, p.timeout_ns);
        }
    } else if (MASK && warp == 6) {
        // ------------------------------------------------ mask producer
        if (lane == 0) {
            prefetch_tmap(&tm_mask);
            uint32_t cnt = 0;
            bool ok = true;
            for (int ku = 0, u = unit_at(0); u < p.num_units && ok; u = unit_at(++ku)) {
                const F256Unit w = f256_unit(p, u);
                const int hm = p.mask_hb ? w.h : 0, bm = p.mask_bb ? w.b : 0;
                for (int j = 0; j < w.nkv && ok; ++j, ++cnt) {
                    ok = mbar_wait(&bar.m_empty, (cnt & 1) ^ 1, wc);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&bar.m_full, kMaskBytes);
                    for (int bx = 0; bx < 2; ++bx)
                        tma_load_4d(smem + Cfg::kMaskOff + bx * BM * 128, &tm_mask, &bar.m_full, j * BN + bx * 64,
                                    w.qt * BM, hm, bm);
                }
            }
            if (cnt > 0) drain_wait(&bar.m_full, (cnt - 1) & 1, p.timeout_ns);
        }
    } else if (warp == 5) {
        // ------------------------------------------------ MMA issuer
        const uint32_t tS = tmem, tP = tmem + 128, tO = tmem + 256;
        uint32_t n = 0, n_units = 0, n_s = 0, n_p = 0;
        bool ok = true;
        for (int ku = 0, u = unit_at(0); u < p.num_units && ok; u = unit_at(++ku), ++n_units) {
            const F256Unit w = f256_unit(p, u);
            ok = mbar_wait_warp(&bar.q_full, n_units & 1, wc);
            if (!ok) break;
            tc_fence_after();
            for (int t = 0; t < 2 * w.nkv && ok; ++t) {
                bool is_k;
                int j;
                kv_item(t, w.nkv, &is_k, &j);
                if (is_k) {
                    // S = Q K_j^T once the softmax warps have read the previous S
                    if (n_s > 0) {
                        ok = mbar_wait_warp(&bar.s_free, (n_s - 1) & 1, wc);
                        if (!ok) break;
                    }
                    for (int bx = 0; bx < E::kItemSlots && ok; ++bx, ++n) {
                        const uint32_t s = n % kSlots;
                        ok = mbar_wait_warp(&bar.slot_full[s], (n / kSlots) & 1, wc);
                        if (!ok) break;
                        tc_fence_after();
                        if (elect_one()) {
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)  // four 32-byte k-steps per 128-byte row
                                mma_s<ET>(tS, kbox_desc(sQ + bx * BM * 128, kk), kbox_desc(sRing + s * kSlotBytes, kk),
                                          kIdescS, (bx > 0 || kk > 0) ? 1u : 0u);
                            mma_commit(&bar.slot_empty[s]);
                            if (bx == E::kItemSlots - 1) {
                                mma_commit(&bar.s_full);
                                if (j == w.nkv - 1) mma_commit(&bar.q_empty);  // last read of Q
                            }
                        }
                        __syncwarp();
                    }
                    ++n_s;
                } else {
                    // O += P_j V_j once the softmax warps have stored P_j (and rescaled O)
                    if (j == 0) {  // the unit's first product overwrites O: the last epilogue has read it
                        ok = mbar_wait_warp(&bar.o_empty, (n_units & 1) ^ 1, wc);
                        if (!ok) break;
                    }
                    ok = mbar_wait_warp(&bar.p_full, n_p & 1, wc);
                    if (!ok) break;
                    ++n_p;
                    for (int q4 = 0; q4 < E::kItemSlots && ok; ++q4, ++n) {
                        const uint32_t s = n % kSlots;
                        ok = mbar_wait_warp(&bar.slot_full[s], (n / kSlots) & 1, wc);
                        if (!ok) break;
                        tc_fence_after();
                        if (elect_one()) {
                            // kVKeys keys per slot in k-steps of kStepK; P holds 8 TMEM columns per k-step
#pragma unroll
                            for (int kk = 0; kk < E::kVKeys / E::kStepK; ++kk)
                                mma_t<ET>(tO, tP + (2 * q4 + kk) * 8, vslot_desc<ET>(sRing + s * kSlotBytes, kk),
                                          kIdescO, (j > 0 || q4 > 0 || kk > 0) ? 1u : 0u);
                            mma_commit(&bar.slot_empty[s]);
                            if (q4 == E::kItemSlots - 1) mma_commit(&bar.pv_done);
                        }
                        __syncwarp();
                    }
                }
            }
        }
        // every MMA this warp issued completes before TMEM is released
        if (elect_one()) {
            mma_commit(&bar.drain);
            drain_wait(&bar.drain, 0, p.timeout_ns);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ------------------------------------------------ softmax warpgroup
        const int r = warp * 32 + lane;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const uint32_t tS = tmem + lane_off, tP = tmem + lane_off + 128, tO = tmem + lane_off + 256;
        const uint8_t* mrow = smem + Cfg::kMaskOff + r * 128;
        uint32_t scnt = 0, pvcnt = 0, mcnt = 0;
        bool ok = true;
        for (int ku = 0, u = unit_at(0); u < p.num_units && ok; u = unit_at(++ku)) {
            const F256Unit w = f256_unit(p, u);
            const int row = w.qt * BM + r;
            float m_ref = -INFINITY, m_row = -INFINITY, l = 0.f;
            for (int j = 0; j < w.nkv; ++j) {
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
                mbar_arrive(&bar.s_free);  // S is in registers: the next S may overwrite it
                const bool diag = p.causal && (j == w.nkv - 1);
                const bool tail = (j + 1) * BN > p.N;
                float cc = p.c;
                if (MASK || diag || tail) {
                    const int key0 = j * BN;
                    const int lim_causal = diag ? row - key0 + 1 : BN;  // keys <= row survive
                    const int lim = min(lim_causal, p.N - key0);        // first masked column
                    if (MASK) {
                        ok = mbar_wait(&bar.m_full, mcnt & 1, wc);
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok) break;
                        ++mcnt;
#pragma unroll
                        for (int bx = 0; bx < 2; ++bx) {
#pragma unroll
                            for (int ch = 0; ch < 8; ++ch) {
                                const uint4 mv = *reinterpret_cast<const uint4*>(mrow + bx * BM * 128 +
                                                                                 ((ch ^ (r & 7)) << 4));
                                const uint32_t mw[4] = {mv.x, mv.y, mv.z, mv.w};
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const float2 f = unpack_h16<F16>(mw[e]);
                                    const int col = bx * 64 + ch * 8 + 2 * e;
                                    su[col] = __float_as_uint(fmaf(__uint_as_float(su[col]), p.c, f.x * kLog2e));
                                    su[col + 1] =
                                        __float_as_uint(fmaf(__uint_as_float(su[col + 1]), p.c, f.y * kLog2e));
                                }
                            }
                        }
                        mbar_arrive(&bar.m_empty);
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
                const float alpha = moved ? ex2(m_ref - m_new) : 1.f;  // 0 when m_ref = -inf
                const bool rescale = j > 0 && __any_sync(0xffffffffu, moved && m_ref != -INFINITY);
                m_ref = m_new;
                const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;
                const float2 cc2 = make_float2(cc, cc), nm2 = make_float2(neg_m, neg_m);
                float2 suma = make_float2(0.f, 0.f), sumb = make_float2(0.f, 0.f);
                if constexpr (E::kF8) {
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
                } else {
#pragma unroll
                    for (int i = 0; i < BN / 2; ++i) {
                        const float2 x =
                            ffma2(make_float2(__uint_as_float(su[2 * i]), __uint_as_float(su[2 * i + 1])), cc2, nm2);
                        const float2 pp = make_float2(ex2(x.x), ex2(x.y));
                        if (i & 1)
                            sumb = fadd2(sumb, pp);
                        else
                            suma = fadd2(suma, pp);
                        su[i] = pack_h16<F16>(pp.x, pp.y);
                    }
                }
                if (j > 0) {  // the product of key tile j-1 has read P and written O
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
                                const float2 r2 = fmul2(
                                    make_float2(__uint_as_float(ov[i]), __uint_as_float(ov[i + 1])),
                                    make_float2(alpha, alpha));
                                ov[i] = __float_as_uint(r2.x);
                                ov[i + 1] = __float_as_uint(r2.y);
                            }
                            tmem_st32(tO + c0, ov);
                        }
                    }
                }
                tmem_st32_at<0>(tP + 0, su);
                if constexpr (!E::kF8) tmem_st32_at<32>(tP + 32, su);
                l = l * alpha + ((suma.x + suma.y) + (sumb.x + sumb.y));
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bar.p_full);
            }
            if (!ok) break;
            // epilogue: O / l (0 for fully masked rows), LSE in natural log
            ok = mbar_wait(&bar.pv_done, pvcnt & 1, wc);  // the unit's last product
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            ++pvcnt;
            tc_fence_after();
            const float den = E::kF8 ? o_divisor_e4m3(l, m_row, m_ref) : o_divisor<F16>(l, m_row, m_ref);
            const float inv = den > 0.f ? p.o_factor / den : 0.f;
            __nv_bfloat16* orow = p.o + w.b * p.o_sb + w.h * p.o_sh + (long long)row * p.o_sn;
#pragma unroll 1
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
            mbar_arrive(&bar.o_empty);
            if (row < p.N)
                p.lse[((long long)w.b * p.H + w.h) * p.N + row] = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) tmem_dealloc(tmem, 512);
}

template <bool MASK, int ET>
cudaError_t launch256(const attn_fwd_params& prm, float c, float o_factor, const CUtensorMap& tm_q,
                      const CUtensorMap& tm_k, const CUtensorMap& tm_v, const CUtensorMap& tm_mask,
                      const LaunchCommon& lc, cudaStream_t s) {
    using Cfg = F256Cfg<MASK, ET>;
    static_assert(Cfg::kSmemBytes <= 232448, "shared memory budget");
    cudaError_t e =
        cudaFuncSetAttribute(fwd256_kernel<MASK, ET>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    F256Params p{};
    p.B = prm.B;
    p.H = prm.H;
    p.N = prm.N;
    p.causal = prm.causal;
    p.c = c;
    p.o_factor = o_factor;
    p.lse = prm.lse;
    p.o = static_cast<__nv_bfloat16*>(prm.o);
    p.o_sb = prm.o_stride[0];
    p.o_sh = prm.o_stride[1];
    p.o_sn = prm.o_stride[2];
    p.mask_hb = prm.mask ? (prm.mask_stride[1] != 0) : 0;
    p.mask_bb = prm.mask ? (prm.mask_stride[0] != 0) : 0;
    p.n_qt = (prm.N + BM - 1) / BM;
    p.num_units = p.n_qt * prm.B * prm.H;
    p.head_major = !prm.causal && !MASK;
    p.err = lc.err;
    p.timeout_ns = lc.timeout_ns;
    const int grid = p.num_units < lc.num_sms ? p.num_units : lc.num_sms;
    e = launch_pdl(fwd256_kernel<MASK, ET>, dim3(grid), dim3(kThreads), Cfg::kSmemBytes, s, tm_q, tm_k, tm_v, tm_mask,
                   p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd256(const attn_fwd_params& p, const FwdMaps& maps, const LaunchCommon& lc, cudaStream_t s) {
    const float c = p.scale * kLog2e;
    const bool mask = p.mask != nullptr, f16 = p.dtype == ATTN_F16;
    if (mask)
        return f16 ? launch256<true, kF16>(p, c, 1.f, maps.q, maps.k, maps.v32, maps.mask, lc, s)
                   : launch256<true, kBF16>(p, c, 1.f, maps.q, maps.k, maps.v32, maps.mask, lc, s);
    return f16 ? launch256<false, kF16>(p, c, 1.f, maps.q, maps.k, maps.v32, maps.mask, lc, s)
               : launch256<false, kBF16>(p, c, 1.f, maps.q, maps.k, maps.v32, maps.mask, lc, s);
}

cudaError_t launch_fwd256_fp8(const attn_fwd_fp8_params& p, const Fp8Maps& maps, const LaunchCommon& lc,
                              cudaStream_t s) {
    const float c = p.f.scale * kLog2e * p.q_descale * p.k_descale;
    if (p.f.mask) return launch256<true, kE4M3>(p.f, c, p.v_descale, maps.q, maps.k, maps.v64, maps.mask, lc, s);
    return launch256<false, kE4M3>(p.f, c, p.v_descale, maps.q, maps.k, maps.v64, maps.mask, lc, s);
}

}  // namespace attn
