// attn_bwd256.cu — attention backward at head dim 256 on the sm_103a tensor cores.
//
// The same recomputation as the other backward kernels ("What is FlashAttention?", Step 4;
// "FlashAttention", "What it does not do"):
//     P = exp(scale * Q K^T + mask - LSE),   dV = P^T dO,   dP = dO V^T,
//     dS = P * (dP - D),   dK = scale * dS^T Q,   dQ = scale * dS K,
// with D = rowsum(dO * O) and -LSE * log2(e) from the pre-pass.
//
// At head dim 256 the fp32 dK and dV of a 128-key tile would take all 512 tensor-memory
// columns, leaving none for the scores. A CTA therefore owns a 128-key tile and ONE half of
// the head dimension (columns 128 h .. 128 h + 127) of dK, dV and dQ; the two halves run as
// two CTAs. Each recomputes S^T and dP^T over the whole head dimension (their contraction
// needs all of it), so the path does 7/5 of the minimal tensor work:
//   per 64-query tile i:
//     S^T = K Q_i^T, dP^T = V dO_i^T          (M = 128 keys, N = 64 queries, K = 256)
//     P^T, dS^T (thread = key row)             bf16 pairs into tensor memory over the S^T
//                                              columns just read; dS^T also to shared memory
//     dK_h += dS^T Q_i[:, h], dV_h += P^T dO_i[:, h]        (A operand in tensor memory)
//     dQ_i[:, h]^T = K[:, h]^T dS^T            (M = 128 head-dim columns, N = 64 queries)
// and a drain warpgroup adds scale * dQ into the fp32 accumulator with vector reductions
// (a 4 x 4 transpose within each quad of lanes gives each lane four columns of one row).
//
// Tensor memory (512 columns x 128 lanes):
//   [0,64)     S^T (lane = key, column = query); then per 16 queries u: P^T bf16 pairs at
//              [16u, 16u+8), dS^T at [16u+8, 16u+16)
//   [64,128)   dP^T
//   [128,192)  dQ_h^T (lane = head-dim column of the half, column = query)
//   [256,384)  dV_h        [384,512)  dK_h
// Shared memory: K and V (128 x 256 each), the Q and dO tiles of the current query tile
// (64 x 256 each, released separately after dK and dV), the dS^T tile, the tile's row
// statistics and, with a mask, its 64 x 128 mask tile.
//
// Warps (16): 0-7 two softmax warpgroups (warpgroup g: queries [32g, 32g+32), thread = key
// row); 8-11 dQ drain (thread = head-dim column); 12 TMA producer; 13 TMEM allocator and MMA
// issuer; 14, 15 idle. At the end warpgroup 0 writes dV_h, warpgroup 1 scale * dK_h.
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

using namespace ptx;

constexpr int D = 256;
constexpr int BK = 128;  // keys per CTA
constexpr int BQ = 64;   // queries per tile
constexpr int DH = 128;  // head-dim columns of dK, dV, dQ per CTA

template <bool MASK>
struct B256Cfg {
    static constexpr int kKOff = 0;                     // 4 boxes of 128 keys x 64 columns
    static constexpr int kVOff = kKOff + BK * D * 2;
    static constexpr int kQOff = kVOff + BK * D * 2;    // 4 boxes of 64 queries x 64 columns
    static constexpr int kDoOff = kQOff + BQ * D * 2;
    static constexpr int kDsOff = kDoOff + BQ * D * 2;  // 128 keys x 64 queries
    static constexpr int kMaskOff = kDsOff + BK * BQ * 2;
    static constexpr int kMaskBytes = BQ * BK * 2;      // 2 boxes of 64 queries x 64 keys
    static constexpr int kStatsOff = kMaskOff + (MASK ? kMaskBytes : 0);
    static constexpr int kBarOff = kStatsOff + 512;
    static constexpr int kSmemBytes = kBarOff + 256;
    static constexpr int kThreads = 512;
};

struct B256Params {
    int B, H, N;
    int causal;
    float c;  // scale * log2(e)
    float scale;
    const float* stats;  // [B*H][ceil(N/128)][2][128]: -LSE*log2e, then -D
    float* dq_acc;       // [B, H, N, 256] fp32
    __nv_bfloat16 *dk, *dv;
    long long dk_sb, dk_sh, dk_sn, dv_sb, dv_sh, dv_sn;
    int mask_hb, mask_bb;
    int n_ktiles;
    int* err;
    unsigned long long timeout_ns;
};

struct __align__(8) B256Barriers {
    uint64_t kv_full;
    uint64_t q_full, q_empty, do_full, do_empty;
    uint64_t st_full, st_empty, m_full, m_empty;
    uint64_t s_full, ds_ready, ds_free, dq_full, dq_empty, kv_done, drain;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(B256Barriers) <= 256, "barrier block");

// K-major operand descriptor at k-step kk (16 columns): rows of 128 bytes in 64-column boxes
// of `rows` rows each.
__device__ __forceinline__ uint64_t kdesc(uint32_t tile, int kk, int rows) {
    return sdesc_sw128(tile + (kk >> 2) * (rows * 128) + (kk & 3) * 32, 16, 1024);
}
// MN-major operand descriptor at k-step kk (16 rows); `box` bytes between 64-element boxes
// along the M / N dimension.
__device__ __forceinline__ uint64_t mndesc(uint32_t tile, int kk, uint32_t box) {
    return sdesc_sw128(tile + kk * (16 * 128), box, 1024);
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(a, parity))
        if (globaltimer() - t0 > timeout_ns) break;
}

// 4 x 4 transpose within each quad of lanes: lane 4j + r holds x[q] = M[4j + r][q] on entry and
// M[4j + q][r] on exit, for M[lane][element].
__device__ __forceinline__ void quad_transpose(float (&x)[4], int r) {
    const bool odd = r & 1, hi = r & 2;
#pragma unroll
    for (int k = 0; k < 2; ++k) {  // exchange across lanes r, r ^ 1
        const float send = odd ? x[2 * k] : x[2 * k + 1];
        const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
        x[2 * k] = odd ? recv : x[2 * k];
        x[2 * k + 1] = odd ? x[2 * k + 1] : recv;
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {  // exchange across lanes r, r ^ 2
        const float send = hi ? x[e] : x[2 + e];
        const float recv = __shfl_xor_sync(0xffffffffu, send, 2);
        x[e] = hi ? recv : x[e];
        x[2 + e] = hi ? x[2 + e] : recv;
    }
}

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}
// 8 consecutive 32-bit TMEM columns from r[0 .. 7].
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

template <bool MASK, bool F16>
__global__ void __launch_bounds__(512, 1)
    bwd256_kernel(const __grid_constant__ CUtensorMap tm_q64, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do64,
                  const __grid_constant__ CUtensorMap tm_mask64, const B256Params p) {
    using Cfg = B256Cfg<MASK>;
    constexpr uint32_t kIdescS = idesc_h16(BK, BQ, false, false, F16);  // S^T, dP^T
    constexpr uint32_t kIdescKV = idesc_h16(BK, DH, false, true, F16);  // dK_h, dV_h (A in TMEM)
    constexpr uint32_t kIdescQ = idesc_h16(DH, BQ, true, true, F16);    // dQ_h^T = K_h^T dS^T
    extern __shared__ __align__(1024) uint8_t smem[];
    B256Barriers& bar = *reinterpret_cast<B256Barriers*>(smem + Cfg::kBarOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    WaitCtl wc{p.err, &bar.abort_flag, p.timeout_ns};

    // unit: half hf of the head dim for key tile kt of (b, h); heads outermost (L2 reuse of the
    // head's Q, dO and dQ accumulator), the two halves of a key tile next to each other
    const int hf = blockIdx.x & 1;
    const int kt = (blockIdx.x >> 1) % p.n_ktiles;
    const int bh_i = (blockIdx.x >> 1) / p.n_ktiles;
    const int b = bh_i / p.H, h = bh_i % p.H;
    const int k0 = kt * BK;
    const int nq_all = (p.N + BQ - 1) / BQ;
    const int i_begin = p.causal ? k0 / BQ : 0;  // first query tile reaching the key tile's first key
    const int n_it = nq_all - i_begin;

    if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled tiles need a 1024-byte aligned base
        if (threadIdx.x == 0) atomicExch(p.err, -7);
        return;
    }
    if (threadIdx.x == 0) {
        bar.abort_flag = 0;
        mbar_init(&bar.kv_full, 1);
        mbar_init(&bar.q_full, 1);
        mbar_init(&bar.q_empty, 1);
        mbar_init(&bar.do_full, 1);
        mbar_init(&bar.do_empty, 1);
        mbar_init(&bar.st_full, 1);
        mbar_init(&bar.st_empty, 256);
        mbar_init(&bar.m_full, 1);
        mbar_init(&bar.m_empty, 256);
        mbar_init(&bar.s_full, 1);
        mbar_init(&bar.ds_ready, 256);
        mbar_init(&bar.ds_free, 1);
        mbar_init(&bar.dq_full, 1);
        mbar_init(&bar.dq_empty, 128);
        mbar_init(&bar.kv_done, 1);
        mbar_init(&bar.drain, 1);
        fence_mbar_init();
    }
    if (warp == 13) {
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

    if (warp == 12) {
        // ------------------------------------------------ producer
        // The whole warp walks the schedule and waits; one elected lane issues the copies.
        if (elect_one()) {
            prefetch_tmap(&tm_q64);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_do64);
            if (MASK) prefetch_tmap(&tm_mask64);
            mbar_arrive_expect_tx(&bar.kv_full, 2 * BK * D * 2);
            for (int bx = 0; bx < D / 64; ++bx) {
                tma_load_4d(smem + Cfg::kKOff + bx * BK * 128, &tm_k, &bar.kv_full, bx * 64, k0, h, b);
                tma_load_4d(smem + Cfg::kVOff + bx * BK * 128, &tm_v, &bar.kv_full, bx * 64, k0, h, b);
            }
        }
        __syncwarp();
        const int hm = p.mask_hb ? h : 0, bm = p.mask_bb ? b : 0;
        const int nq128 = (p.N + 127) / 128;
        bool ok = true;
        int it = 0;
        for (; it < n_it && ok; ++it) {
            const int q0 = (i_begin + it) * BQ;
            const uint32_t ph = (it & 1) ^ 1;
            ok = mbar_wait_warp(&bar.q_empty, ph, wc);
            if (!ok) break;
            if (elect_one()) {
                mbar_arrive_expect_tx(&bar.q_full, BQ * D * 2);
                for (int bx = 0; bx < D / 64; ++bx)
                    tma_load_4d(smem + Cfg::kQOff + bx * BQ * 128, &tm_q64, &bar.q_full, bx * 64, q0, h, b);
            }
            __syncwarp();
            ok = mbar_wait_warp(&bar.do_empty, ph, wc);
            if (!ok) break;
            if (elect_one()) {
                mbar_arrive_expect_tx(&bar.do_full, BQ * D * 2);
                for (int bx = 0; bx < D / 64; ++bx)
                    tma_load_4d(smem + Cfg::kDoOff + bx * BQ * 128, &tm_do64, &bar.do_full, bx * 64, q0, h, b);
            }
            __syncwarp();
            ok = mbar_wait_warp(&bar.st_empty, ph, wc);
            if (MASK) ok = ok && mbar_wait_warp(&bar.m_empty, ph, wc);
            if (!ok) break;
            if (elect_one()) {
                // the tile's 64 rows of the tile-padded statistics: -LSE*log2e, then -D
                const float* src = p.stats + ((long long)bh_i * nq128 + (q0 >> 7)) * 256 + (q0 & 127);
                mbar_arrive_expect_tx(&bar.st_full, 512);
                bulk_load(smem + Cfg::kStatsOff, src, 256, &bar.st_full);
                bulk_load(smem + Cfg::kStatsOff + 256, src + 128, 256, &bar.st_full);
                if (MASK) {
                    mbar_arrive_expect_tx(&bar.m_full, Cfg::kMaskBytes);
                    for (int bx = 0; bx < 2; ++bx)
                        tma_load_4d(smem + Cfg::kMaskOff + bx * BQ * 128, &tm_mask64, &bar.m_full, k0 + bx * 64, q0,
                                    hm, bm);
                }
            }
            __syncwarp();
        }
        // every copy issued lands before the CTA exits
        if (lane == 0 && it > 0) {
            const uint32_t last = (it - 1) & 1;
            drain_wait(&bar.q_full, last, p.timeout_ns);
            drain_wait(&bar.do_full, last, p.timeout_ns);
            drain_wait(&bar.st_full, last, p.timeout_ns);
            if (MASK) drain_wait(&bar.m_full, last, p.timeout_ns);
        }
        if (lane == 0) drain_wait(&bar.kv_full, 0, p.timeout_ns);
    } else if (warp == 13) {
        // ------------------------------------------------ MMA issuer
        // Converged warp; one elected lane (always the same one) issues MMAs and commits.
        const uint32_t sK = smem_u32(smem + Cfg::kKOff), sV = smem_u32(smem + Cfg::kVOff);
        const uint32_t sQ = smem_u32(smem + Cfg::kQOff), sDo = smem_u32(smem + Cfg::kDoOff);
        const uint32_t sDs = smem_u32(smem + Cfg::kDsOff);
        bool ok = mbar_wait_warp(&bar.kv_full, 0, wc);
        tc_fence_after();
        for (int it = 0; it < n_it && ok; ++it) {
            const uint32_t ph = it & 1;
            // S^T and dP^T overwrite the previous tile's P^T / dS^T only after its dK / dV below
            // (MMAs issued by one thread run in order)
            ok = mbar_wait_warp(&bar.q_full, ph, wc);
            if (!ok) break;
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + 0, kdesc(sK, kk, BK), kdesc(sQ, kk, BQ), kIdescS, kk > 0 ? 1u : 0u);
            }
            __syncwarp();
            ok = mbar_wait_warp(&bar.do_full, ph, wc);
            if (!ok) break;
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + 64, kdesc(sV, kk, BK), kdesc(sDo, kk, BQ), kIdescS, kk > 0 ? 1u : 0u);
                mma_commit(&bar.s_full);
            }
            __syncwarp();
            ok = mbar_wait_warp(&bar.ds_ready, ph, wc);
            if (!ok) break;
            tc_fence_after();
            if (elect_one()) {
                // dK first, so that the next Q tile starts loading while dV and dQ run
#pragma unroll
                for (int kk = 0; kk < BQ / 16; ++kk)
                    mma_ts(tmem + 384, tmem + 16 * kk + 8, mndesc(sQ + 2 * hf * BQ * 128, kk, BQ * 128), kIdescKV,
                           (it > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&bar.q_empty);
#pragma unroll
                for (int kk = 0; kk < BQ / 16; ++kk)
                    mma_ts(tmem + 256, tmem + 16 * kk, mndesc(sDo + 2 * hf * BQ * 128, kk, BQ * 128), kIdescKV,
                           (it > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&bar.do_empty);
            }
            __syncwarp();
            if (it > 0) {  // dQ_h^T of the previous tile has been read out of tensor memory
                ok = mbar_wait_warp(&bar.dq_empty, (it - 1) & 1, wc);
                if (!ok) break;
                tc_fence_after();
            }
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    mma_ss(tmem + 128, mndesc(sK + 2 * hf * BK * 128, kk, BK * 128), mndesc(sDs, kk, BQ * 128),
                           kIdescQ, kk > 0 ? 1u : 0u);
                mma_commit(&bar.dq_full);
                mma_commit(&bar.ds_free);
            }
            __syncwarp();
        }
        if (elect_one()) {
            if (ok) mma_commit(&bar.kv_done);
            mma_commit(&bar.drain);
            drain_wait(&bar.drain, 0, p.timeout_ns);
        }
        __syncwarp();
    } else if (warp >= 8 && warp < 12) {
        // ------------------------------------------------ dQ drain (warps 8-11)
        // Thread = head-dim column dd0 + lane of the half (its TMEM lane); the tile's 64 queries are
        // read out, then per 4 queries a quad transpose and one vector reduction of 4 columns of
        // one query row.
        const int dd0 = (warp & 3) * 32;
        const uint32_t tDq = tmem + ((uint32_t)dd0 << 16) + 128;
        const int r = lane & 3;
        float* acc = p.dq_acc + (long long)bh_i * p.N * D + hf * DH + dd0 + (lane & ~3);
        bool ok = true;
        for (int it = 0; it < n_it && ok; ++it) {
            const int q0 = (i_begin + it) * BQ;
            ok = mbar_wait(&bar.dq_full, it & 1, wc);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            uint32_t v[BQ];
            tmem_ld32_at<0>(tDq + 0, v);
            tmem_ld32_at<32>(tDq + 32, v);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(&bar.dq_empty);  // dQ_h^T is in registers: the columns may be reused
#pragma unroll
            for (int gq = 0; gq < BQ / 4; ++gq) {
                float x[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) x[e] = __uint_as_float(v[4 * gq + e]) * p.scale;
                quad_transpose(x, r);  // now columns 4 (lane / 4) .. +3 of query 4 gq + r
                const int row = q0 + 4 * gq + r;
                if (row < p.N) red_add_v4(acc + (long long)row * D, x[0], x[1], x[2], x[3]);
            }
        }
    } else if (warp < 8) {
        // ------------------------------------------------ P^T, dS^T (warps 0-7)
        // Warpgroup g takes queries [32 g, 32 g + 32) of each tile, thread = key row kr.
        const int g = warp >> 2;
        const int kr = (warp & 3) * 32 + lane;
        const int kg = k0 + kr;
        const uint32_t tRow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const float2 c2 = make_float2(p.c, p.c);
        const bool key_ok = kg < p.N;
        const float* nlv = reinterpret_cast<const float*>(smem + Cfg::kStatsOff);  // -LSE*log2e
        const float* ndv = nlv + 64;                                                // -D
        // mask rows of the tile: two 64-key boxes of 64 rows x 128 bytes (128-byte swizzle)
        const uint8_t* mrow = smem + Cfg::kMaskOff + (kr >> 6) * (BQ * 128) + (kr & 7) * 2;
        const int mkc = (kr & 63) >> 3;
        const int c0 = 32 * g;  // this warpgroup's queries within the tile
        bool ok = true;
        for (int it = 0; it < n_it && ok; ++it) {
            const int q0 = (i_begin + it) * BQ;
            const uint32_t ph = it & 1;
            ok = mbar_wait(&bar.s_full, ph, wc);
            // the tile's statistics (and mask) are visible once their copies completed
            ok = ok && mbar_wait(&bar.st_full, ph, wc);
            if (MASK) ok = ok && mbar_wait(&bar.m_full, ph, wc);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const bool diag = p.causal && (q0 < k0 + BK);  // tiles that reach the causal diagonal
            uint32_t sv[32], pv[32];
            tmem_ld32(tRow + c0, sv);
            tmem_ld32(tRow + 64 + c0, pv);
            tmem_wait_ld();
            uint32_t pk[16], dsr[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                const int q = c0 + i;
                const float2 nl = *reinterpret_cast<const float2*>(nlv + q);
                const float2 nd = *reinterpret_cast<const float2*>(ndv + q);
                float2 x = ffma2(make_float2(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])), c2, nl);
                if (MASK) {
                    const float m0 =
                        h16_to_float<F16>(*reinterpret_cast<const uint16_t*>(mrow + q * 128 + ((mkc ^ (q & 7)) << 4)));
                    const float m1 = h16_to_float<F16>(
                        *reinterpret_cast<const uint16_t*>(mrow + (q + 1) * 128 + ((mkc ^ ((q + 1) & 7)) << 4)));
                    x = ffma2(make_float2(m0, m1), make_float2(kLog2e, kLog2e), x);
                }
                if (!key_ok || (diag && q0 + q < kg)) x.x = -INFINITY;
                if (!key_ok || (diag && q0 + q + 1 < kg)) x.y = -INFINITY;
                const float2 pr = make_float2(ex2(x.x), ex2(x.y));
                const float2 ds =
                    fmul2(pr, fadd2(make_float2(__uint_as_float(pv[i]), __uint_as_float(pv[i + 1])), nd));
                pk[i / 2] = pack_h16<F16>(pr.x, pr.y);
                dsr[i / 2] = pack_h16<F16>(ds.x, ds.y);
            }
            mbar_arrive(&bar.st_empty);
            if (MASK) mbar_arrive(&bar.m_empty);
            // 16 queries u = c0 / 16 + hh: P^T at columns [16 u, 16 u + 8), dS^T at [16 u + 8, 16 u + 16)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                tmem_st8(tRow + c0 + 16 * hh, pk + 8 * hh);
                tmem_st8(tRow + c0 + 16 * hh + 8, dsr + 8 * hh);
            }
            if (it > 0) {  // the dQ product of the previous tile has read the dS^T buffer
                ok = mbar_wait(&bar.ds_free, (it - 1) & 1, wc);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
            }
            // dS^T row kr (128 bytes = 64 queries), this warpgroup's 16-byte chunks 4g .. 4g+3
            uint8_t* row = smem + Cfg::kDsOff + kr * 128;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch)
                *reinterpret_cast<uint4*>(row + (((4 * g + ch) ^ (kr & 7)) << 4)) =
                    make_uint4(dsr[4 * ch], dsr[4 * ch + 1], dsr[4 * ch + 2], dsr[4 * ch + 3]);
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bar.ds_ready);
        }
        // epilogue: warpgroup 0 writes dV_h, warpgroup 1 scale * dK_h of this key tile
        if (ok) ok = mbar_wait(&bar.kv_done, 0, wc);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            tc_fence_after();
            __nv_bfloat16* dst_row = g == 0 ? p.dv + b * p.dv_sb + h * p.dv_sh + (long long)kg * p.dv_sn
                                            : p.dk + b * p.dk_sb + h * p.dk_sh + (long long)kg * p.dk_sn;
            dst_row += hf * DH;
            const float mul = g == 0 ? 1.f : p.scale;
#pragma unroll
            for (int cc = 0; cc < DH; cc += 32) {
                uint32_t v[32];
                tmem_ld32(tRow + 256 + g * DH + cc, v);
                tmem_wait_ld();
                if (kg < p.N) {
                    uint4* dst = reinterpret_cast<uint4*>(dst_row + cc);
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
    if (warp == 13) tmem_dealloc(tmem, 512);
}

template <bool MASK, bool F16>
cudaError_t launch_t(const attn_bwd_params& prm, const Bwd256Maps& maps, const BwdWorkspace& ws,
                     const LaunchCommon& lc, cudaStream_t s) {
    using Cfg = B256Cfg<MASK>;
    static_assert(Cfg::kSmemBytes <= 232448, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(bwd256_kernel<MASK, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    const attn_fwd_params& f = prm.fwd;
    B256Params p{};
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
    const unsigned grid = 2u * (unsigned)p.n_ktiles * (unsigned)f.B * (unsigned)f.H;
    e = launch_pdl(bwd256_kernel<MASK, F16>, dim3(grid), dim3(Cfg::kThreads), Cfg::kSmemBytes, s, maps.q64, maps.k,
                   maps.v, maps.do64, maps.mask64, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd256(const attn_bwd_params& p, const Bwd256Maps& maps, const BwdWorkspace& ws,
                          const LaunchCommon& lc, cudaStream_t s) {
    const bool mask = p.fwd.mask != nullptr, f16 = p.fwd.dtype == ATTN_F16;
    if (mask) return f16 ? launch_t<true, true>(p, maps, ws, lc, s) : launch_t<true, false>(p, maps, ws, lc, s);
    return f16 ? launch_t<false, true>(p, maps, ws, lc, s) : launch_t<false, false>(p, maps, ws, lc, s);
}

}  // namespace attn
