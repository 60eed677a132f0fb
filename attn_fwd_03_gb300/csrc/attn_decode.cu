// attn_decode.cu — split-KV decode: a few query rows against a long key/value
// sequence.
//
// A decode step has no N x N matrix to avoid: its cost is one read of the
// keys and values, and with a small batch that read must be spread over the
// sequence to occupy the GPU ("FlashAttention", "What it does not do"). Each
// CTA therefore takes one (b, h) and one contiguous key range (a split), runs
// the online softmax of "Explain FlashAttention and why it is IO-aware" over
// that range for every query row, and writes the row's partial state: the
// running max m, the sum l of 2^(s - m) and the unnormalised o. A second
// kernel merges the splits of a row with the same rescaling that merges
// tiles: M = max m_s, L = sum l_s 2^(m_s - M), O = sum o_s 2^(m_s - M) / L.
//
// The work is bound by HBM bandwidth (every key and value is read once, at
// about nq FLOP per byte), so the split kernel runs on the CUDA cores:
// 64-key blocks of K and V are staged in shared memory with cp.async,
// 256 threads compute the nq x 64 scores, one warp per query row
// updates (m, l) and the probabilities, and the threads accumulate o in
// registers, each over its own subset of the keys, reduced once at the end.
// Three blocks are in flight per CTA and, up to 8 query rows, two CTAs share
// an SM, so about 190 KB of loads per SM cover the memory latency at full
// bandwidth.
// Scores are in the log2 domain: s = c * (q . k) with c = scale * log2(e).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int KB = 64;        // keys per block iteration
constexpr int kStages = 3;    // K/V blocks in flight per CTA (two CTAs per SM)
constexpr int kThreads = 256;
constexpr unsigned kFull = 0xffffffffu;

struct DecodeArgs {
    const uint8_t *q, *k, *v;
    uint8_t* o;
    float* lse;
    long long q_sb, q_sh, q_sn, k_sb, k_sh, k_sn, v_sb, v_sh, v_sn, o_sb, o_sh, o_sn;  // elements
    int B, H, nq, nk, causal;
    int splits, chunk;  // key ranges per (b, h) and keys per range (a multiple of KB)
    float c;            // scale * log2(e)
    float* part;        // [B*H][splits][nq][D + 4]: m, l, 2 unused, o[D]
};

template <int D>
constexpr int rec_floats() {
    return D + 4;
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc, bool valid) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    const int src_bytes = valid ? 16 : 0;  // 0: the 16 bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(gsrc), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// NQP: query rows rounded up to a power of two (1 .. 16); F16: IEEE half storage, else bf16.
template <int D, int NQP, bool F16>
__global__ void __launch_bounds__(kThreads, 2) decode_split_kernel(DecodeArgs a) {
    constexpr int ROW = D * 2 + 16;  // bytes per staged K/V row (padded against bank conflicts)
    constexpr int CH = D / 8;        // 16-byte chunks per row
    // score phase: NQP x KB dot products, PARTS threads per product or DPT products per thread
    constexpr int DOTS = NQP * KB;
    constexpr int PARTS = DOTS >= kThreads ? 1 : kThreads / DOTS;
    constexpr int DPT = DOTS >= kThreads ? DOTS / kThreads : 1;
    constexpr int PART_CH = CH / PARTS;  // chunks per part
    // PV phase: NQP x CH (row, chunk) pairs, KL threads per pair splitting the keys
    constexpr int PAIRS = NQP * CH;
    constexpr int KL = kThreads / PAIRS;
    static_assert(PAIRS * KL == kThreads && KL >= 1 && KL <= 32, "PV thread mapping");
    static_assert(PART_CH >= 1 && PARTS * PART_CH == CH, "score thread mapping");

    extern __shared__ __align__(16) uint8_t sm[];
    float* q_s = reinterpret_cast<float*>(sm);                     // [NQP][D], scaled by c
    uint8_t* kv_s = sm + NQP * D * 4;                              // [kStages buffers][K, V][KB][ROW]
    float* p_s = reinterpret_cast<float*>(kv_s + kStages * 2 * KB * ROW);  // [NQP][KB] scores, then probabilities
    float* alpha_s = p_s + NQP * KB;                                // [NQP]

    const int split = blockIdx.x, bh = blockIdx.y;
    const int b = bh / a.H, h = bh % a.H;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int k_begin = split * a.chunk;
    const int k_end = min(a.nk, k_begin + a.chunk);
    const int nblk = (k_end - k_begin + KB - 1) / KB;
    const uint8_t* kbase = a.k + (b * a.k_sb + h * a.k_sh) * 2;
    const uint8_t* vbase = a.v + (b * a.v_sb + h * a.v_sh) * 2;

    // queries (fp32, scaled), rows beyond nq zero
    for (int idx = t; idx < NQP * D; idx += kThreads) {
        const int i = idx / D, e = idx % D;
        float x = 0.f;
        if (i < a.nq) {
            const uint16_t raw =
                *reinterpret_cast<const uint16_t*>(a.q + ((b * a.q_sb + h * a.q_sh + (long long)i * a.q_sn) + e) * 2);
            x = ptx::h16_to_float<F16>(raw) * a.c;
        }
        q_s[idx] = x;
    }

    auto stage = [&](int blk, int buf) {
        const int key0 = k_begin + blk * KB;
        for (int idx = t; idx < 2 * KB * CH; idx += kThreads) {
            const int which = idx / (KB * CH);  // 0 = K, 1 = V
            const int r = (idx / CH) % KB, ch = idx % CH;
            const int key = key0 + r;
            const bool valid = key < k_end;
            const uint8_t* src = which == 0 ? kbase + (long long)(valid ? key : 0) * a.k_sn * 2
                                            : vbase + (long long)(valid ? key : 0) * a.v_sn * 2;
            cp_async16(kv_s + ((buf * 2 + which) * KB + r) * ROW + ch * 16, src + ch * 16, valid);
        }
        cp_async_commit();
    };

    // per query row owned by this warp (rows warp and warp + 8): running max and sum
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    // PV accumulator of this thread: row pi, chunk pc, keys kl, kl + KL, ...
    const int kl = t % KL, pair = t / KL, pi = pair / CH, pc = pair % CH;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};

    // one commit group per block (empty past the end), so "all but the newest kStages - 1
    // groups complete" always means "block blk has landed"
#pragma unroll
    for (int st = 0; st < kStages - 1; ++st) {
        if (st < nblk) stage(st, st);
        else cp_async_commit();
    }
    for (int blk = 0; blk < nblk; ++blk) {
        const int buf = blk % kStages;
        if (blk + kStages - 1 < nblk) stage(blk + kStages - 1, (blk + kStages - 1) % kStages);
        else cp_async_commit();
        cp_async_wait<kStages - 1>();
        __syncthreads();  // block blk staged; previous block's probabilities consumed
        const uint8_t* k_s = kv_s + (buf * 2 + 0) * KB * ROW;
        const uint8_t* v_s = kv_s + (buf * 2 + 1) * KB * ROW;
        const int key0 = k_begin + blk * KB;

        // ---- scores s = c * q . k, masked to -inf outside the range and above the causal limit
#pragma unroll
        for (int r = 0; r < DPT; ++r) {
            const int dot = t / PARTS + r * (kThreads / PARTS);
            const int i = dot / KB, j = dot % KB;
            const int part = t % PARTS;
            const float* qrow = q_s + i * D + part * PART_CH * 8;
            const uint8_t* krow = k_s + j * ROW + part * PART_CH * 16;
            float s = 0.f;
#pragma unroll
            for (int ch = 0; ch < PART_CH; ++ch) {
                const uint4 kv = *reinterpret_cast<const uint4*>(krow + ch * 16);
                const uint32_t w[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 kf = ptx::unpack_h16<F16>(w[e]);
                    s = fmaf(qrow[ch * 8 + 2 * e], kf.x, s);
                    s = fmaf(qrow[ch * 8 + 2 * e + 1], kf.y, s);
                }
            }
#pragma unroll
            for (int o = PARTS / 2; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
            if (part == 0) {
                const int key = key0 + j;
                const bool ok = key < k_end && i < a.nq && (!a.causal || key <= a.nk - a.nq + i);
                p_s[i * KB + j] = ok ? s : -INFINITY;
            }
        }
        __syncthreads();

        // ---- online softmax per row: warp w owns rows w and w + 8
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int i = warp + 8 * rr;
            if (i >= NQP) break;
            const float s0 = p_s[i * KB + lane], s1 = p_s[i * KB + lane + 32];
            float mx = fmaxf(s0, s1);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
            const float m_new = fmaxf(m_run[rr], mx);
            float p0 = 0.f, p1 = 0.f, alpha = 1.f;
            if (m_new != -INFINITY) {
                p0 = ptx::ex2(s0 - m_new);
                p1 = ptx::ex2(s1 - m_new);
                alpha = ptx::ex2(m_run[rr] - m_new);  // 0 when the row had no key yet
            }
            float sum = p0 + p1;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
            l_run[rr] = l_run[rr] * alpha + sum;
            m_run[rr] = m_new;
            p_s[i * KB + lane] = p0;
            p_s[i * KB + lane + 32] = p1;
            if (lane == 0) alpha_s[i] = alpha;
        }
        __syncthreads();

        // ---- o = alpha o + sum_j p_j v_j over this thread's keys kl, kl + KL, ...
        {
            const float al = alpha_s[pi];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] *= al;
#pragma unroll 4
            for (int j = kl; j < KB; j += KL) {
                const float pj = p_s[pi * KB + j];
                const uint4 vv = *reinterpret_cast<const uint4*>(v_s + j * ROW + pc * 16);
                const uint32_t w[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 vf = ptx::unpack_h16<F16>(w[e]);
                    acc[2 * e] = fmaf(pj, vf.x, acc[2 * e]);
                    acc[2 * e + 1] = fmaf(pj, vf.y, acc[2 * e + 1]);
                }
            }
        }
        __syncthreads();  // buffer buf and the probabilities may be overwritten
    }

    // ---- partial state of each row: (m, l) from the owner warp, o reduced over the key lanes
    float* rec0 = a.part + ((long long)bh * a.splits + split) * a.nq * rec_floats<D>();
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int i = warp + 8 * rr;
        if (i < a.nq && lane == 0) {
            rec0[i * rec_floats<D>() + 0] = m_run[rr];
            rec0[i * rec_floats<D>() + 1] = l_run[rr];
        }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e)
#pragma unroll
        for (int o = KL / 2; o > 0; o >>= 1) acc[e] += __shfl_xor_sync(kFull, acc[e], o);
    if (kl == 0 && pi < a.nq) {
        float4* dst = reinterpret_cast<float4*>(rec0 + pi * rec_floats<D>() + 4 + pc * 8);
        dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
}

// Up to four query rows: each warp streams its own keys straight into registers
// (no shared memory, no block-wide barriers). A key row is split over LPK lanes
// (16 bytes each), so one 16-byte load per lane covers KPI keys; every lane
// group (the LPK lanes of one key slot) keeps its own running (m, l, o) for
// the keys it sees, rescaling once per group of U keys, and the groups' states
// are merged through shared memory at the end. Loads of the next group are
// issued before the current one is used.
template <int D, int NQP, bool F16>
__global__ void __launch_bounds__(kThreads) decode_stream_kernel(DecodeArgs a) {
    constexpr int LPK = D / 8;        // lanes per key row
    constexpr int KPI = 32 / LPK;     // keys per warp-wide load
    constexpr int U = 4;              // loads per lane per group
    constexpr int G = KPI * U;        // keys per warp per group
    constexpr int NW = kThreads / 32;
    constexpr int SLOTS = NW * KPI;   // lane groups per CTA
    __shared__ float st_m[NQP][SLOTS], st_l[NQP][SLOTS];
    __shared__ __align__(16) float st_o[NQP][SLOTS][D];

    const int split = blockIdx.x, bh = blockIdx.y;
    const int b = bh / a.H, h = bh % a.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot_in_warp = lane / LPK, cl = lane % LPK;
    const int k_begin = split * a.chunk;
    const int k_end = min(a.nk, k_begin + a.chunk);
    const uint8_t* kbase = a.k + (b * a.k_sb + h * a.k_sh) * 2 + cl * 16;
    const uint8_t* vbase = a.v + (b * a.v_sb + h * a.v_sh) * 2 + cl * 16;

    float q[NQP][8];
#pragma unroll
    for (int i = 0; i < NQP; ++i) {
        uint4 raw = make_uint4(0u, 0u, 0u, 0u);
        if (i < a.nq)
            raw = *reinterpret_cast<const uint4*>(a.q + (b * a.q_sb + h * a.q_sh + (long long)i * a.q_sn) * 2 + cl * 16);
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = ptx::unpack_h16<F16>(w[e]);
            q[i][2 * e] = f.x * a.c;
            q[i][2 * e + 1] = f.y * a.c;
        }
    }
    float m[NQP], l[NQP], o[NQP][8];
#pragma unroll
    for (int i = 0; i < NQP; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) o[i][e] = 0.f;
    }

    // this warp's groups: keys k_begin + (g * NW + warp) * G + u * KPI + slot_in_warp
    const int ngroups = (k_end - k_begin + G - 1) / G;
    auto key_of = [&](int g, int u) { return k_begin + (g * NW + warp) * G + u * KPI + slot_in_warp; };
    auto load = [&](int g, uint4 (&kr)[U], uint4 (&vr)[U]) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            int key = key_of(g, u);
            key = key < k_end ? key : k_end - 1;  // stay in bounds; masked below
            kr[u] = __ldg(reinterpret_cast<const uint4*>(kbase + (long long)key * a.k_sn * 2));
            vr[u] = __ldg(reinterpret_cast<const uint4*>(vbase + (long long)key * a.v_sn * 2));
        }
    };
    uint4 kc[U], vc[U], kn[U], vn[U];
    int g = 0;
    if (warp < ngroups) load(0, kc, vc);
    for (; g * NW + warp < ngroups; ++g) {
        const bool more = (g + 1) * NW + warp < ngroups;
        if (more) load(g + 1, kn, vn);
        float s[NQP][U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t w[4] = {kc[u].x, kc[u].y, kc[u].z, kc[u].w};
            float2 kf[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) kf[e] = ptx::unpack_h16<F16>(w[e]);
            const int key = key_of(g, u);
#pragma unroll
            for (int i = 0; i < NQP; ++i) {
                float x = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    x = fmaf(q[i][2 * e], kf[e].x, x);
                    x = fmaf(q[i][2 * e + 1], kf[e].y, x);
                }
#pragma unroll
                for (int sh = LPK / 2; sh > 0; sh >>= 1) x += __shfl_xor_sync(kFull, x, sh);
                const bool ok = key < k_end && i < a.nq && (!a.causal || key <= a.nk - a.nq + i);
                s[i][u] = ok ? x : -INFINITY;
            }
        }
#pragma unroll
        for (int i = 0; i < NQP; ++i) {
            float mx = s[i][0];
#pragma unroll
            for (int u = 1; u < U; ++u) mx = fmaxf(mx, s[i][u]);
            const float m_new = fmaxf(m[i], mx);
            if (m_new == -INFINITY) continue;  // nothing seen yet by this lane group
            const float alpha = ptx::ex2(m[i] - m_new);  // 0 when the group had no key yet
            float p[U];
            float ps = 0.f;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                p[u] = ptx::ex2(s[i][u] - m_new);
                ps += p[u];
            }
            l[i] = l[i] * alpha + ps;
            m[i] = m_new;
#pragma unroll
            for (int e = 0; e < 8; ++e) o[i][e] *= alpha;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint32_t w[4] = {vc[u].x, vc[u].y, vc[u].z, vc[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 vf = ptx::unpack_h16<F16>(w[e]);
                    o[i][2 * e] = fmaf(p[u], vf.x, o[i][2 * e]);
                    o[i][2 * e + 1] = fmaf(p[u], vf.y, o[i][2 * e + 1]);
                }
            }
        }
        if (more) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                kc[u] = kn[u];
                vc[u] = vn[u];
            }
        }
    }

    // merge the CTA's lane-group states into the split's partial record
    const int slot = warp * KPI + slot_in_warp;
#pragma unroll
    for (int i = 0; i < NQP; ++i) {
        if (cl == 0) {
            st_m[i][slot] = m[i];
            st_l[i][slot] = l[i];
        }
        *reinterpret_cast<float4*>(&st_o[i][slot][cl * 8]) = make_float4(o[i][0], o[i][1], o[i][2], o[i][3]);
        *reinterpret_cast<float4*>(&st_o[i][slot][cl * 8 + 4]) = make_float4(o[i][4], o[i][5], o[i][6], o[i][7]);
    }
    __syncthreads();
    float* rec0 = a.part + ((long long)bh * a.splits + split) * a.nq * rec_floats<D>();
    for (int idx = threadIdx.x; idx < NQP * D; idx += kThreads) {
        const int i = idx / D, e = idx % D;
        if (i >= a.nq) continue;
        float M = -INFINITY;
        for (int sl = 0; sl < SLOTS; ++sl) M = fmaxf(M, st_m[i][sl]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
            for (int sl = 0; sl < SLOTS; ++sl) {
                const float w = ptx::ex2(st_m[i][sl] - M);  // 0 for a group that saw no key
                L = fmaf(w, st_l[i][sl], L);
                O = fmaf(w, st_o[i][sl][e], O);
            }
        }
        rec0[i * rec_floats<D>() + 4 + e] = O;
        if (e == 0) {
            rec0[i * rec_floats<D>() + 0] = M;
            rec0[i * rec_floats<D>() + 1] = L;
        }
    }
}

template <int D, int NQP, bool F16>
cudaError_t launch_stream(const DecodeArgs& a, cudaStream_t s) {
    decode_stream_kernel<D, NQP, F16><<<dim3(a.splits, a.B * a.H), kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

// One warp per (b, h, row): merge the row's split states into O and LSE.
template <int D, bool F16>
__global__ void __launch_bounds__(256) decode_combine_kernel(DecodeArgs a) {
    constexpr int PER = D / 32;  // output columns per lane
    const int warp_g = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    const int rows = a.B * a.H * a.nq;
    if (warp_g >= rows) return;
    const int i = warp_g % a.nq, bh = warp_g / a.nq;
    const int b = bh / a.H, h = bh % a.H;
    const float* base = a.part + (long long)bh * a.splits * a.nq * rec_floats<D>() + i * rec_floats<D>();
    const long long sstride = (long long)a.nq * rec_floats<D>();
    float M = -INFINITY;
    for (int s = lane; s < a.splits; s += 32) M = fmaxf(M, base[s * sstride]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
    float L = 0.f, out[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) out[e] = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < a.splits; ++s) {
            const float* r = base + s * sstride;
            const float w = ptx::ex2(r[0] - M);  // 0 for a split that saw no key of this row
            L += w * r[1];
#pragma unroll
            for (int e = 0; e < PER; ++e) out[e] = fmaf(w, r[4 + lane * PER + e], out[e]);
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint16_t* orow = reinterpret_cast<uint16_t*>(a.o) + (b * a.o_sb + h * a.o_sh + (long long)i * a.o_sn);
    if constexpr (PER == 2) {
        *reinterpret_cast<uint32_t*>(orow + lane * 2) = ptx::pack_h16<F16>(out[0] * inv, out[1] * inv);
    } else {
        *reinterpret_cast<uint2*>(orow + lane * 4) =
            make_uint2(ptx::pack_h16<F16>(out[0] * inv, out[1] * inv), ptx::pack_h16<F16>(out[2] * inv, out[3] * inv));
    }
    if (lane == 0) a.lse[(long long)bh * a.nq + i] = L > 0.f ? (M + __log2f(L)) * kLn2 : -INFINITY;
}

template <int D, int NQP, bool F16>
cudaError_t launch_split(const DecodeArgs& a, cudaStream_t s) {
    constexpr int ROW = D * 2 + 16;
    constexpr size_t smem = NQP * D * 4 + kStages * 2 * KB * ROW + NQP * KB * 4 + NQP * 4;
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D, NQP, F16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    decode_split_kernel<D, NQP, F16><<<dim3(a.splits, a.B * a.H), kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

template <int D, bool F16>
cudaError_t launch_d(const DecodeArgs& a, cudaStream_t s) {
    cudaError_t e;
    if (a.nq <= 1)
        e = launch_stream<D, 1, F16>(a, s);
    else if (a.nq <= 2)
        e = launch_stream<D, 2, F16>(a, s);
    else if (a.nq <= 4)
        e = launch_stream<D, 4, F16>(a, s);
    else if (a.nq <= 8)
        e = launch_split<D, 8, F16>(a, s);
    else
        e = launch_split<D, 16, F16>(a, s);
    if (e != cudaSuccess) return e;
    const int rows = a.B * a.H * a.nq;
    decode_combine_kernel<D, F16><<<(rows + 7) / 8, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

DecodeSplit decode_split_plan(const attn_decode_params& p, int num_sms) {
    const int max_splits = (p.nk + KB - 1) / KB;
    int splits = p.num_splits;
    if (splits <= 0) {
        // at least four waves of two CTAs per SM, so the last wave's shortfall stays small;
        // each range at least 256 keys
        const long long bh = (long long)p.B * p.H;
        const long long want = (8LL * num_sms + bh - 1) / (bh > 0 ? bh : 1);
        const int by_len = (p.nk + 255) / 256;
        splits = (int)(want < by_len ? want : by_len);
    }
    if (splits < 1) splits = 1;
    if (splits > max_splits) splits = max_splits;
    int chunk = (p.nk + splits - 1) / splits;
    chunk = (chunk + KB - 1) / KB * KB;
    splits = (p.nk + chunk - 1) / chunk;  // no empty range
    DecodeSplit plan;
    plan.splits = splits;
    plan.chunk = chunk;
    plan.workspace_bytes = (size_t)p.B * p.H * splits * p.nq * (p.d + 4) * sizeof(float);
    return plan;
}

cudaError_t launch_decode(const attn_decode_params& p, const DecodeSplit& plan, cudaStream_t s) {
    DecodeArgs a{};
    a.q = static_cast<const uint8_t*>(p.q);
    a.k = static_cast<const uint8_t*>(p.k);
    a.v = static_cast<const uint8_t*>(p.v);
    a.o = static_cast<uint8_t*>(p.o);
    a.lse = p.lse;
    a.q_sb = p.q_stride[0];
    a.q_sh = p.q_stride[1];
    a.q_sn = p.q_stride[2];
    a.k_sb = p.k_stride[0];
    a.k_sh = p.k_stride[1];
    a.k_sn = p.k_stride[2];
    a.v_sb = p.v_stride[0];
    a.v_sh = p.v_stride[1];
    a.v_sn = p.v_stride[2];
    a.o_sb = p.o_stride[0];
    a.o_sh = p.o_stride[1];
    a.o_sn = p.o_stride[2];
    a.B = p.B;
    a.H = p.H;
    a.nq = p.nq;
    a.nk = p.nk;
    a.causal = p.causal;
    a.splits = plan.splits;
    a.chunk = plan.chunk;
    a.c = p.scale * kLog2e;
    a.part = static_cast<float*>(p.workspace);
    const bool f16 = p.dtype == ATTN_F16;
    if (p.d == 64) return f16 ? launch_d<64, true>(a, s) : launch_d<64, false>(a, s);
    return f16 ? launch_d<128, true>(a, s) : launch_d<128, false>(a, s);
}

}  // namespace attn
