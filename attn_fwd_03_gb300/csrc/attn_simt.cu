// attn_simt.cu — CUDA-core (SIMT) attention kernels.
//
//  * fwd_simt_kernel<float, D>: the fp32-input forward. Tensor-core fp32
//    (tf32) would miss a 1e-4 tolerance, so the fp32 path runs the online
//    softmax on the FP32 pipes ("Explain FlashAttention and why it is
//    IO-aware", "Keep only the state needed for the final weighted average").
//  * bwd_prepass_kernel: D_i = <dO_i, O_i> and -LSE_i * log2(e) per row into a
//    tile-padded statistics block, and zeroes the fp32 dQ accumulator in the
//    same pass (bandwidth bound: one read of O and dO).
//  * bwd_dq_finalize_kernel: fp32 dQ accumulator -> output dtype.
//
// Layout conventions match include/attn.h: [B, H, N, d] with element strides
// for (b, h, n) and a contiguous last dimension; LSE and D are [B, H, N] fp32.
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr unsigned kFull = 0xffffffffu;

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) {
    return x;
}
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) {
    return x;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

struct Tensor4 {
    const void* ptr;
    long long sb, sh, sn;  // element strides
};

struct SimtArgs {
    Tensor4 q, k, v, o, mask, dout, dq, dk, dv;
    float* lse;
    int B, H, N;
    int causal;
    int has_mask;
    float c;      // scale * log2(e): scores in the log2 domain
    float scale;  // plain softmax scale
};

template <typename T>
__device__ __forceinline__ const T* row_ptr(const Tensor4& t, int b, int h, long long n) {
    return static_cast<const T*>(t.ptr) + b * t.sb + h * t.sh + n * t.sn;
}

// Log2-domain score of (query gi, key gj) with scale, mask, causal and tail.
template <typename T>
__device__ __forceinline__ float finish_score(float dot, const SimtArgs& a, int b, int h, int gi, int gj) {
    if (gj >= a.N || gi >= a.N || (a.causal && gj > gi)) return -INFINITY;
    float s = dot * a.c;
    if (a.has_mask) s += to_f<T>(row_ptr<T>(a.mask, b, h, gi)[gj]) * kLog2e;
    return s;
}

// ------------------------------------------------------------------ forward
// Block: 4 warps, 8 query rows (2 per warp), so even a single head of a few
// hundred rows spreads over dozens of SMs. Key tiles of 32 keys staged in
// shared memory; lane j scores key j of the tile for one row at a time, the
// row's (m, l) live in every lane, lane owns output dims lane + 32 t.
constexpr int kSimtRows = 8;
template <typename T, int D>
__global__ void __launch_bounds__(128) fwd_simt_kernel(SimtArgs a) {
    constexpr int BR = kSimtRows, BC = 32, RPW = BR / 4, DT = D / 32;
    extern __shared__ float sm[];
    float(*Qs)[D] = reinterpret_cast<float(*)[D]>(sm);
    float(*Ks)[D + 1] = reinterpret_cast<float(*)[D + 1]>(sm + BR * D);
    float(*Vs)[D] = reinterpret_cast<float(*)[D]>(sm + BR * D + BC * (D + 1));
    const int b = blockIdx.z, h = blockIdx.y, r0 = blockIdx.x * BR;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = a.N;

    for (int idx = threadIdx.x; idx < BR * D; idx += blockDim.x) {
        const int r = idx / D, c = idx % D;
        Qs[r][c] = (r0 + r < N) ? to_f<T>(row_ptr<T>(a.q, b, h, r0 + r)[c]) : 0.f;
    }
    float m[RPW], l[RPW], acc[RPW][DT];
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int t = 0; t < DT; ++t) acc[i][t] = 0.f;
    }
    const int kv_end = a.causal ? min(N, r0 + BR) : N;
    for (int j0 = 0; j0 < kv_end; j0 += BC) {
        __syncthreads();
        for (int idx = threadIdx.x; idx < BC * D; idx += blockDim.x) {
            const int r = idx / D, c = idx % D;
            const bool in = j0 + r < N;
            Ks[r][c] = in ? to_f<T>(row_ptr<T>(a.k, b, h, j0 + r)[c]) : 0.f;
            Vs[r][c] = in ? to_f<T>(row_ptr<T>(a.v, b, h, j0 + r)[c]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
            const int r = warp * RPW + rr, gi = r0 + r;
            float dot = 0.f;
#pragma unroll 8
            for (int t = 0; t < D; ++t) dot = fmaf(Qs[r][t], Ks[lane][t], dot);
            const float s = finish_score<T>(dot, a, b, h, gi, j0 + lane);
            const float m_new = fmaxf(m[rr], warp_max(s));
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float p = ptx::ex2(s - m_use);
            const float alpha = ptx::ex2(m[rr] - m_use);
            l[rr] = l[rr] * alpha + warp_sum(p);
#pragma unroll
            for (int t = 0; t < DT; ++t) acc[rr][t] *= alpha;
#pragma unroll 4
            for (int j = 0; j < BC; ++j) {
                const float pj = __shfl_sync(kFull, p, j);
#pragma unroll
                for (int t = 0; t < DT; ++t) acc[rr][t] = fmaf(pj, Vs[j][lane + 32 * t], acc[rr][t]);
            }
            m[rr] = m_new;
        }
    }
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
        const int gi = r0 + warp * RPW + rr;
        if (gi >= N) continue;
        const float inv = l[rr] > 0.f ? 1.f / l[rr] : 0.f;
        T* orow = const_cast<T*>(row_ptr<T>(a.o, b, h, gi));
#pragma unroll
        for (int t = 0; t < DT; ++t) orow[lane + 32 * t] = from_f<T>(acc[rr][t] * inv);
        if (lane == 0)
            a.lse[((long long)b * a.H + h) * N + gi] = l[rr] > 0.f ? (m[rr] + log2f(l[rr])) * kLn2 : -INFINITY;
    }
}

// ------------------------------------------------------------ bwd pre-pass
// G = D/8 threads per row, 8 elements (16 B) each. Rows run over the padded
// range [B*H][ceil(N/128)*128]. For a real row it writes -D = -<dO, O> and
// -LSE * log2(e) into the stats block and zeroes the row of the fp32 dQ
// accumulator; a padding row gets (-inf, 0) so the backward kernel can copy
// whole 128-row tiles of statistics without bounds checks.
// 16-byte accesses check their addresses; a misaligned one is recorded in the
// device error word and skipped rather than executed.
constexpr int kErrMisaligned = -7;
__device__ __forceinline__ bool aligned16(const void* p, int* err) {
    if ((reinterpret_cast<uintptr_t>(p) & 15u) == 0) return true;
    atomicExch(err, kErrMisaligned);
    return false;
}

// Both kernels below are bound by HBM bandwidth. A thread covers 8 elements of a
// row (16-byte accesses) for kRowsPerThread rows spaced one grid apart, so each
// thread keeps several independent loads in flight; row decomposition uses
// 32-bit arithmetic when the row count allows it (IDX = unsigned), else 64-bit.
constexpr int kRowsPerThread = 4;

template <int D, typename IDX, bool F16>
__global__ void __launch_bounds__(256) bwd_prepass_kernel(SimtArgs a, float* stats, float* dq_acc, int* err) {
    ptx::grid_dep_wait();    // O and LSE may come from the forward just before
    ptx::grid_dep_launch();  // the main kernel may start its prologue
    constexpr int G = D / 8;            // threads per row
    constexpr int RPB = 256 / G;        // rows per block and step
    const IDX n_pad = (IDX)((a.N + 127) / 128 * 128);
    const IDX rows = (IDX)a.B * (IDX)a.H * n_pad;
    const IDX step = (IDX)gridDim.x * RPB;
    const int part = threadIdx.x % G;
    IDX prow = (IDX)blockIdx.x * RPB + threadIdx.x / G;
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k, prow += step) {
        const IDX n = prow % n_pad;
        const IDX bh = prow / n_pad;
        float sum = 0.f;
        bool ok = prow < rows && n < (IDX)a.N;
        const __nv_bfloat16 *op = nullptr, *gp = nullptr;
        float* zp = nullptr;
        if (ok) {
            const int h = (int)(bh % (IDX)a.H);
            const int b = (int)(bh / (IDX)a.H);
            op = row_ptr<__nv_bfloat16>(a.o, b, h, (long long)n) + part * 8;
            gp = row_ptr<__nv_bfloat16>(a.dout, b, h, (long long)n) + part * 8;
            zp = dq_acc + ((long long)bh * a.N + (long long)n) * D + part * 8;
            ok = aligned16(op, err) && aligned16(gp, err) && aligned16(zp, err);
        }
        if (ok) {
            const uint4 ov = *reinterpret_cast<const uint4*>(op);
            const uint4 gv = *reinterpret_cast<const uint4*>(gp);
            const uint32_t o2[4] = {ov.x, ov.y, ov.z, ov.w}, g2[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 of = ptx::unpack_h16<F16>(o2[i]);
                const float2 gf = ptx::unpack_h16<F16>(g2[i]);
                sum = fmaf(of.x, gf.x, sum);
                sum = fmaf(of.y, gf.y, sum);
            }
            float4* z = reinterpret_cast<float4*>(zp);
            z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int o = G / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o, G);
        if (prow < rows && part == 0) {
            float nl = -INFINITY, dd = 0.f;
            if (n < (IDX)a.N) {
                const float l = a.lse[(long long)bh * a.N + (long long)n];
                nl = (l == -INFINITY) ? -INFINITY : -l * kLog2e;
                dd = -sum;
            }
            float* tile = stats + ((long long)bh * (n_pad / 128) + n / 128) * 256;
            tile[n % 128] = nl;
            tile[128 + n % 128] = dd;
        }
    }
}

// ------------------------------------------------------------ dQ finalize
template <int D, typename IDX, bool F16>
__global__ void __launch_bounds__(256) bwd_dq_finalize_kernel(SimtArgs a, const float* dq_acc, int* err) {
    ptx::grid_dep_wait();  // every reduction into the accumulator has landed
    constexpr int G = D / 8;
    constexpr int RPB = 256 / G;
    const IDX rows = (IDX)a.B * (IDX)a.H * (IDX)a.N;
    const IDX step = (IDX)gridDim.x * RPB;
    const int part = threadIdx.x % G;
    IDX row = (IDX)blockIdx.x * RPB + threadIdx.x / G;
    float4 x[kRowsPerThread], y[kRowsPerThread];
    uint4* dst[kRowsPerThread];
    // all loads first, then all stores
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k, row += step) {
        dst[k] = nullptr;
        if (row >= rows) continue;
        const IDX n = row % (IDX)a.N;
        const IDX bhr = row / (IDX)a.N;
        const int h = (int)(bhr % (IDX)a.H);
        const int b = (int)(bhr / (IDX)a.H);
        const float4* src = reinterpret_cast<const float4*>(dq_acc + (long long)row * D + part * 8);
        uint4* d = reinterpret_cast<uint4*>(const_cast<__nv_bfloat16*>(row_ptr<__nv_bfloat16>(a.dq, b, h, (long long)n))) +
                   part;
        if (!aligned16(src, err) || !aligned16(d, err)) continue;
        x[k] = src[0];
        y[k] = src[1];
        dst[k] = d;
    }
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) {
        if (dst[k] == nullptr) continue;
        uint4 out;
        out.x = ptx::pack_h16<F16>(x[k].x, x[k].y);
        out.y = ptx::pack_h16<F16>(x[k].z, x[k].w);
        out.z = ptx::pack_h16<F16>(y[k].x, y[k].y);
        out.w = ptx::pack_h16<F16>(y[k].z, y[k].w);
        *dst[k] = out;
    }
}

Tensor4 tensor4(const void* p, const int64_t* s) { return Tensor4{p, (long long)s[0], (long long)s[1], (long long)s[2]}; }

SimtArgs make_args(const attn_fwd_params& p) {
    SimtArgs a{};
    a.q = tensor4(p.q, p.q_stride);
    a.k = tensor4(p.k, p.k_stride);
    a.v = tensor4(p.v, p.v_stride);
    a.o = tensor4(p.o, p.o_stride);
    a.mask = tensor4(p.mask, p.mask_stride);
    a.lse = p.lse;
    a.B = p.B;
    a.H = p.H;
    a.N = p.N;
    a.causal = p.causal;
    a.has_mask = p.mask != nullptr;
    a.scale = p.scale;
    a.c = p.scale * kLog2e;
    return a;
}

SimtArgs make_bwd_args(const attn_bwd_params& p, const BwdWorkspace& ws) {
    SimtArgs a = make_args(p.fwd);
    a.dout = tensor4(p.dout, p.do_stride);
    a.dq = tensor4(p.dq, p.dq_stride);
    a.dk = tensor4(p.dk, p.dk_stride);
    a.dv = tensor4(p.dv, p.dv_stride);

    return a;
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename T, int D>
cudaError_t fwd_simt_launch(const SimtArgs& a, cudaStream_t s) {
    const size_t smem = sizeof(float) * (kSimtRows * D + 32 * (D + 1) + 32 * D);
    cudaError_t e = set_smem(fwd_simt_kernel<T, D>, smem);
    if (e != cudaSuccess) return e;
    dim3 grid((a.N + kSimtRows - 1) / kSimtRows, a.H, a.B);
    fwd_simt_kernel<T, D><<<grid, 128, smem, s>>>(a);
    e = cudaGetLastError();
    if (e == cudaSuccess) note_launch(reinterpret_cast<const void*>(fwd_simt_kernel<T, D>));
    return e;
}

}  // namespace

cudaError_t launch_fwd_simt(const attn_fwd_params& p, cudaStream_t s) {
    const SimtArgs a = make_args(p);
    return p.d == 64 ? fwd_simt_launch<float, 64>(a, s) : fwd_simt_launch<float, 128>(a, s);
}

namespace {
// blocks for `rows` rows, kRowsPerThread rows per thread; 32-bit indexing if every
// row index (plus one grid step of slack) fits
struct RowGrid {
    unsigned blocks;
    bool idx32;
};
RowGrid row_grid(long long rows, int d) {
    const long long rpb = 256 / (d / 8);
    const long long per_block = rpb * kRowsPerThread;
    const long long blocks = (rows + per_block - 1) / per_block;
    return RowGrid{(unsigned)blocks, rows + blocks * rpb < (1ll << 31)};
}
template <int D, bool F16>
cudaError_t prepass_t(const RowGrid& g, const SimtArgs& a, const BwdWorkspace& ws, int* err, cudaStream_t s) {
    if (g.idx32)
        return launch_pdl(bwd_prepass_kernel<D, unsigned, F16>, dim3(g.blocks), dim3(256), 0, s, a, ws.stats,
                          ws.dq_acc, err);
    return launch_pdl(bwd_prepass_kernel<D, unsigned long long, F16>, dim3(g.blocks), dim3(256), 0, s, a, ws.stats,
                      ws.dq_acc, err);
}
template <int D, bool F16>
cudaError_t finalize_t(const RowGrid& g, const SimtArgs& a, const BwdWorkspace& ws, int* err, cudaStream_t s) {
    const float* acc = ws.dq_acc;
    if (g.idx32)
        return launch_pdl(bwd_dq_finalize_kernel<D, unsigned, F16>, dim3(g.blocks), dim3(256), 0, s, a, acc, err);
    return launch_pdl(bwd_dq_finalize_kernel<D, unsigned long long, F16>, dim3(g.blocks), dim3(256), 0, s, a, acc,
                      err);
}
}  // namespace

cudaError_t launch_bwd_prepass(const attn_bwd_params& p, const BwdWorkspace& ws, int* err, cudaStream_t s) {
    const SimtArgs a = make_bwd_args(p, ws);
    const RowGrid g = row_grid((long long)p.fwd.B * p.fwd.H * ((p.fwd.N + 127) / 128 * 128), p.fwd.d);
    const bool f16 = p.fwd.dtype == ATTN_F16;
    cudaError_t e;
    if (p.fwd.d == 64)
        e = f16 ? prepass_t<64, true>(g, a, ws, err, s) : prepass_t<64, false>(g, a, ws, err, s);
    else if (p.fwd.d == 128)
        e = f16 ? prepass_t<128, true>(g, a, ws, err, s) : prepass_t<128, false>(g, a, ws, err, s);
    else
        e = f16 ? prepass_t<256, true>(g, a, ws, err, s) : prepass_t<256, false>(g, a, ws, err, s);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_bwd_dq_finalize(const attn_bwd_params& p, const BwdWorkspace& ws, int* err, cudaStream_t s) {
    const SimtArgs a = make_bwd_args(p, ws);
    const RowGrid g = row_grid((long long)p.fwd.B * p.fwd.H * p.fwd.N, p.fwd.d);
    const bool f16 = p.fwd.dtype == ATTN_F16;
    cudaError_t e;
    if (p.fwd.d == 64)
        e = f16 ? finalize_t<64, true>(g, a, ws, err, s) : finalize_t<64, false>(g, a, ws, err, s);
    else if (p.fwd.d == 128)
        e = f16 ? finalize_t<128, true>(g, a, ws, err, s) : finalize_t<128, false>(g, a, ws, err, s);
    else
        e = f16 ? finalize_t<256, true>(g, a, ws, err, s) : finalize_t<256, false>(g, a, ws, err, s);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace attn
