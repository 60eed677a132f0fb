// attn_decode.cu — split-KV decode: a few query rows against a long key/value
// sequence.
//
// A decode step has no N x N matrix to avoid: its cost is one read of the
// keys and values, and with a small batch that read must be spread over the
// sequence to occupy the GPU ("FlashAttention", "What it does not do"). Each
// work unit therefore takes one (b, h) and one contiguous key range (a
// split), runs the online softmax of "Explain FlashAttention and why it is
// IO-aware" over that range for every query row, and writes the row's
// partial state: the running max m, the sum l of 2^(s - m), the divisor lo
// of o (l with its largest term as rounded for the P V product: see
// o_divisor in ptx.cuh) and the unnormalised o. The per-split pass runs on
// the tensor cores (attn_decode_tc.cu). The combine kernel here merges the
// splits of a row with the same rescaling that merges tiles:
//   M = max m_s, w_s = 2^(m_s - M), O = sum w_s o_s / sum w_s lo_s,
//   LSE = ln 2 (M + log2 sum w_s l_s).
// Scores are in the log2 domain: s = c * (q . k) with c = scale * log2(e).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int KB = 64;  // split lengths are multiples of this many keys
constexpr unsigned kFull = 0xffffffffu;

// What the combine kernel reads and writes.
struct CombineArgs {
    uint8_t* o;
    float* lse;
    long long o_sb, o_sh, o_sn;  // elements
    int B, H, nq;
    int splits;    // key ranges per (b, h)
    float* part;   // [B*H][splits][nq][D + 4]: m, l, lo, 1 unused, o[D]
};

template <int D>
constexpr int rec_floats() {
    return D + 4;
}

template <int D, bool F16>
__global__ void __launch_bounds__(256) decode_combine_kernel(CombineArgs a) {
    ptx::grid_dep_wait();  // the split pass's records have landed
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
    float L = 0.f, Lo = 0.f, out[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) out[e] = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < a.splits; ++s) {
            const float* r = base + s * sstride;
            const float w = ptx::ex2(r[0] - M);  // 0 for a split that saw no key of this row
            L += w * r[1];
            Lo += w * r[2];
#pragma unroll
            for (int e = 0; e < PER; ++e) out[e] = fmaf(w, r[4 + lane * PER + e], out[e]);
        }
    }
    const float inv = Lo > 0.f ? 1.f / Lo : 0.f;
    uint16_t* orow = reinterpret_cast<uint16_t*>(a.o) + (b * a.o_sb + h * a.o_sh + (long long)i * a.o_sn);
    if constexpr (PER == 2) {
        *reinterpret_cast<uint32_t*>(orow + lane * 2) = ptx::pack_h16<F16>(out[0] * inv, out[1] * inv);
    } else {
        *reinterpret_cast<uint2*>(orow + lane * 4) =
            make_uint2(ptx::pack_h16<F16>(out[0] * inv, out[1] * inv), ptx::pack_h16<F16>(out[2] * inv, out[3] * inv));
    }
    if (lane == 0) a.lse[(long long)bh * a.nq + i] = L > 0.f ? (M + __log2f(L)) * kLn2 : -INFINITY;
}

template <int D, bool F16>
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s) {
    const int rows = a.B * a.H * a.nq;
    const cudaError_t e = launch_pdl(decode_combine_kernel<D, F16>, dim3((rows + 7) / 8), dim3(256), 0, s, a);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

DecodeSplit decode_split_plan(const attn_decode_params& p, int num_sms) {
    const int max_splits = (p.nk + KB - 1) / KB;
    int splits = p.num_splits;
    if (splits <= 0) {
        // about eight units per SM for the persistent split pass (one CTA per SM), so the
        // last round of units leaves few SMs idle; each range at least 256 keys
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

cudaError_t launch_decode(const attn_decode_params& p, const DecodeSplit& plan, const DecodeMaps& maps,
                          const LaunchCommon& lc, cudaStream_t s) {
    cudaError_t e = launch_decode_tc(p, plan, maps, lc, s);
    if (e != cudaSuccess) return e;
    CombineArgs a{};
    a.o = static_cast<uint8_t*>(p.o);
    a.lse = p.lse;
    a.o_sb = p.o_stride[0];
    a.o_sh = p.o_stride[1];
    a.o_sn = p.o_stride[2];
    a.B = p.B;
    a.H = p.H;
    a.nq = p.nq;
    a.splits = plan.splits;
    a.part = static_cast<float*>(p.workspace);
    const bool f16 = p.dtype == ATTN_F16;
    if (p.d == 64) return f16 ? launch_combine<64, true>(a, s) : launch_combine<64, false>(a, s);
    return f16 ? launch_combine<128, true>(a, s) : launch_combine<128, false>(a, s);
}

}  // namespace attn
