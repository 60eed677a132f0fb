// internal.h — declarations shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/attn.h"

namespace attn {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// What every launch needs besides the problem itself.
struct LaunchCommon {
    int* err;             // device error word of the current device
    uint64_t timeout_ns;  // bound on any single in-kernel wait
    int32_t stall_after;  // test hook: load warp stops after this many K/V tiles (0 = off)
    int num_sms;          // SM count of the current device
};

// Records one kernel launch of the library on the calling host thread (the launch log that
// attn_debug_launch_count / attn_debug_launch_name read back). Called once a launch has been
// issued without error.
void note_launch(const void* kernel);

// Launches `kernel` with programmatic stream serialization, so that it may start while the
// kernel before it in the stream still runs. Every kernel launched this way executes
// griddepcontrol.wait before its first global memory access, which returns once the previous
// kernel has completed and its writes are visible; a kernel that follows a non-kernel
// operation is serialised as usual.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       const Args&... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    if (e == cudaSuccess) note_launch(reinterpret_cast<const void*>(kernel));
    return e;
}

// Tensor maps for the tcgen05 forward (built by the host API).
struct FwdMaps {
    CUtensorMap q, k, v, o, mask;
    CUtensorMap v32;  // d = 256 only: V with 32-row boxes
};

// Tensor maps for the tcgen05 backward.
struct BwdMaps {
    CUtensorMap q, k, v, dout, mask;
    CUtensorMap dq_acc;  // fp32 view of the workspace's dQ accumulator (32 x 128 boxes, 128-byte swizzle)
    CUtensorMap dk, dv;  // outputs (64 x 128 boxes, 128-byte swizzle) for TMA stores of dK / dV tiles
};

// Tensor maps for the head-dim-256 backward: K, V with 128-row boxes; Q, dO and the mask with
// 64-row boxes (64-query tiles).
struct Bwd256Maps {
    CUtensorMap q64, k, v, do64, mask64;
};

// The two parts of the backward workspace.
//  stats:  per (b, h) and 128-row query tile, 128 values of -LSE * log2(e)
//          (-inf for fully masked rows and padding rows) followed by 128 values
//          of -D = -rowsum(dO * O); fp32 [B*H][ceil(N/128)][2][128]
//  dq_acc: fp32 [B, H, N, d] dQ accumulator (already multiplied by the scale)
struct BwdWorkspace {
    float* stats;
    float* dq_acc;
};
size_t bwd_workspace_bytes(const attn_fwd_params& p);
BwdWorkspace bwd_workspace_split(const attn_bwd_params& p);

// attn_api.cu — shared by entry points that supply their own workspace storage.
attn_status_t report_error(attn_status_t st, const char* fmt, ...);
attn_status_t bwd_check_inputs(const attn_bwd_params* p, bool* empty);  // all but the workspace
BwdWorkspace bwd_workspace_at(void* base, const attn_fwd_params& f);
attn_status_t bwd_launch_with(const attn_bwd_params& p, const BwdWorkspace& ws, void* stream);
attn_status_t build_dq_acc_map(const attn_fwd_params& p, float* dq_acc, CUtensorMap* m);

// attn_decode.cu — split-KV decode. The plan (key ranges per (b, h) and their
// length) fixes the workspace size, so the host API and the launch share it.
struct DecodeSplit {
    int splits;
    int chunk;  // keys per range, a multiple of 64
    size_t workspace_bytes;
};
DecodeSplit decode_split_plan(const attn_decode_params& p, int num_sms);
// Tensor maps of the tensor-core split pass: q, k, v with 64-column x 128-row boxes.
struct DecodeMaps {
    CUtensorMap q, k, v;
};
// The tensor-core split pass (attn_decode_tc.cu), then the combine kernel (attn_decode.cu).
cudaError_t launch_decode(const attn_decode_params& p, const DecodeSplit& plan, const DecodeMaps& maps,
                          const LaunchCommon& lc, cudaStream_t s);
cudaError_t launch_decode_tc(const attn_decode_params& p, const DecodeSplit& plan, const DecodeMaps& maps,
                             const LaunchCommon& lc, cudaStream_t s);

// attn_fwd_sm103.cu — tcgen05 forward (bf16).
cudaError_t launch_fwd_tc(const attn_fwd_params& p, const FwdMaps& maps, const LaunchCommon& lc, cudaStream_t s);

// Tensor maps for the FP8 forward: E4M3 q, k, v (128-byte x 128-row boxes), bf16 mask, and
// for head dim 256 V again with 64-row boxes.
struct Fp8Maps {
    CUtensorMap q, k, v, mask, v64;
};
// attn_fwd_fp8.cu — tcgen05 kind::f8f6f4 forward, head dim 128.
cudaError_t launch_fwd_fp8(const attn_fwd_fp8_params& p, const Fp8Maps& maps, const LaunchCommon& lc,
                           cudaStream_t s);
// attn_fwd256.cu — the same for head dim 256.
cudaError_t launch_fwd256_fp8(const attn_fwd_fp8_params& p, const Fp8Maps& maps, const LaunchCommon& lc,
                              cudaStream_t s);

// attn_fwd256.cu — tcgen05 forward for head dim 256 (bf16 / fp16).
cudaError_t launch_fwd256(const attn_fwd_params& p, const FwdMaps& maps, const LaunchCommon& lc, cudaStream_t s);

// attn_bwd_sm103.cu — tcgen05 backward main kernel (bf16).
cudaError_t launch_bwd_tc(const attn_bwd_params& p, const BwdMaps& maps, const BwdWorkspace& ws,
                          const LaunchCommon& lc, cudaStream_t s);

// attn_bwd256.cu — tcgen05 backward at head dim 256 (one half of the head dim of dK, dV, dQ per CTA).
cudaError_t launch_bwd256(const attn_bwd_params& p, const Bwd256Maps& maps, const BwdWorkspace& ws,
                          const LaunchCommon& lc, cudaStream_t s);

// attn_bwd_dq.cu — query-stationary tcgen05 dQ kernel (fixed order of additions); writes dQ
// in the dtype of Q from the row statistics in ws.stats.
cudaError_t launch_bwd_dq(const attn_bwd_params& p, const BwdMaps& maps, const BwdWorkspace& ws,
                          const LaunchCommon& lc, cudaStream_t s);

// attn_simt.cu — CUDA-core kernels.
cudaError_t launch_fwd_simt(const attn_fwd_params& p, cudaStream_t s);  // fp32 inputs
cudaError_t launch_bwd_prepass(const attn_bwd_params& p, const BwdWorkspace& ws, int* err, cudaStream_t s);
cudaError_t launch_bwd_dq_finalize(const attn_bwd_params& p, const BwdWorkspace& ws, int* err, cudaStream_t s);

}  // namespace attn
