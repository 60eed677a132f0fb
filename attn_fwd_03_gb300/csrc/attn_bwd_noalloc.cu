// attn_bwd_noalloc.cu — the backward pass with library-owned scratch memory.
//
// attn_bwd needs a caller-provided device workspace (the per-tile row
// statistics and the fp32 dQ accumulator). Some callers cannot provide one:
// code that must not call cudaMalloc (or a framework allocator) at that point,
// for example inside a custom allocator's own callback, in a plug-in whose
// host process owns every allocation, or on a path with a fixed memory budget.
// attn_bwd_noalloc serves them: the workspace lives in a fixed-size array that
// the library declares in device memory, so the call allocates nothing. The
// caller still passes every input and output buffer.
//
// The array is a file-scope static __device__ object. Every GPU that loads
// this library holds it (kStaticWorkspaceBytes) for the life of the process.
// Host code only sees a stand-in symbol for it, so its device address is
// looked up with cudaGetSymbolAddress once per device and handed to the
// kernels.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"

namespace attn {
namespace {

// 40 MiB: enough for B*H*N*d fp32 dQ rows plus statistics up to about 10 M
// elements, e.g. B=4, H=16, N=2048, d=64.
constexpr size_t kStaticWorkspaceBytes = size_t(40) << 20;

static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

constexpr int kMaxDevices = 64;
std::mutex g_ws_mu;
void* g_ws_ptr[kMaxDevices] = {};

// Device address of the array on the current device, looked up on first use.
attn_status_t static_workspace(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return report_error(ATTN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return report_error(ATTN_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_ws_mu);
    if (!g_ws_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_workspace);
        if (e != cudaSuccess || p == nullptr)
            return report_error(ATTN_ERR_CUDA, "cudaGetSymbolAddress(static workspace): %s", cudaGetErrorString(e));
        g_ws_ptr[dev] = p;
    }
    *out = g_ws_ptr[dev];
    return ATTN_OK;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" attn_status_t attn_bwd_noalloc(const attn_bwd_params* p, void* stream) {
    bool empty = false;
    attn_status_t st = bwd_check_inputs(p, &empty);
    if (st != ATTN_OK || empty) return st;
    const size_t need = bwd_workspace_bytes(p->fwd);
    if (need > kStaticWorkspaceBytes)
        return report_error(ATTN_ERR_WORKSPACE,
                            "attn_bwd_noalloc: this problem needs %zu bytes of scratch, the built-in area holds %zu "
                            "(use attn_bwd with a caller workspace)",
                            need, kStaticWorkspaceBytes);
    void* base = nullptr;
    if ((st = static_workspace(&base)) != ATTN_OK) return st;
    // The pre-pass rewrites every statistic and zeroes every dQ accumulator row
    // this call uses, so nothing left from an earlier call leaks into the result.
    return bwd_launch_with(*p, bwd_workspace_at(base, p->fwd), stream);
}
