// attn_api.cu — the C ABI (include/attn.h): argument checks, the device error
// word, TMA tensor-map construction and kernel launches.
//
// Nothing here allocates device memory. Argument errors are detected before
// any launch and returned with a message (attn_last_error); in-kernel errors
// (a bounded wait that ran out) land in a per-device error word that
// attn_status() reads and clears.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace attn {

__device__ int g_error_word;  // one per device; ATTN_ERR_TIMEOUT when a kernel gave up

namespace {

thread_local char t_last_error[512] = "";
thread_local int32_t t_stall_after = 0;
thread_local void* t_bwd_events[4] = {nullptr, nullptr, nullptr, nullptr};
thread_local bool t_bwd_events_on = false;

constexpr uint32_t kLaunchLog = 16;
thread_local uint64_t t_launches = 0;
thread_local const void* t_launch_fn[kLaunchLog] = {};

cudaError_t record_bwd_event(int i, cudaStream_t s) {
    if (!t_bwd_events_on) return cudaSuccess;
    return cudaEventRecord(static_cast<cudaEvent_t>(t_bwd_events[i]), s);
}
uint64_t g_timeout_ns = 2000000000ull;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_err_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

attn_status_t fail(attn_status_t st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
    va_end(ap);
    return st;
}

attn_status_t cuda_fail(cudaError_t e, const char* what) {
    return fail(ATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Device error word address and SM count of the current device, set up once.
attn_status_t device_setup(LaunchCommon* lc) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_error_word);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        g_err_ptr[dev] = static_cast<int*>(p);
        g_num_sms[dev] = sms;
    }
    lc->err = g_err_ptr[dev];
    lc->num_sms = g_num_sms[dev];
    lc->timeout_ns = g_timeout_ns;
    lc->stall_after = t_stall_after;
    return ATTN_OK;
}

size_t elem_size(int32_t dtype) { return dtype == ATTN_F32 ? 4 : 2; }

bool misaligned_ptr(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

attn_status_t check_tensor(const char* name, const void* ptr, const int64_t* st, size_t es, bool allow_zero) {
    if (!ptr) return fail(ATTN_ERR_INVALID, "%s is NULL", name);
    for (int i = 0; i < 3; ++i) {
        if (st[i] < 0 || (!allow_zero && st[i] == 0))
            return fail(ATTN_ERR_INVALID, "%s stride[%d] = %lld is not positive", name, i, (long long)st[i]);
        if (((uint64_t)st[i] * es) % 16 != 0)
            return fail(ATTN_ERR_ALIGN, "%s stride[%d] = %lld elements is not a multiple of 16 bytes", name, i,
                        (long long)st[i]);
        if ((uint64_t)st[i] * es >= (1ull << 40))
            return fail(ATTN_ERR_UNSUPPORTED, "%s stride[%d] too large", name, i);
    }
    if (misaligned_ptr(ptr)) return fail(ATTN_ERR_ALIGN, "%s is not 16-byte aligned", name);
    return ATTN_OK;
}

// Checks shared by forward and backward. *empty = nothing to compute.
attn_status_t check_fwd(const attn_fwd_params* p, bool* empty) {
    if (!p) return fail(ATTN_ERR_INVALID, "params is NULL");
    if (p->B < 0 || p->H < 0 || p->N < 0)
        return fail(ATTN_ERR_INVALID, "negative size B=%d H=%d N=%d", p->B, p->H, p->N);
    if (p->dtype == ATTN_E4M3) return fail(ATTN_ERR_UNSUPPORTED, "E4M3 inputs go through attn_fwd_fp8");
    if (p->dtype != ATTN_BF16 && p->dtype != ATTN_F32 && p->dtype != ATTN_F16)
        return fail(ATTN_ERR_INVALID, "unknown dtype %d", p->dtype);
    if (p->causal != 0 && p->causal != 1) return fail(ATTN_ERR_INVALID, "causal must be 0 or 1, got %d", p->causal);
    if (p->reserved0 != 0) return fail(ATTN_ERR_INVALID, "reserved0 must be 0");
    if (!std::isfinite(p->scale) || !(p->scale > 0.f))
        return fail(ATTN_ERR_INVALID, "scale must be positive and finite");
    if (p->d != 64 && p->d != 128 && p->d != 256)
        return fail(ATTN_ERR_UNSUPPORTED, "head dim %d not built (64, 128 or 256)", p->d);
    if (p->d == 256 && p->dtype == ATTN_F32)
        return fail(ATTN_ERR_UNSUPPORTED, "head dim 256 is built for bf16 and fp16 only");
    if (p->B > 65535 || p->H > 65535) return fail(ATTN_ERR_UNSUPPORTED, "B and H are limited to 65535");
    *empty = (p->B == 0 || p->H == 0 || p->N == 0);
    if (*empty) return ATTN_OK;
    const size_t es = elem_size(p->dtype);
    attn_status_t st;
    if ((st = check_tensor("q", p->q, p->q_stride, es, false)) != ATTN_OK) return st;
    if ((st = check_tensor("k", p->k, p->k_stride, es, false)) != ATTN_OK) return st;
    if ((st = check_tensor("v", p->v, p->v_stride, es, false)) != ATTN_OK) return st;
    if ((st = check_tensor("o", p->o, p->o_stride, es, false)) != ATTN_OK) return st;
    if (!p->lse) return fail(ATTN_ERR_INVALID, "lse is NULL");
    if (misaligned_ptr(p->lse)) return fail(ATTN_ERR_ALIGN, "lse is not 16-byte aligned");
    if (p->mask && (st = check_tensor("mask", p->mask, p->mask_stride, es, true)) != ATTN_OK) return st;
    if (p->mask && p->mask_stride[2] == 0 && p->N > 1)
        return fail(ATTN_ERR_INVALID, "mask row stride must be positive");
    return ATTN_OK;
}

// ---------------------------------------------------------------- tensor maps
attn_status_t get_encoder() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode) return ATTN_OK;
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return ATTN_OK;
}

// 4-D map of 16-bit elements (bf16 or fp16, as `dtype` says) over (col, row, h, b)
// with a 64 x box_rows box and the 128-byte swizzle: one box is box_rows rows of
// 128 bytes.
attn_status_t encode_h16_map(CUtensorMap* m, const char* name, const void* base, uint64_t cols, uint64_t rows,
                             uint64_t hs, uint64_t bs, const int64_t* st, uint32_t box_rows, int32_t dtype) {
    cuuint64_t dims[4] = {cols, rows, hs, bs};
    cuuint64_t strides[3] = {(cuuint64_t)st[2] * 2, (cuuint64_t)st[1] * 2, (cuuint64_t)st[0] * 2};
    // a dimension of extent 1 may carry stride 0 (broadcast); give it a legal one
    for (int i = 0; i < 3; ++i)
        if (strides[i] == 0) strides[i] = 16;
    cuuint32_t box[4] = {64, box_rows, 1, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    const CUtensorMapDataType dt =
        dtype == ATTN_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUresult r = g_encode(m, dt, 4, const_cast<void*>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", name, (int)r);
    return ATTN_OK;
}

// fp32 map over the dQ accumulator [B, H, N, d] (contiguous), 32-column x 128-row
// boxes with the 128-byte swizzle, used by the TMA reductions of the backward.
attn_status_t encode_dq_acc_map(const attn_fwd_params& p, float* dq_acc, CUtensorMap* m) {
    attn_status_t st = get_encoder();
    if (st != ATTN_OK) return st;
    const uint64_t d = (uint64_t)p.d, N = (uint64_t)p.N;
    cuuint64_t dims[4] = {d, N, (cuuint64_t)p.H, (cuuint64_t)p.B};
    cuuint64_t strides[3] = {d * 4, N * d * 4, (cuuint64_t)p.H * N * d * 4};
    cuuint32_t box[4] = {32, 128, 1, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dq_acc, dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled(dq accumulator) failed with %d", (int)r);
    return ATTN_OK;
}

attn_status_t build_fwd_maps(const attn_fwd_params& p, FwdMaps* m) {
    attn_status_t st = get_encoder();
    if (st != ATTN_OK) return st;
    const uint64_t N = (uint64_t)p.N, d = (uint64_t)p.d;
    const int32_t DT = p.dtype;
    if ((st = encode_h16_map(&m->q, "q", p.q, d, N, p.H, p.B, p.q_stride, 128, DT)) != ATTN_OK) return st;
    if ((st = encode_h16_map(&m->k, "k", p.k, d, N, p.H, p.B, p.k_stride, 128, DT)) != ATTN_OK) return st;
    if ((st = encode_h16_map(&m->v, "v", p.v, d, N, p.H, p.B, p.v_stride, 128, DT)) != ATTN_OK) return st;
    if ((st = encode_h16_map(&m->o, "o", p.o, d, N, p.H, p.B, p.o_stride, 128, DT)) != ATTN_OK) return st;
    if (p.d == 256) {
        if ((st = encode_h16_map(&m->v32, "v", p.v, d, N, p.H, p.B, p.v_stride, 32, DT)) != ATTN_OK) return st;
    } else {
        m->v32 = m->v;  // unused below head dim 256
    }
    if (p.mask) {
        const uint64_t hm = p.mask_stride[1] != 0 ? (uint64_t)p.H : 1;
        const uint64_t bm = p.mask_stride[0] != 0 ? (uint64_t)p.B : 1;
        if ((st = encode_h16_map(&m->mask, "mask", p.mask, N, N, hm, bm, p.mask_stride, 128, DT)) != ATTN_OK)
            return st;
    } else {
        m->mask = m->q;  // unused by the kernel variant without a mask
    }
    return ATTN_OK;
}

// 4-D map of E4M3 codes over (col, row, h, b) with 128-byte x box_rows boxes and the 128-byte swizzle.
attn_status_t encode_u8_map(CUtensorMap* m, const char* name, const void* base, uint64_t cols, uint64_t rows,
                            uint64_t hs, uint64_t bs, const int64_t* st, uint32_t box_rows) {
    cuuint64_t dims[4] = {cols, rows, hs, bs};
    cuuint64_t strides[3] = {(cuuint64_t)st[2], (cuuint64_t)st[1], (cuuint64_t)st[0]};
    for (int i = 0; i < 3; ++i)
        if (strides[i] == 0) strides[i] = 16;
    cuuint32_t box[4] = {128, box_rows, 1, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", name, (int)r);
    return ATTN_OK;
}

attn_status_t check_fwd_fp8(const attn_fwd_fp8_params* p, bool* empty) {
    if (!p) return fail(ATTN_ERR_INVALID, "params is NULL");
    const attn_fwd_params& f = p->f;
    if (f.B < 0 || f.H < 0 || f.N < 0) return fail(ATTN_ERR_INVALID, "negative size B=%d H=%d N=%d", f.B, f.H, f.N);
    if (f.dtype != ATTN_E4M3) return fail(ATTN_ERR_UNSUPPORTED, "attn_fwd_fp8 takes ATTN_E4M3 inputs, got %d", f.dtype);
    if (f.causal != 0 && f.causal != 1) return fail(ATTN_ERR_INVALID, "causal must be 0 or 1, got %d", f.causal);
    if (f.reserved0 != 0 || p->reserved1 != 0) return fail(ATTN_ERR_INVALID, "reserved fields must be 0");
    if (!std::isfinite(f.scale) || !(f.scale > 0.f)) return fail(ATTN_ERR_INVALID, "scale must be positive and finite");
    const float ds[3] = {p->q_descale, p->k_descale, p->v_descale};
    for (int i = 0; i < 3; ++i)
        if (!std::isfinite(ds[i]) || !(ds[i] > 0.f))
            return fail(ATTN_ERR_INVALID, "descale factors must be positive and finite");
    if (f.d != 128 && f.d != 256)
        return fail(ATTN_ERR_UNSUPPORTED, "the FP8 forward is built for head dims 128 and 256, got %d", f.d);
    if (f.B > 65535 || f.H > 65535) return fail(ATTN_ERR_UNSUPPORTED, "B and H are limited to 65535");
    *empty = (f.B == 0 || f.H == 0 || f.N == 0);
    if (*empty) return ATTN_OK;
    attn_status_t st;
    if ((st = check_tensor("q", f.q, f.q_stride, 1, false)) != ATTN_OK) return st;
    if ((st = check_tensor("k", f.k, f.k_stride, 1, false)) != ATTN_OK) return st;
    if ((st = check_tensor("v", f.v, f.v_stride, 1, false)) != ATTN_OK) return st;
    if ((st = check_tensor("o", f.o, f.o_stride, 2, false)) != ATTN_OK) return st;
    if (!f.lse) return fail(ATTN_ERR_INVALID, "lse is NULL");
    if (misaligned_ptr(f.lse)) return fail(ATTN_ERR_ALIGN, "lse is not 16-byte aligned");
    if (f.mask && (st = check_tensor("mask", f.mask, f.mask_stride, 2, true)) != ATTN_OK) return st;
    if (f.mask && f.mask_stride[2] == 0 && f.N > 1) return fail(ATTN_ERR_INVALID, "mask row stride must be positive");
    return ATTN_OK;
}

attn_status_t build_fp8_maps(const attn_fwd_fp8_params& p, Fp8Maps* m) {
    attn_status_t st = get_encoder();
    if (st != ATTN_OK) return st;
    const attn_fwd_params& f = p.f;
    const uint64_t N = (uint64_t)f.N, d = (uint64_t)f.d;
    if ((st = encode_u8_map(&m->q, "q", f.q, d, N, f.H, f.B, f.q_stride, 128)) != ATTN_OK) return st;
    if ((st = encode_u8_map(&m->k, "k", f.k, d, N, f.H, f.B, f.k_stride, 128)) != ATTN_OK) return st;
    if ((st = encode_u8_map(&m->v, "v", f.v, d, N, f.H, f.B, f.v_stride, 128)) != ATTN_OK) return st;
    if (f.d == 256) {
        if ((st = encode_u8_map(&m->v64, "v", f.v, d, N, f.H, f.B, f.v_stride, 64)) != ATTN_OK) return st;
    } else {
        m->v64 = m->v;  // unused below head dim 256
    }
    if (f.mask) {
        const uint64_t hm = f.mask_stride[1] != 0 ? (uint64_t)f.H : 1;
        const uint64_t bm = f.mask_stride[0] != 0 ? (uint64_t)f.B : 1;
        return encode_h16_map(&m->mask, "mask", f.mask, N, N, hm, bm, f.mask_stride, 128, ATTN_BF16);
    }
    m->mask = m->q;  // unused by the kernel variant without a mask
    return ATTN_OK;
}

// Checks of a decode problem (all but the workspace). *empty = nothing to compute.
attn_status_t check_decode(const attn_decode_params* p, bool* empty) {
    if (!p) return fail(ATTN_ERR_INVALID, "params is NULL");
    if (p->B < 0 || p->H < 0 || p->nq < 0)
        return fail(ATTN_ERR_INVALID, "negative size B=%d H=%d nq=%d", p->B, p->H, p->nq);
    if (p->nk < 1) return fail(ATTN_ERR_INVALID, "nk must be at least 1, got %d", p->nk);
    if (p->dtype == ATTN_F32) return fail(ATTN_ERR_UNSUPPORTED, "decode is built for bf16 and fp16 only");
    if (p->dtype != ATTN_BF16 && p->dtype != ATTN_F16) return fail(ATTN_ERR_INVALID, "unknown dtype %d", p->dtype);
    if (p->causal != 0 && p->causal != 1) return fail(ATTN_ERR_INVALID, "causal must be 0 or 1, got %d", p->causal);
    if (p->reserved0 != 0) return fail(ATTN_ERR_INVALID, "reserved0 must be 0");
    if (p->num_splits < 0) return fail(ATTN_ERR_INVALID, "num_splits must be >= 0");
    if (!std::isfinite(p->scale) || !(p->scale > 0.f))
        return fail(ATTN_ERR_INVALID, "scale must be positive and finite");
    if (p->d != 64 && p->d != 128) return fail(ATTN_ERR_UNSUPPORTED, "head dim %d not built (64 or 128)", p->d);
    if (p->nq > 128) return fail(ATTN_ERR_UNSUPPORTED, "decode takes at most 128 query rows, got %d", p->nq);
    if ((long long)p->B * p->H > 65535) return fail(ATTN_ERR_UNSUPPORTED, "B * H is limited to 65535");
    *empty = (p->B == 0 || p->H == 0 || p->nq == 0);
    if (*empty) return ATTN_OK;
    attn_status_t st;
    if ((st = check_tensor("q", p->q, p->q_stride, 2, false)) != ATTN_OK) return st;
    if ((st = check_tensor("k", p->k, p->k_stride, 2, false)) != ATTN_OK) return st;
    if ((st = check_tensor("v", p->v, p->v_stride, 2, false)) != ATTN_OK) return st;
    if ((st = check_tensor("o", p->o, p->o_stride, 2, false)) != ATTN_OK) return st;
    if (!p->lse) return fail(ATTN_ERR_INVALID, "lse is NULL");
    if (misaligned_ptr(p->lse)) return fail(ATTN_ERR_ALIGN, "lse is not 16-byte aligned");
    return ATTN_OK;
}

attn_status_t build_bwd_maps(const attn_bwd_params& p, BwdMaps* m) {
    FwdMaps f;
    attn_status_t st = build_fwd_maps(p.fwd, &f);
    if (st != ATTN_OK) return st;
    m->q = f.q;
    m->k = f.k;
    m->v = f.v;
    m->mask = f.mask;
    const uint64_t N = (uint64_t)p.fwd.N, d = (uint64_t)p.fwd.d;
    const int32_t DT = p.fwd.dtype;
    if ((st = encode_h16_map(&m->dk, "dk", p.dk, d, N, p.fwd.H, p.fwd.B, p.dk_stride, 128, DT)) != ATTN_OK) return st;
    if ((st = encode_h16_map(&m->dv, "dv", p.dv, d, N, p.fwd.H, p.fwd.B, p.dv_stride, 128, DT)) != ATTN_OK) return st;
    return encode_h16_map(&m->dout, "dout", p.dout, d, N, p.fwd.H, p.fwd.B, p.do_stride, 128, DT);
}

attn_status_t build_bwd256_maps(const attn_bwd_params& p, Bwd256Maps* m) {
    FwdMaps f;
    attn_status_t st = build_fwd_maps(p.fwd, &f);
    if (st != ATTN_OK) return st;
    m->k = f.k;
    m->v = f.v;
    const uint64_t N = (uint64_t)p.fwd.N, d = (uint64_t)p.fwd.d;
    const int32_t DT = p.fwd.dtype;
    if ((st = encode_h16_map(&m->q64, "q", p.fwd.q, d, N, p.fwd.H, p.fwd.B, p.fwd.q_stride, 64, DT)) != ATTN_OK)
        return st;
    if ((st = encode_h16_map(&m->do64, "dout", p.dout, d, N, p.fwd.H, p.fwd.B, p.do_stride, 64, DT)) != ATTN_OK)
        return st;
    if (p.fwd.mask) {
        const uint64_t hm = p.fwd.mask_stride[1] != 0 ? (uint64_t)p.fwd.H : 1;
        const uint64_t bm = p.fwd.mask_stride[0] != 0 ? (uint64_t)p.fwd.B : 1;
        return encode_h16_map(&m->mask64, "mask", p.fwd.mask, N, N, hm, bm, p.fwd.mask_stride, 64, DT);
    }
    m->mask64 = m->q64;  // unused by the kernel variant without a mask
    return ATTN_OK;
}

// The recompute kernel of a backward pass: head dim 256 has its own kernel and maps.
attn_status_t launch_bwd_main(const attn_bwd_params& p, const BwdWorkspace& ws, const LaunchCommon& lc,
                              cudaStream_t s) {
    attn_status_t st;
    cudaError_t e;
    if (p.fwd.d == 256) {
        Bwd256Maps maps;
        if ((st = build_bwd256_maps(p, &maps)) != ATTN_OK) return st;
        e = launch_bwd256(p, maps, ws, lc, s);
    } else {
        BwdMaps maps;
        if ((st = build_bwd_maps(p, &maps)) != ATTN_OK) return st;
        if ((st = encode_dq_acc_map(p.fwd, ws.dq_acc, &maps.dq_acc)) != ATTN_OK) return st;
        e = launch_bwd_tc(p, maps, ws, lc, s);
    }
    return e != cudaSuccess ? cuda_fail(e, "backward main launch") : ATTN_OK;
}

}  // namespace

static size_t stats_bytes(const attn_fwd_params& p) {
    const size_t tiles = (size_t)p.B * p.H * (((size_t)p.N + 127) / 128);
    return tiles * 2 * 128 * sizeof(float);  // a multiple of 1024
}

size_t bwd_workspace_bytes(const attn_fwd_params& p) {
    const size_t rows = (size_t)p.B * p.H * p.N;
    if (rows == 0) return 0;
    return stats_bytes(p) + rows * (size_t)p.d * sizeof(float);
}

BwdWorkspace bwd_workspace_split(const attn_bwd_params& p) {
    char* base = static_cast<char*>(p.workspace);
    return BwdWorkspace{reinterpret_cast<float*>(base), reinterpret_cast<float*>(base + stats_bytes(p.fwd))};
}

void note_launch(const void* kernel) {
    t_launch_fn[t_launches % kLaunchLog] = kernel;
    ++t_launches;
}

// ---- helpers for entry points that supply their own workspace storage
attn_status_t report_error(attn_status_t st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
    va_end(ap);
    return st;
}

attn_status_t bwd_check_inputs(const attn_bwd_params* p, bool* empty) {
    if (!p) return fail(ATTN_ERR_INVALID, "params is NULL");
    attn_status_t st = check_fwd(&p->fwd, empty);
    if (st != ATTN_OK) return st;
    if (p->fwd.dtype == ATTN_F32) return fail(ATTN_ERR_UNSUPPORTED, "backward is built for bf16 and fp16 only");
    if (*empty) return ATTN_OK;
    if ((st = check_tensor("dout", p->dout, p->do_stride, 2, false)) != ATTN_OK) return st;
    if ((st = check_tensor("dq", p->dq, p->dq_stride, 2, false)) != ATTN_OK) return st;
    if ((st = check_tensor("dk", p->dk, p->dk_stride, 2, false)) != ATTN_OK) return st;
    return check_tensor("dv", p->dv, p->dv_stride, 2, false);
}

attn_status_t build_dq_acc_map(const attn_fwd_params& p, float* dq_acc, CUtensorMap* m) {
    return encode_dq_acc_map(p, dq_acc, m);
}

BwdWorkspace bwd_workspace_at(void* base, const attn_fwd_params& f) {
    char* b = static_cast<char*>(base);
    return BwdWorkspace{reinterpret_cast<float*>(b), reinterpret_cast<float*>(b + stats_bytes(f))};
}

attn_status_t bwd_launch_with(const attn_bwd_params& p, const BwdWorkspace& ws, void* stream) {
    LaunchCommon lc;
    attn_status_t st = device_setup(&lc);
    if (st != ATTN_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_bwd_prepass(p, ws, lc.err, s);
    if (e != cudaSuccess) return cuda_fail(e, "backward pre-pass launch");
    if ((st = launch_bwd_main(p, ws, lc, s)) != ATTN_OK) return st;
    if ((e = launch_bwd_dq_finalize(p, ws, lc.err, s)) != cudaSuccess)
        return cuda_fail(e, "backward dQ finalize launch");
    return ATTN_OK;
}

}  // namespace attn

using namespace attn;

extern "C" {

attn_status_t attn_fwd(const attn_fwd_params* p, void* stream) {
    bool empty = false;
    attn_status_t st = check_fwd(p, &empty);
    if (st != ATTN_OK || empty) return st;
    LaunchCommon lc;
    if ((st = device_setup(&lc)) != ATTN_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (p->dtype == ATTN_F32) {
        e = launch_fwd_simt(*p, s);
    } else {
        FwdMaps maps;
        if ((st = build_fwd_maps(*p, &maps)) != ATTN_OK) return st;
        e = p->d == 256 ? launch_fwd256(*p, maps, lc, s) : launch_fwd_tc(*p, maps, lc, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "attn_fwd launch");
    return ATTN_OK;
}

attn_status_t attn_fwd_fp8(const attn_fwd_fp8_params* p, void* stream) {
    bool empty = false;
    attn_status_t st = check_fwd_fp8(p, &empty);
    if (st != ATTN_OK || empty) return st;
    LaunchCommon lc;
    if ((st = device_setup(&lc)) != ATTN_OK) return st;
    Fp8Maps maps;
    if ((st = build_fp8_maps(*p, &maps)) != ATTN_OK) return st;
    const cudaError_t e = p->f.d == 256 ? launch_fwd256_fp8(*p, maps, lc, static_cast<cudaStream_t>(stream))
                                        : launch_fwd_fp8(*p, maps, lc, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "attn_fwd_fp8 launch");
    return ATTN_OK;
}

size_t attn_bwd_workspace_size(const attn_fwd_params* p) {
    if (!p || p->B < 0 || p->H < 0 || p->N < 0 || (p->d != 64 && p->d != 128 && p->d != 256)) return 0;
    return bwd_workspace_bytes(*p);
}

attn_status_t attn_bwd(const attn_bwd_params* p, void* stream) {
    bool empty = false;
    attn_status_t st = bwd_check_inputs(p, &empty);
    if (st != ATTN_OK || empty) return st;
    const size_t need = bwd_workspace_bytes(p->fwd);
    if (!p->workspace || p->workspace_bytes < need)
        return fail(ATTN_ERR_WORKSPACE, "workspace of %zu bytes given, %zu needed", p->workspace_bytes, need);
    if ((reinterpret_cast<uintptr_t>(p->workspace) & 255u) != 0)
        return fail(ATTN_ERR_ALIGN, "workspace is not 256-byte aligned");
    LaunchCommon lc;
    if ((st = device_setup(&lc)) != ATTN_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const BwdWorkspace ws = bwd_workspace_split(*p);
    cudaError_t e = record_bwd_event(0, s);
    if (e == cudaSuccess) e = launch_bwd_prepass(*p, ws, lc.err, s);
    if (e != cudaSuccess) return cuda_fail(e, "attn_bwd pre-pass launch");
    if ((e = record_bwd_event(1, s)) != cudaSuccess) return cuda_fail(e, "attn_bwd event record");
    if ((st = launch_bwd_main(*p, ws, lc, s)) != ATTN_OK) return st;
    if ((e = record_bwd_event(2, s)) == cudaSuccess) e = launch_bwd_dq_finalize(*p, ws, lc.err, s);
    if (e != cudaSuccess) return cuda_fail(e, "attn_bwd dQ finalize launch");
    if ((e = record_bwd_event(3, s)) != cudaSuccess) return cuda_fail(e, "attn_bwd event record");
    return ATTN_OK;
}

attn_status_t attn_bwd_deterministic(const attn_bwd_params* p, void* stream) {
    if (p && p->fwd.d == 256)
        return fail(ATTN_ERR_UNSUPPORTED, "the deterministic backward is built for head dim 64 and 128");
    bool empty = false;
    attn_status_t st = bwd_check_inputs(p, &empty);
    if (st != ATTN_OK || empty) return st;
    const size_t need = bwd_workspace_bytes(p->fwd);
    if (!p->workspace || p->workspace_bytes < need)
        return fail(ATTN_ERR_WORKSPACE, "workspace of %zu bytes given, %zu needed", p->workspace_bytes, need);
    if ((reinterpret_cast<uintptr_t>(p->workspace) & 255u) != 0)
        return fail(ATTN_ERR_ALIGN, "workspace is not 256-byte aligned");
    LaunchCommon lc;
    if ((st = device_setup(&lc)) != ATTN_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const BwdWorkspace ws = bwd_workspace_split(*p);
    BwdMaps maps;
    if ((st = build_bwd_maps(*p, &maps)) != ATTN_OK) return st;
    if ((st = encode_dq_acc_map(p->fwd, ws.dq_acc, &maps.dq_acc)) != ATTN_OK) return st;
    // dK and dV come from the key-stationary kernel, whose sums over query tiles run in a
    // fixed order; its dQ accumulator output is not used. dQ comes from the query-stationary
    // kernel, which sums over key tiles in a fixed order and writes dQ itself.
    cudaError_t e = launch_bwd_prepass(*p, ws, lc.err, s);
    if (e != cudaSuccess) return cuda_fail(e, "attn_bwd_deterministic pre-pass launch");
    if ((e = launch_bwd_tc(*p, maps, ws, lc, s)) != cudaSuccess)
        return cuda_fail(e, "attn_bwd_deterministic dK/dV launch");
    if ((e = launch_bwd_dq(*p, maps, ws, lc, s)) != cudaSuccess)
        return cuda_fail(e, "attn_bwd_deterministic dQ launch");
    return ATTN_OK;
}

size_t attn_decode_workspace_size(const attn_decode_params* p) {
    bool empty = false;
    if (check_decode(p, &empty) != ATTN_OK || empty) return 0;
    LaunchCommon lc;
    if (device_setup(&lc) != ATTN_OK) return 0;
    return decode_split_plan(*p, lc.num_sms).workspace_bytes;
}

attn_status_t attn_decode(const attn_decode_params* p, void* stream) {
    bool empty = false;
    attn_status_t st = check_decode(p, &empty);
    if (st != ATTN_OK || empty) return st;
    LaunchCommon lc;
    if ((st = device_setup(&lc)) != ATTN_OK) return st;
    const DecodeSplit plan = decode_split_plan(*p, lc.num_sms);
    if (!p->workspace) return fail(ATTN_ERR_INVALID, "workspace is NULL");
    if ((reinterpret_cast<uintptr_t>(p->workspace) & 255u) != 0)
        return fail(ATTN_ERR_ALIGN, "workspace is not 256-byte aligned");
    if (p->workspace_bytes < plan.workspace_bytes)
        return fail(ATTN_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", p->workspace_bytes,
                    plan.workspace_bytes);
    DecodeMaps maps;
    if ((st = get_encoder()) != ATTN_OK) return st;
    const uint64_t d = (uint64_t)p->d;
    if ((st = encode_h16_map(&maps.q, "q", p->q, d, (uint64_t)p->nq, p->H, p->B, p->q_stride, 128, p->dtype)) !=
        ATTN_OK)
        return st;
    if ((st = encode_h16_map(&maps.k, "k", p->k, d, (uint64_t)p->nk, p->H, p->B, p->k_stride, 128, p->dtype)) !=
        ATTN_OK)
        return st;
    if ((st = encode_h16_map(&maps.v, "v", p->v, d, (uint64_t)p->nk, p->H, p->B, p->v_stride, 128, p->dtype)) !=
        ATTN_OK)
        return st;
    cudaError_t e = launch_decode(*p, plan, maps, lc, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "attn_decode launch");
    return ATTN_OK;
}

attn_status_t attn_status(void* stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "asynchronous CUDA error");
    LaunchCommon lc;
    attn_status_t st = device_setup(&lc);
    if (st != ATTN_OK) return st;
    int word = 0;
    e = cudaMemcpyFromSymbol(&word, g_error_word, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    if (word != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int));
        if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
        if (word == ATTN_ERR_TIMEOUT) return fail(ATTN_ERR_TIMEOUT, "a kernel's bounded wait ran out");
        if (word == -7) return fail(ATTN_ERR_CUDA, "a kernel skipped a misaligned access or buffer");
        return fail(ATTN_ERR_CUDA, "device error word %d", word);
    }
    return ATTN_OK;
}

const char* attn_last_error(void) { return t_last_error; }

void attn_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns = ns < 1000000ull ? 1000000ull : ns; }

void attn_debug_set_producer_stall(int32_t kv_tiles) { t_stall_after = kv_tiles > 0 ? kv_tiles : 0; }

void attn_debug_set_bwd_events(void* const events[4]) {
    t_bwd_events_on = events != nullptr;
    for (int i = 0; i < 4; ++i) t_bwd_events[i] = events ? events[i] : nullptr;
}

uint64_t attn_debug_launch_count(void) { return t_launches; }

const char* attn_debug_launch_name(uint32_t back) {
    if (back >= kLaunchLog || back >= t_launches) return nullptr;
    const void* fn = t_launch_fn[(t_launches - 1 - back) % kLaunchLog];
    const char* name = nullptr;
    if (cudaFuncGetName(&name, fn) != cudaSuccess || !name) return "?";
    return name;
}

int32_t attn_version(void) { return 100; }

}  // extern "C"
