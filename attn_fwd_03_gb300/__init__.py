"""Exact tiled attention for GB300 (sm_103a): a C-ABI CUDA library and its
thin Python binding.

    from attn_fwd_03_gb300 import attn_fwd, attn_bwd
    o, lse = attn_fwd(q, k, v, causal=True)            # q, k, v: [B, H, N, d] on cuda
    dq, dk, dv = attn_bwd(q, k, v, o, lse, do, causal=True)
    o1, lse1 = attn_decode(q1, k_cache, v_cache, causal=True)  # q1: [B, H, nq <= 128, d]
    o8, lse8 = attn_fwd_fp8(q8, k8, v8, q_descale, k_descale, v_descale)  # E4M3 inputs, d = 128

The kernels live in csrc/ (built in-tree by build.py); the public C header is
include/attn.h at the repository root.
"""
from ._binding import (  # noqa: F401
    ATTN_BF16, ATTN_E4M3, ATTN_ERR_ALIGN, ATTN_ERR_CUDA, ATTN_ERR_INVALID, ATTN_ERR_TIMEOUT, ATTN_ERR_UNSUPPORTED,
    ATTN_ERR_WORKSPACE, ATTN_F16, ATTN_F32, ATTN_OK, EXPORTED, LIB_PATH, AttnError, BwdParams, DecodeParams,
    Fp8Params, FwdParams, attn_bwd, attn_bwd_deterministic, attn_bwd_noalloc, attn_decode, attn_fwd, attn_fwd_fp8,
    attn_status, bwd_workspace_size, debug_set_bwd_events, debug_set_producer_stall, decode_workspace_size,
    last_error, launch_count, launch_names, lib, set_wait_timeout_ns, version,
)
