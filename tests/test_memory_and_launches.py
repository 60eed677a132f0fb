"""The checks the pages run on a real system ("FlashAttention", "Checking it on a
real system"): peak memory grows linearly with N, because the N x N score
matrix is never stored, and each call runs as fused kernels rather than as a
chain of separate matmul / softmax / matmul launches.

Here the library allocates nothing at all: with outputs and the backward
workspace allocated by the caller, the peak allocated memory does not move
during a call, at any N. The only per-call memory is the caller's O(N) buffers.
The forward is one kernel launch, and the backward is three (pre-pass, main,
dQ finalize).
"""
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attn_fwd_03_gb300 as m
    return m


def _inputs(N, d=64, B=1, H=4, seed=900):
    return [W.random_tensor((B, H, N, d), seed + i, torch.bfloat16).cuda() for i in range(4)]


@pytest.mark.parametrize("N", [1024, 2048, 4096, 8192])
def test_calls_allocate_nothing(A, N):
    q, k, v, do = _inputs(N)
    o, lse = torch.empty_like(q), torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(A.bwd_workspace_size(q), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    before = torch.cuda.memory_allocated()
    A.attn_fwd(q, k, v, causal=True, out=o, lse=lse)
    A.attn_bwd(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv, workspace=ws)
    torch.cuda.synchronize()
    assert A.attn_status() == A.ATTN_OK, A.last_error()
    assert torch.cuda.max_memory_allocated() == before
    # the caller's buffers are O(N): inputs, outputs and the workspace are linear in N
    per_row = (q.numel() * 2 * 4 + o.numel() * 2 * 4 + lse.numel() * 4 + ws.numel()) / (q.shape[0] * q.shape[1] * N)
    assert per_row < 64 * 2 * 8 + 4 + 64 * 4 + 16  # bytes per (b, h, row): no N-sized factor


def test_one_fused_kernel_per_forward_three_per_backward(A):
    from torch.profiler import ProfilerActivity, profile
    q, k, v, do = _inputs(2048)
    o, lse = A.attn_fwd(q, k, v, causal=True)
    A.attn_bwd(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        o, lse = A.attn_fwd(q, k, v, causal=True)
        torch.cuda.synchronize()
    fwd = [e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA]
    if not fwd:
        pytest.skip("the profiler recorded no CUDA activity on this machine")
    fwd_kernels = [n for n in fwd if "kernel" in n]
    assert len(fwd_kernels) == 1 and "fwd_tc_kernel" in fwd_kernels[0], fwd
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(A.bwd_workspace_size(q), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        A.attn_bwd(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv, workspace=ws)
        torch.cuda.synchronize()
    bwd = [e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA and "kernel" in e.name]
    assert len(bwd) == 3, bwd
    assert "bwd_prepass_kernel" in bwd[0] and "bwd_tc64_kernel" in bwd[1] and "bwd_dq_finalize_kernel" in bwd[2], bwd
