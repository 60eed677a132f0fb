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


def _launched(A, call):
    """Run `call` and return the names of the kernels the library launched for it, from the
    library's own launch log (counted on the host as each launch is issued)."""
    before = A.launch_count()
    call()
    torch.cuda.synchronize()
    assert A.attn_status() == A.ATTN_OK, A.last_error()
    n = A.launch_count() - before
    assert 0 <= n <= 16, n
    return A.launch_names(n)


@pytest.mark.parametrize("d", [64, 128])
def test_one_fused_kernel_per_forward_three_per_backward(A, d):
    q, k, v, do = _inputs(2048, d=d)
    o, lse = torch.empty_like(q), torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(A.bwd_workspace_size(q), dtype=torch.uint8, device="cuda")
    fwd = _launched(A, lambda: A.attn_fwd(q, k, v, causal=True, out=o, lse=lse))
    assert len(fwd) == 1 and "fwd_tc_kernel" in fwd[0], fwd
    bwd = _launched(A, lambda: A.attn_bwd(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv, workspace=ws))
    main = "bwd_tc64_kernel" if d == 64 else "bwd_tc_kernel"
    assert len(bwd) == 3, bwd
    assert "bwd_prepass_kernel" in bwd[0] and main in bwd[1] and "bwd_dq_finalize_kernel" in bwd[2], bwd


def test_launch_counts_of_the_other_entry_points(A):
    q, k, v, do = _inputs(1024, d=128)
    o, lse = A.attn_fwd(q, k, v, causal=True)
    det = _launched(A, lambda: A.attn_bwd_deterministic(q, k, v, o, lse, do, causal=True))
    assert len(det) == 3 and "bwd_dq_kernel" in det[2], det
    q1 = q[:, :, -8:].contiguous()
    dec = _launched(A, lambda: A.attn_decode(q1, k, v, causal=True))
    assert len(dec) == 2 and "decode_tc_kernel" in dec[0] and "decode_combine_kernel" in dec[1], dec
    f32 = [t.float() for t in (q, k, v)]
    simt = _launched(A, lambda: A.attn_fwd(*f32, causal=True))
    assert len(simt) == 1 and "fwd_simt_kernel" in simt[0], simt
