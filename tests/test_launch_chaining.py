"""Back-to-back calls on one stream with no synchronisation in between.

Consecutive kernels are launched with programmatic stream serialization, so a kernel may
start while the one before it is finishing; each waits for its predecessor before touching
memory. These tests reuse O, LSE and the backward workspace across calls. A kernel that
wrote a buffer its predecessor was still reading, or read one it had not finished writing,
would change the results against the same calls run one at a time.
"""
import pytest
import torch

import workloads as W
from parity_util import assert_close_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attn_fwd_03_gb300 as m
    return m


def _inputs(shape, seed, dtype=torch.bfloat16):
    return [W.random_tensor(shape, seed + i, dtype).cuda() for i in range(4)]  # q, k, v, dO


def _alone(A, q, k, v, do, causal):
    o, lse = A.attn_fwd(q, k, v, causal=causal)
    dq, dk, dv = A.attn_bwd(q, k, v, o, lse, do, causal=causal)
    torch.cuda.synchronize()
    assert A.attn_status() == A.ATTN_OK, A.last_error()
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_chained_calls_reusing_buffers(A, d, causal):
    shape = (2, 8, 1024, d)
    first, second = _inputs(shape, 3100), _inputs(shape, 3200)
    want1, want2 = _alone(A, *first, causal), _alone(A, *second, causal)

    # one stream, no synchronisation: the second forward overwrites the O and LSE the first
    # backward reads, and the second backward zeroes the workspace the first one finalises from
    o = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(shape[:3], dtype=torch.float32, device="cuda")
    ws = torch.empty(A.bwd_workspace_size(first[0]), dtype=torch.uint8, device="cuda")
    grads = [[torch.empty(shape, dtype=torch.bfloat16, device="cuda") for _ in range(3)] for _ in range(2)]
    saved = []
    for (q, k, v, do), g in zip((first, second), grads):
        A.attn_fwd(q, k, v, causal=causal, out=o, lse=lse)
        A.attn_bwd(q, k, v, o, lse, do, causal=causal, dq=g[0], dk=g[1], dv=g[2], workspace=ws)
        saved.append((o.clone(), lse.clone()))  # a copy kernel on the same stream, also chained
    torch.cuda.synchronize()
    assert A.attn_status() == A.ATTN_OK, A.last_error()

    for (o_got, lse_got), g, want in zip(saved, grads, (want1, want2)):
        assert torch.equal(o_got, want[0]) and torch.equal(lse_got, want[1])
        assert torch.equal(g[1], want[3]) and torch.equal(g[2], want[4])  # dK, dV: fixed order
        assert_close_bf16("dQ", g[0], want[2].double().cpu().numpy(), relative_max=True)


def test_chained_deterministic_backward_and_decode(A):
    shape = (2, 4, 768, 64)
    q, k, v, do = _inputs(shape, 3300)
    o, lse = A.attn_fwd(q, k, v, causal=True)
    want = A.attn_bwd_deterministic(q, k, v, o, lse, do, causal=True)
    qd = q[:, :, -8:].contiguous()
    od, lsed = A.attn_decode(qd, k, v, causal=True)
    torch.cuda.synchronize()
    assert A.attn_status() == A.ATTN_OK, A.last_error()

    ws = torch.empty(A.bwd_workspace_size(q), dtype=torch.uint8, device="cuda")
    got = [torch.empty_like(q) for _ in range(3)]
    for _ in range(3):  # repeated without synchronisation, sharing the workspace
        A.attn_bwd_deterministic(q, k, v, o, lse, do, causal=True, dq=got[0], dk=got[1], dv=got[2],
                                 workspace=ws)
        od2, lsed2 = A.attn_decode(qd, k, v, causal=True)
    torch.cuda.synchronize()
    assert A.attn_status() == A.ATTN_OK, A.last_error()
    for a, b in zip(got, want):
        assert torch.equal(a, b)
    assert torch.equal(od2, od) and torch.equal(lsed2, lsed)
