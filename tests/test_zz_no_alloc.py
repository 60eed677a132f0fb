"""attn_bwd_noalloc: the backward pass for callers that cannot allocate device
memory when they run it (an allocator callback, a plug-in whose host owns all
memory, a fixed memory budget). It uses the library's built-in scratch array
instead of a caller workspace, so its results must match attn_bwd's.

The file name sorts last, so a plain sequential run reaches it after the other
tests; nothing here depends on that order, and each test passes run alone.
"""
import math

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


def _problem(seed, B=2, H=3, N=300, d=64):
    t = {n: W.random_tensor((B, H, N, d), seed + i, torch.bfloat16).cuda() for i, n in enumerate(("q", "k", "v", "do"))}
    return t, 1.0 / math.sqrt(d)


def test_matches_caller_workspace_backward_on_two_calls_in_a_row(A):
    # two different problems back to back: the second call must not see the first one's scratch
    for seed, d, causal in ((1200, 64, True), (1300, 128, False)):
        t, scale = _problem(seed, d=d)
        o, lse = A.attn_fwd(t["q"], t["k"], t["v"], scale=scale, causal=causal)
        ref = A.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], scale=scale, causal=causal)
        got = A.attn_bwd_noalloc(t["q"], t["k"], t["v"], o, lse, t["do"], scale=scale, causal=causal)
        torch.cuda.synchronize()
        assert A.attn_status() == A.ATTN_OK, A.last_error()
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            assert_close_bf16(name, g, r, relative_max=True)
        # dK and dV are reduced in a fixed order: identical bits
        assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])


def test_back_to_back_calls_on_one_stream_without_synchronising(A):
    # three different problems queued on one stream with no synchronisation in between: each
    # call's pre-pass rewrites the shared scratch while the previous call's kernels may still be
    # finishing, so this checks that every call waits for the one before it
    probs = []
    for seed, d, causal, N in ((1400, 64, True, 300), (1500, 128, False, 517), (1600, 64, False, 129)):
        t, scale = _problem(seed, N=N, d=d)
        o, lse = A.attn_fwd(t["q"], t["k"], t["v"], scale=scale, causal=causal)
        want = A.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], scale=scale, causal=causal)
        probs.append((t, scale, causal, o, lse, want))
    torch.cuda.synchronize()
    assert A.attn_status() == A.ATTN_OK, A.last_error()
    got = [A.attn_bwd_noalloc(t["q"], t["k"], t["v"], o, lse, t["do"], scale=scale, causal=causal)
           for t, scale, causal, o, lse, _ in probs]
    torch.cuda.synchronize()
    assert A.attn_status() == A.ATTN_OK, A.last_error()
    for g, (_, _, _, _, _, want) in zip(got, probs):
        for name, a, b in zip(("dQ", "dK", "dV"), g, want):
            assert_close_bf16(name, a, b, relative_max=True)
        assert torch.equal(g[1], want[1]) and torch.equal(g[2], want[2])


def test_rejects_problems_beyond_the_built_in_scratch(A):
    B, H, N, d = 1, 1, 100_000, 128  # needs ~52 MB of scratch, the built-in area holds 40 MiB
    q = torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    with pytest.raises(A.AttnError) as ei:
        A.attn_bwd_noalloc(q, q, q, q, lse, q)
    assert ei.value.status == A.ATTN_ERR_WORKSPACE
    assert "built-in" in str(ei.value)
