"""Failure detection without a GPU fault.

The forward's load warp is told (through a test hook of the C ABI) to stop
after one key/value tile, so the MMA and softmax warps' bounded waits run
out. The kernel must record ATTN_ERR_TIMEOUT in the device error word and
return; attn_status() reports it once and clears it, and the context stays
usable: the next call computes the right answer. No trap, no bad address,
no endless loop is involved.
"""
import math

import pytest
import torch

import workloads as W
from oracle import ref
from parity_util import assert_close_bf16, assert_lse, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attn_fwd_03_gb300 as m
    return m


def test_stalled_producer_reports_timeout_and_context_survives(A):
    B, H, N, d = 1, 2, 1024, 64
    t = {n: W.random_tensor((B, H, N, d), 950 + i, torch.bfloat16) for i, n in enumerate(("q", "k", "v"))}
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    assert A.attn_status() == A.ATTN_OK
    A.set_wait_timeout_ns(100_000_000)  # 0.1 s per wait
    A.debug_set_producer_stall(1)
    try:
        A.attn_fwd(q, k, v, causal=False)
        torch.cuda.synchronize()  # the kernel returns on its own
        assert A.attn_status() == A.ATTN_ERR_TIMEOUT
        assert "wait" in A.last_error()
        assert A.attn_status() == A.ATTN_OK  # reported once, then cleared
    finally:
        A.debug_set_producer_stall(0)
        A.set_wait_timeout_ns(2_000_000_000)
    o, lse = A.attn_fwd(q, k, v, causal=False)
    torch.cuda.synchronize()
    assert A.attn_status() == A.ATTN_OK
    O, L = ref.attention_forward(to64(t["q"]), to64(t["k"]), to64(t["v"]), 1 / math.sqrt(d), False)
    assert_close_bf16("O", o, O)
    assert_lse(lse, L)
