"""Split-KV decode (attn_decode) against the fp64 oracle's decode_forward.

nq <= 128 query rows per (b, h) against nk keys; with causal the queries are
the last nq positions. The per-split pass runs on the tensor cores with the
query rows in a zero-padded 128-row tile. Cases cover one and several rows
(up to 128, four softmax warps), key counts that are
and are not multiples of the 64-key blocks, a single key, more query rows
than keys (rows that see no key), both head dims, both 16-bit types and
forced split counts from one range to one range per 64 keys.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import ref
from parity_util import assert_close_bf16, assert_lse, assert_masked_rows_zero, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attn_fwd_03_gb300 as m
    return m


def _case(B, H, nq, nk, d, dtype, seed):
    q = W.random_tensor((B, H, nq, d), seed, dtype)
    k = W.random_tensor((B, H, nk, d), seed + 1, dtype)
    v = W.random_tensor((B, H, nk, d), seed + 2, dtype)
    return q, k, v


def _check(A, q, k, v, causal, num_splits=0):
    scale = 1 / math.sqrt(q.shape[-1])
    o, lse = A.attn_decode(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=causal, num_splits=num_splits)
    torch.cuda.synchronize()
    assert A.attn_status() == A.ATTN_OK, A.last_error()
    O, L = ref.decode_forward(to64(q), to64(k), to64(v), scale, causal)
    assert_close_bf16("O", o, O)
    assert_lse(lse, L)
    assert_masked_rows_zero(o, L)
    return o, lse


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("shape", [
    (2, 3, 1, 1000, 64),
    (1, 4, 4, 4096, 128),
    (2, 2, 16, 777, 128),
    (1, 2, 7, 130, 64),
    (1, 1, 3, 1, 64),
    (1, 2, 16, 8, 128),   # causal: the first 8 rows see no key
    (3, 1, 2, 64, 128),
    (1, 2, 33, 1000, 128),  # two softmax warps
    (1, 1, 128, 300, 64),   # causal: rows beyond the keys see nothing
    (2, 1, 100, 2500, 128),
])
@pytest.mark.parametrize("causal", [False, True])
def test_decode_matches_oracle(A, dtype, shape, causal):
    B, H, nq, nk, d = shape
    q, k, v = _case(B, H, nq, nk, d, dtype, 600 + nq + nk)
    _check(A, q, k, v, causal)


@pytest.mark.parametrize("num_splits", [1, 2, 3, 7, 1000])
def test_decode_forced_split_counts(A, num_splits):
    q, k, v = _case(1, 2, 5, 1500, 128, torch.bfloat16, 700)
    o1, l1 = _check(A, q, k, v, True, num_splits)
    o2, l2 = _check(A, q, k, v, True, 0)
    # different splits only reorder fp32 sums: results agree to bf16 rounding of O
    assert torch.allclose(o1.float(), o2.float(), atol=2e-2, rtol=0)


def test_decode_strided_cache(A):
    # K/V laid out [B, nk, H, d] (a cache), queries [B, nq, H, d], viewed as [B, H, n, d]
    B, H, nq, nk, d = 2, 4, 3, 2000, 64
    kb = W.random_tensor((B, nk, H, d), 710, torch.bfloat16)
    vb = W.random_tensor((B, nk, H, d), 711, torch.bfloat16)
    qb = W.random_tensor((B, nq, H, d), 712, torch.bfloat16)
    k, v, q = (t.cuda().transpose(1, 2) for t in (kb, vb, qb))
    o, lse = A.attn_decode(q, k, v, causal=True)
    torch.cuda.synchronize()
    O, L = ref.decode_forward(to64(qb.transpose(1, 2)), to64(kb.transpose(1, 2)), to64(vb.transpose(1, 2)),
                              1 / math.sqrt(d), True)
    assert_close_bf16("O", o, O)
    assert_lse(lse, L)


def test_decode_long_cache_sampled_heads(A):
    # the decode benchmark shape, B=8 H=32 nq=1 nk=8192 d=128, checked on sampled heads
    B, H, nq, nk, d = 8, 32, 1, 8192, 128
    q, k, v = _case(B, H, nq, nk, d, torch.bfloat16, 720)
    o, lse = A.attn_decode(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert A.attn_status() == A.ATTN_OK, A.last_error()
    for b, h in ((0, 0), (B - 1, H - 1), (3, 17)):
        O, L = ref.decode_forward(to64(q[b:b + 1, h:h + 1]), to64(k[b:b + 1, h:h + 1]), to64(v[b:b + 1, h:h + 1]),
                                  1 / math.sqrt(d), True)
        assert_close_bf16(f"O[{b},{h}]", o[b:b + 1, h:h + 1], O)
        assert_lse(lse[b:b + 1, h:h + 1], L)


@pytest.mark.parametrize("nq", [8, 16])
def test_decode_benchmark_shape_tensor_core_pass(A, nq):
    # B=8 H=32 nk=8192 d=128 with 8 and 16 rows: the tensor-core split pass at full size
    B, H, nk, d = 8, 32, 8192, 128
    q, k, v = _case(B, H, nq, nk, d, torch.bfloat16, 730 + nq)
    o, lse = A.attn_decode(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert A.attn_status() == A.ATTN_OK, A.last_error()
    for b, h in ((0, 0), (B - 1, H - 1), (5, 9)):
        O, L = ref.decode_forward(to64(q[b:b + 1, h:h + 1]), to64(k[b:b + 1, h:h + 1]), to64(v[b:b + 1, h:h + 1]),
                                  1 / math.sqrt(d), True)
        assert_close_bf16(f"O[{b},{h}]", o[b:b + 1, h:h + 1], O)
        assert_lse(lse[b:b + 1, h:h + 1], L)
