"""The head-dim-256 forward (its own tensor-core kernel: one query tile per CTA,
K and V streamed through 16 KB slots) against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import ref
from parity_util import assert_close_bf16, assert_lse, assert_masked_rows_zero, padded_mask, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attn_fwd_03_gb300 as m
    return m


def _inputs(shape, seed, dtype=torch.bfloat16, mult=1.0):
    t = {n: W.random_tensor(shape, seed + i, torch.float32) for i, n in enumerate(("q", "k", "v"))}
    t["q"], t["k"] = t["q"] * mult, t["k"] * mult
    return {n: x.to(dtype) for n, x in t.items()}


def _run_check(A, inp, causal, scale, mask=None):
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    mdev = None if mask is None else (padded_mask(mask, device="cuda") if mask.shape[-1] % 8 else mask.cuda())
    o, lse = A.attn_fwd(q, k, v, scale=scale, causal=causal, mask=mdev)
    torch.cuda.synchronize()
    assert A.attn_status() == A.ATTN_OK, A.last_error()
    O, L = ref.attention_forward(to64(inp["q"]), to64(inp["k"]), to64(inp["v"]), scale, causal,
                                 None if mask is None else to64(mask))
    assert_close_bf16("O", o, O)
    assert_lse(lse, L)
    assert_masked_rows_zero(o, L)
    return o, lse, L


@pytest.mark.parametrize("N", [1, 2, 127, 128, 129, 255, 257, 700])
@pytest.mark.parametrize("causal", [False, True])
def test_edge_lengths(A, N, causal):
    _run_check(A, _inputs((1, 2, N, 256), 3000 + N), causal, 1 / 16)


@pytest.mark.parametrize("causal", [False, True])
def test_several_units_per_cta(A, causal):
    # 2 x 12 heads x 8 query tiles = 192 units: persistent CTAs carry the ring, the
    # barrier phases and the O accumulator across units
    _run_check(A, _inputs((2, 12, 1024, 256), 3100), causal, 1 / 16)


def test_large_scores_rescale(A):
    # scores of std ~30 (Q and K times sqrt 30): the running max moves often and O is rescaled
    _run_check(A, _inputs((1, 2, 600, 256), 3200, mult=math.sqrt(30.0)), True, 1 / 16)


@pytest.mark.parametrize("per_head", [False, True])
def test_additive_mask_with_masked_rows(A, per_head):
    B, H, N = 2, 2, 300
    g = torch.Generator().manual_seed(33)
    mask = torch.randn(B, H if per_head else 1, N, N, generator=g) * 2
    mask[torch.rand(mask.shape, generator=g) < 0.2] = float("-inf")
    mask[:, :, 3, :] = float("-inf")
    mask = mask.to(torch.bfloat16)
    for causal in (False, True):
        _, _, L = _run_check(A, _inputs((B, H, N, 256), 3300), causal, 1 / 16, mask=mask)
        assert np.isneginf(L[:, :, 3]).all()


def test_fp16(A):
    _run_check(A, _inputs((2, 2, 333, 256), 3400, dtype=torch.float16), True, 1 / 16)


def test_same_bits_every_call(A):
    inp = _inputs((1, 4, 900, 256), 3500)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o1, l1 = A.attn_fwd(q, k, v, causal=True)
    o2, l2 = A.attn_fwd(q, k, v, causal=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_poisoned_outputs_fully_written(A):
    inp = _inputs((1, 3, 383, 256), 3600)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), device="cuda")
    A.attn_fwd(q, k, v, causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()


@pytest.mark.parametrize("idx", sorted(W.D256_WORKLOADS))
def test_full_size_sampled(A, idx):
    w = W.D256_WORKLOADS[idx]
    inp = W.make_inputs(w, with_grad=False)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = A.attn_fwd(q, k, v, scale=w.scale, causal=w.causal)
    torch.cuda.synchronize()
    assert A.attn_status() == A.ATTN_OK, A.last_error()
    r = np.random.default_rng(400 + idx)
    for b, h in ((0, 0), (w.B - 1, w.H - 1), (0, w.H // 2)):
        rows = np.array(sorted(set(r.choice(w.N, size=48, replace=False).tolist()) | {0, w.N - 1, 127, 128}))
        O, L = ref.forward_head(to64(inp["q"][b, h]), to64(inp["k"][b, h]), to64(inp["v"][b, h]), w.scale, w.causal,
                                None, rows=rows)
        assert_close_bf16(f"O[{b},{h}]", o[b, h, rows], O)
        assert_lse(lse[b, h, rows], L)


def test_bnhd_strided_layout(A):
    # [B, N, H, d] storage seen as [B, H, N, d] views: row stride H * d
    inp = _inputs((2, 3, 200, 256), 3800)
    q, k, v = (x.permute(0, 2, 1, 3).contiguous().cuda().permute(0, 2, 1, 3) for x in (inp["q"], inp["k"], inp["v"]))
    o = torch.empty((2, 200, 3, 256), dtype=torch.bfloat16, device="cuda").permute(0, 2, 1, 3)
    A.attn_fwd(q, k, v, scale=1 / 16, causal=True, out=o)
    torch.cuda.synchronize()
    O, _ = ref.attention_forward(to64(inp["q"]), to64(inp["k"]), to64(inp["v"]), 1 / 16, True)
    assert_close_bf16("O", o, O)
