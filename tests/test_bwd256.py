"""The head-dim-256 backward (its own tensor-core kernel: each CTA owns a 128-key tile and one
half of the head dimension of dK, dV and dQ, recomputing the scores over the whole head
dimension) against the fp64 stored-output oracle, with the same bounds as the other head dims."""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import ref
from parity_util import assert_grad, padded_mask, storage_of, stored_forward, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attn_fwd_03_gb300 as m
    return m


def _inputs(shape, seed, dtype=torch.bfloat16, mult=1.0):
    t = {n: W.random_tensor(shape, seed + i, torch.float32) for i, n in enumerate(("q", "k", "v", "do"))}
    t["q"], t["k"] = t["q"] * mult, t["k"] * mult
    return {n: x.to(dtype) for n, x in t.items()}


def _dev_mask(mask):
    if mask is None:
        return None
    return padded_mask(mask, device="cuda") if mask.shape[-1] % 8 else mask.cuda()


def _check(A, inp, causal, scale, mask=None, chained=False):
    """Backward on the oracle's saved O and LSE (and, with chained=True, also on the kernel
    forward's own), against the stored-output oracle."""
    if mask is not None:
        inp = dict(inp, mask=mask)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    md = _dev_mask(mask)
    args = (to64(inp["q"]), to64(inp["k"]), to64(inp["v"]), to64(inp["do"]), scale, causal,
            None if mask is None else to64(mask))
    stored = ref.attention_backward(*args, o_storage=storage_of(inp["q"].dtype))
    pure = ref.attention_backward(*args)
    saved = [stored_forward(inp, causal, scale)]
    if chained:
        saved.append(A.attn_fwd(q, k, v, scale=scale, causal=causal, mask=md))
    for o, lse in saved:
        grads = A.attn_bwd(q, k, v, o, lse, do, scale=scale, causal=causal, mask=md)
        torch.cuda.synchronize()
        assert A.attn_status() == A.ATTN_OK, A.last_error()
        for i, (name, g) in enumerate(zip(("dQ", "dK", "dV"), grads)):
            assert_grad(name, g, stored[i], pure[i])
    return grads


@pytest.mark.parametrize("N", [1, 2, 63, 64, 65, 127, 128, 129, 257])
@pytest.mark.parametrize("causal", [False, True])
def test_edge_lengths(A, N, causal):
    _check(A, _inputs((1, 2, N, 256), 5000 + N), causal, 1 / 16)


@pytest.mark.parametrize("causal", [False, True])
def test_several_heads_and_key_tiles(A, causal):
    # 2 x 3 heads x 4 key tiles x 2 head-dim halves = 48 CTAs, each over several query tiles
    _check(A, _inputs((2, 3, 500, 256), 5100), causal, 1 / 16, chained=True)


def test_large_scores(A):
    # scores of std ~30 (Q and K times sqrt 30): sharply peaked rows, where dS cancels
    _check(A, _inputs((1, 2, 600, 256), 5200, mult=math.sqrt(30.0)), True, 1 / 16, chained=True)


@pytest.mark.parametrize("per_head", [False, True])
def test_additive_mask_with_masked_rows(A, per_head):
    B, H, N = 2, 2, 300
    g = torch.Generator().manual_seed(27)
    mask = torch.randn(B, H if per_head else 1, N, N, generator=g) * 2
    mask[torch.rand(mask.shape, generator=g) < 0.2] = float("-inf")
    mask[:, :, 11, :] = float("-inf")  # fully masked rows
    mask[:, :, 290, :] = float("-inf")
    inp = _inputs((B, H, N, 256), 5300)
    for causal in (False, True):
        dq, dk, dv = _check(A, inp, causal, 0.07, mask=mask.to(torch.bfloat16))
        assert torch.all(dq[:, :, 11] == 0) and torch.all(dq[:, :, 290] == 0)


def test_fp16(A):
    _check(A, _inputs((1, 2, 333, 256), 5400, dtype=torch.float16), True, 1 / 16, chained=True)


def test_strided_layout(A):
    base = _inputs((2, 200, 3, 256), 5500)  # stored [B, N, H, d]
    inp = {n: t.transpose(1, 2) for n, t in base.items()}
    q, k, v, do = (base[n].cuda().transpose(1, 2) for n in ("q", "k", "v", "do"))
    o_s, lse = stored_forward(inp, True, 1 / 16)
    o = torch.empty((2, 200, 3, 256), dtype=torch.bfloat16, device="cuda").transpose(1, 2)
    o.copy_(o_s)
    grads = [torch.empty((2, 200, 3, 256), dtype=torch.bfloat16, device="cuda").transpose(1, 2) for _ in range(3)]
    A.attn_bwd(q, k, v, o, lse, do, scale=1 / 16, causal=True, dq=grads[0], dk=grads[1], dv=grads[2])
    torch.cuda.synchronize()
    assert A.attn_status() == A.ATTN_OK, A.last_error()
    args = tuple(to64(inp[n]) for n in ("q", "k", "v", "do")) + (1 / 16, True, None)
    stored = ref.attention_backward(*args, o_storage="bf16")
    for i, (name, g) in enumerate(zip(("dQ", "dK", "dV"), grads)):
        assert_grad(name, g, stored[i])


def test_dk_dv_identical_across_calls(A):
    """dK and dV of a key tile are summed in one CTA in a fixed order, so repeated calls give the
    same bits (dQ's reductions from different CTAs may land in any order)."""
    inp = {n: t.cuda() for n, t in _inputs((1, 3, 700, 256), 5700).items()}
    o, lse = A.attn_fwd(inp["q"], inp["k"], inp["v"], causal=True)
    first = A.attn_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], causal=True)
    for _ in range(3):
        again = A.attn_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], causal=True)
        torch.cuda.synchronize()
        assert A.attn_status() == A.ATTN_OK, A.last_error()
        assert torch.equal(first[1], again[1]) and torch.equal(first[2], again[2])
        assert (first[0] - again[0]).abs().max().item() <= 1e-2 * max(1.0, first[0].abs().max().item())


def test_deterministic_entry_rejects_head_dim_256(A):
    inp = {n: t.cuda() for n, t in _inputs((1, 1, 128, 256), 5600).items()}
    o, lse = A.attn_fwd(inp["q"], inp["k"], inp["v"])
    with pytest.raises(A.AttnError) as ei:
        A.attn_bwd_deterministic(inp["q"], inp["k"], inp["v"], o, lse, inp["do"])
    assert ei.value.status == A.ATTN_ERR_UNSUPPORTED


@pytest.mark.parametrize("idx", [7, 8])
def test_full_size_whole_head(A, idx):
    """B=1 H=16 N=8192 d=256 (non-causal and causal) in the benchmark's launch configuration; one
    whole head element by element, fed the oracle's saved O and LSE for that head, then
    chained on the kernel forward."""
    w = W.D256_WORKLOADS[idx]
    inp = W.make_inputs(w, with_grad=True)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = A.attn_fwd(q, k, v, scale=w.scale, causal=w.causal)
    b, h = 0, w.H // 2
    hargs = tuple(to64(inp[n][b, h]) for n in ("q", "k", "v", "do")) + (w.scale, w.causal, None)
    stored = ref.backward_head(*hargs, o_storage="bf16")
    pure = ref.backward_head(*hargs)
    chained = [g[b, h].cpu() for g in A.attn_bwd(q, k, v, o, lse, do, scale=w.scale, causal=w.causal)]
    O, L = ref.forward_head(*hargs[:3], w.scale, w.causal)
    o[b, h] = torch.from_numpy(ref.round_bf16(O)).to(o.dtype).to(o.device)
    lse[b, h] = torch.from_numpy(L).to(torch.float32).to(lse.device)
    fed = A.attn_bwd(q, k, v, o, lse, do, scale=w.scale, causal=w.causal)
    torch.cuda.synchronize()
    assert A.attn_status() == A.ATTN_OK, A.last_error()
    for t in fed:
        assert torch.isfinite(t).all()
    for label, grads in (("oracle-saved O, LSE", [g[b, h] for g in fed]), ("chained", chained)):
        for i, (name, g) in enumerate(zip(("dQ", "dK", "dV"), grads)):
            e = assert_grad(f"{label} {name}", g, stored[i], pure[i])
            print(f"[{w.name} b={b} h={h}] {label} {name}: stored max-abs {e['stored'][0]:.3e} rel-L2 "
                  f"{e['stored'][1]:.3e}")
