"""attn_bwd_deterministic: the backward pass whose dQ is summed over key tiles
in a fixed order by a query-stationary kernel. Its gradients are checked
against the fp64 oracle like attn_bwd's, and against themselves bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import ref
from parity_util import assert_close_bf16, assert_grad, padded_mask, storage_of, stored_forward, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attn_fwd_03_gb300 as m
    return m


def _dev(x):
    if x is None:
        return None
    if x.dim() == 4 and x.shape[-1] == x.shape[-2] and x.shape[-1] % 8 != 0:  # a mask: keep rows 16-byte aligned
        return padded_mask(x, device="cuda")
    return x.to("cuda")


def _run(A, inp, causal, scale, entry="attn_bwd_deterministic", saved="oracle"):
    """The backward on the oracle's saved O and LSE (saved="oracle": the function the
    stored-output oracle defines) or on the kernel forward's own (saved="kernel")."""
    q, k, v, mask, do = (_dev(inp.get(n)) for n in ("q", "k", "v", "mask", "do"))
    if saved == "oracle":
        o, lse = stored_forward(inp, causal, scale)
    else:
        o, lse = A.attn_fwd(q, k, v, scale=scale, causal=causal, mask=mask)
    grads = getattr(A, entry)(q, k, v, o, lse, do, scale=scale, causal=causal, mask=mask)
    torch.cuda.synchronize()
    assert A.attn_status() == A.ATTN_OK, A.last_error()
    return grads


def _check(grads, inp, causal, scale):
    mask = inp.get("mask")
    args = (to64(inp["q"]), to64(inp["k"]), to64(inp["v"]), to64(inp["do"]), scale, causal,
            None if mask is None else to64(mask))
    stored = ref.attention_backward(*args, o_storage=storage_of(inp["q"].dtype))
    pure = ref.attention_backward(*args)
    for i, (name, g) in enumerate(zip(("dQ", "dK", "dV"), grads)):
        assert_grad(name, g, stored[i], pure[i])


def _inputs(shape, seed, dtype=torch.bfloat16):
    return {n: W.random_tensor(shape, seed + i, dtype) for i, n in enumerate(("q", "k", "v", "do"))}


@pytest.mark.parametrize("idx,shape", [
    (2, (2, 3, 300, 64)),
    (4, (2, 2, 520, 128)),
    (5, (1, 2, 777, 128)),
])
def test_reduced_workloads(A, idx, shape):
    w = W.WORKLOADS[idx]
    inp = W.make_inputs(w, with_grad=True, shape=shape)
    _check(_run(A, inp, w.causal, w.scale), inp, w.causal, w.scale)
    _check(_run(A, inp, w.causal, w.scale, saved="kernel"), inp, w.causal, w.scale)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 127, 129, 257])
@pytest.mark.parametrize("causal", [False, True])
def test_edge_lengths(A, d, N, causal):
    inp = _inputs((1, 2, N, d), 1500)
    scale = 1 / math.sqrt(d)
    _check(_run(A, inp, causal, scale), inp, causal, scale)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_several_units_per_cta(A, d, causal):
    # 2 x 12 heads x 8 query tiles = 192 units, more than one per SM: persistent CTAs carry
    # barrier phases, tensor-memory buffers and the dQ accumulator across units
    inp = _inputs((2, 12, 1024, d), 1600)
    scale = 1 / math.sqrt(d)
    _check(_run(A, inp, causal, scale), inp, causal, scale)


def test_additive_mask_with_masked_rows(A):
    B, H, N, d = 2, 2, 300, 128
    inp = _inputs((B, H, N, d), 1700)
    g = torch.Generator().manual_seed(17)
    mask = torch.randn(B, H, N, N, generator=g) * 2
    mask[torch.rand(mask.shape, generator=g) < 0.2] = float("-inf")
    mask[:, :, 5, :] = float("-inf")
    mask[:, :, 299, :] = float("-inf")
    inp["mask"] = mask.to(torch.bfloat16)
    for causal in (False, True):
        dq, dk, dv = _run(A, inp, causal, 0.1)
        _check((dq, dk, dv), inp, causal, 0.1)
        assert torch.all(dq[:, :, 5] == 0) and torch.all(dq[:, :, 299] == 0)


def test_fp16(A):
    inp = _inputs((2, 2, 333, 64), 1800, torch.float16)
    _check(_run(A, inp, True, 0.125), inp, True, 0.125)


def test_all_rows_masked(A):
    inp = _inputs((1, 1, 130, 64), 1900)
    inp["mask"] = torch.full((1, 1, 130, 130), float("-inf"), dtype=torch.bfloat16)
    dq, dk, dv = _run(A, inp, False, 0.125)
    assert torch.all(dq == 0) and torch.all(dk == 0) and torch.all(dv == 0)


def test_same_bits_every_call_and_agrees_with_attn_bwd(A):
    inp = _inputs((2, 6, 1000, 64), 2000)
    first = _run(A, inp, True, 0.125)
    other = _inputs((1, 3, 400, 128), 2100)
    _run(A, other, False, 0.09)  # a different problem in between
    again = _run(A, inp, True, 0.125)
    for name, a, b in zip(("dQ", "dK", "dV"), first, again):
        assert torch.equal(a, b), name
    atomic = _run(A, inp, True, 0.125, entry="attn_bwd")
    # dK and dV come from the same kernel; dQ sums the same terms in another order
    assert torch.equal(first[1], atomic[1]) and torch.equal(first[2], atomic[2])
    assert_close_bf16("dQ vs attn_bwd", first[0], atomic[0].double().cpu().numpy(), relative_max=True)


def test_poisoned_dq_fully_written(A):
    inp = _inputs((1, 3, 383, 128), 2200)
    q, k, v, do = (_dev(inp[n]) for n in ("q", "k", "v", "do"))
    o, lse = A.attn_fwd(q, k, v, causal=True)
    dq = torch.full_like(q, float("nan"))
    A.attn_bwd_deterministic(q, k, v, o, lse, do, causal=True, dq=dq)
    torch.cuda.synchronize()
    assert A.attn_status() == A.ATTN_OK, A.last_error()
    assert not torch.isnan(dq).any()


def test_empty_problem(A):
    q = torch.empty((0, 2, 128, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((0, 2, 128), dtype=torch.float32, device="cuda")
    dq, dk, dv = A.attn_bwd_deterministic(q, q, q, q, lse, q)
    assert dq.shape == q.shape


@pytest.mark.parametrize("idx", [2, 4, 5])
def test_full_size_whole_head(A, idx):
    """Full size, one whole head element by element: the head's saved O and LSE from the
    oracle, then chained on the kernel forward's own (see the attn_bwd test of the same name)."""
    w = W.WORKLOADS[idx]
    inp = W.make_inputs(w)
    q, k, v, mask, do = (_dev(inp.get(n)) for n in ("q", "k", "v", "mask", "do"))
    o, lse = A.attn_fwd(q, k, v, scale=w.scale, causal=w.causal, mask=mask)
    b, h = w.B - 1, w.H // 2
    maskh = None if inp.get("mask") is None else to64(inp["mask"][b, 0])
    hargs = (to64(inp["q"][b, h]), to64(inp["k"][b, h]), to64(inp["v"][b, h]), to64(inp["do"][b, h]), w.scale,
             w.causal, maskh)
    stored = ref.backward_head(*hargs, o_storage="bf16")
    pure = ref.backward_head(*hargs)
    chained = A.attn_bwd_deterministic(q, k, v, o, lse, do, scale=w.scale, causal=w.causal, mask=mask)
    chained = [g[b, h].cpu() for g in chained]
    O, L = ref.forward_head(*hargs[:3], w.scale, w.causal, maskh)
    o[b, h] = torch.from_numpy(ref.round_bf16(O)).to(o.dtype).to(o.device)
    lse[b, h] = torch.from_numpy(L).to(torch.float32).to(lse.device)
    fed = A.attn_bwd_deterministic(q, k, v, o, lse, do, scale=w.scale, causal=w.causal, mask=mask)
    torch.cuda.synchronize()
    assert A.attn_status() == A.ATTN_OK, A.last_error()
    for t in fed:
        assert torch.isfinite(t).all()
    for label, grads in (("oracle-saved O, LSE", [g[b, h] for g in fed]), ("chained", chained)):
        for i, (name, g) in enumerate(zip(("dQ", "dK", "dV"), grads)):
            e = assert_grad(f"{label} {name}", g, stored[i], pure[i])
            print(f"[{w.name} b={b} h={h}] deterministic {label} {name}: stored max-abs {e['stored'][0]:.3e} "
                  f"rel-L2 {e['stored'][1]:.3e}; pure max-abs {e['pure'][0]:.3e} rel-L2 {e['pure'][1]:.3e}")


def test_bnhd_strided_layout(A):
    inp = _inputs((2, 300, 3, 64), 2300)  # stored [B, N, H, d]
    view = {n: x.cuda().permute(0, 2, 1, 3) for n, x in inp.items()}
    o, lse = A.attn_fwd(view["q"], view["k"], view["v"], scale=0.125, causal=True)
    grads = [torch.empty((2, 300, 3, 64), dtype=torch.bfloat16, device="cuda").permute(0, 2, 1, 3) for _ in range(3)]
    A.attn_bwd_deterministic(view["q"], view["k"], view["v"], o, lse, view["do"], scale=0.125, causal=True,
                             dq=grads[0], dk=grads[1], dv=grads[2])
    torch.cuda.synchronize()
    assert A.attn_status() == A.ATTN_OK, A.last_error()
    _check(grads, {n: x.permute(0, 2, 1, 3) for n, x in inp.items()}, True, 0.125)
