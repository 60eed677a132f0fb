"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Small cases are compared element by element; they span several 128-row tiles
and a ragged tail. Full-size workloads run in the launch configuration the
benchmark times and are checked on sampled rows the oracle computes one by
one (and, for the backward, on whole sampled heads).
"""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import ref
from parity_util import (assert_close_bf16, assert_close_f32, assert_grad, assert_lse, assert_masked_rows_zero,
                         padded_mask, storage_of, stored_forward, to64)

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


def _oracle_mask(mask):
    return None if mask is None else to64(mask)


def _run_fwd(A, inp, causal, scale):
    q, k, v, mask = (_dev(inp.get(n)) for n in ("q", "k", "v", "mask"))
    o, lse = A.attn_fwd(q, k, v, scale=scale, causal=causal, mask=mask)
    torch.cuda.synchronize()
    assert A.attn_status() == A.ATTN_OK, A.last_error()
    return o, lse


def _run_bwd(A, inp, causal, scale, o, lse):
    q, k, v, mask, do = (_dev(inp.get(n)) for n in ("q", "k", "v", "mask", "do"))
    dq, dk, dv = A.attn_bwd(q, k, v, o, lse, do, scale=scale, causal=causal, mask=mask)
    torch.cuda.synchronize()
    assert A.attn_status() == A.ATTN_OK, A.last_error()
    return dq, dk, dv


def _check_fwd(o, lse, inp, causal, scale, f32=False):
    O, L = ref.attention_forward(to64(inp["q"]), to64(inp["k"]), to64(inp["v"]), scale, causal,
                                 _oracle_mask(inp.get("mask")))
    if f32:
        assert_close_f32("O", o, O)
        assert_lse(lse, L, atol=1e-4)
    else:
        assert_close_bf16("O", o, O)
        assert_lse(lse, L)
    assert_masked_rows_zero(o, L)
    return O, L


def _check_bwd(grads, inp, causal, scale):
    """dQ, dK, dV against the oracle whose D comes from its own stored (bf16 / half) O."""
    args = (to64(inp["q"]), to64(inp["k"]), to64(inp["v"]), to64(inp["do"]), scale, causal,
            _oracle_mask(inp.get("mask")))
    stored = ref.attention_backward(*args, o_storage=storage_of(inp["q"].dtype))
    pure = ref.attention_backward(*args)
    return {name: assert_grad(name, g, stored[i], pure[i]) for i, (name, g) in enumerate(zip(("dQ", "dK", "dV"), grads))}


def _bwd_from_oracle_outputs(A, inp, causal, scale):
    """The backward run on the O and LSE the oracle saves (O rounded to the input dtype,
    LSE in fp32): it then computes exactly the function the stored-output oracle defines,
    and every difference is the kernel's own rounding."""
    o, lse = stored_forward(inp, causal, scale)
    return _run_bwd(A, inp, causal, scale, o, lse)


# --------------------------------------------------------------- small cases
@pytest.mark.parametrize("idx", [1])
def test_fp32_workload_full_size(A, idx):
    w = W.WORKLOADS[idx]
    inp = W.make_inputs(w)
    o, lse = _run_fwd(A, inp, w.causal, w.scale)
    _check_fwd(o, lse, inp, w.causal, w.scale, f32=True)


@pytest.mark.parametrize("idx,shape", [
    (2, (2, 3, 300, 64)),
    (3, (1, 2, 1000, 128)),
    (4, (2, 2, 520, 128)),
    (5, (1, 2, 777, 128)),
])
def test_reduced_workloads(A, idx, shape):
    w = W.WORKLOADS[idx]
    inp = W.make_inputs(w, with_grad=w.backward, shape=shape)
    o, lse = _run_fwd(A, inp, w.causal, w.scale)
    _check_fwd(o, lse, inp, w.causal, w.scale)
    if w.backward:
        _check_bwd(_bwd_from_oracle_outputs(A, inp, w.causal, w.scale), inp, w.causal, w.scale)
        # and chained on the kernel's own forward outputs, against the same oracle
        _check_bwd(_run_bwd(A, inp, w.causal, w.scale, o, lse), inp, w.causal, w.scale)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 2, 127, 128, 129, 255, 257])
@pytest.mark.parametrize("causal", [False, True])
def test_edge_lengths(A, d, N, causal):
    inp = {n: W.random_tensor((1, 2, N, d), 100 + i, torch.bfloat16) for i, n in enumerate(("q", "k", "v", "do"))}
    scale = 1 / math.sqrt(d)
    o, lse = _run_fwd(A, inp, causal, scale)
    _check_fwd(o, lse, inp, causal, scale)
    _check_bwd(_bwd_from_oracle_outputs(A, inp, causal, scale), inp, causal, scale)


@pytest.mark.parametrize("d", [64, 128])
def test_fp32_edge_lengths(A, d):
    for N in (1, 33, 200):
        inp = {n: W.random_tensor((2, 1, N, d), 200 + i) for i, n in enumerate(("q", "k", "v"))}
        for causal in (False, True):
            o, lse = _run_fwd(A, inp, causal, 0.1)
            _check_fwd(o, lse, inp, causal, 0.1, f32=True)


@pytest.mark.parametrize("causal", [True, False])
def test_backward_several_units_per_cta(A, causal):
    # 2 x 12 heads x 8 key tiles = 192 units: more than one CTA per SM's worth, so
    # persistent CTAs carry barrier phases, buffers and accumulators across units
    B, H, N, d = 2, 12, 1024, 64
    inp = {n: W.random_tensor((B, H, N, d), 800 + i, torch.bfloat16) for i, n in enumerate(("q", "k", "v", "do"))}
    scale = 1 / math.sqrt(d)
    o, lse = _run_fwd(A, inp, causal, scale)
    _check_fwd(o, lse, inp, causal, scale)
    _check_bwd(_bwd_from_oracle_outputs(A, inp, causal, scale), inp, causal, scale)


def test_bnhd_strided_layout(A):
    B, H, N, d = 2, 3, 333, 128
    base = {n: W.random_tensor((B, N, H, d), 300 + i, torch.bfloat16) for i, n in enumerate(("q", "k", "v", "do"))}
    inp = {n: t.transpose(1, 2) for n, t in base.items()}  # [B, H, N, d] views, n stride = H d
    q, k, v, do = (base[n].to("cuda").transpose(1, 2) for n in ("q", "k", "v", "do"))
    o = torch.empty((B, N, H, d), dtype=torch.bfloat16, device="cuda").transpose(1, 2)
    o, lse = A.attn_fwd(q, k, v, causal=True, out=o)
    torch.cuda.synchronize()
    _check_fwd(o, lse, inp, True, 1 / math.sqrt(d))
    o_s, lse_s = stored_forward(inp, True, 1 / math.sqrt(d))
    o.copy_(o_s)  # the oracle's saved O, in the same strided layout
    grads = A.attn_bwd(q, k, v, o, lse_s, do, causal=True)
    torch.cuda.synchronize()
    _check_bwd(grads, inp, True, 1 / math.sqrt(d))


@pytest.mark.parametrize("per_head", [False, True])
def test_additive_mask_with_masked_rows(A, per_head):
    B, H, N, d = 2, 2, 300, 64
    inp = {n: W.random_tensor((B, H, N, d), 400 + i, torch.bfloat16) for i, n in enumerate(("q", "k", "v", "do"))}
    g = torch.Generator().manual_seed(7)
    mask = torch.randn(B, H if per_head else 1, N, N, generator=g) * 2
    mask[torch.rand(mask.shape, generator=g) < 0.2] = float("-inf")
    mask[:, :, 17, :] = float("-inf")  # fully masked rows
    mask[:, :, 250, :] = float("-inf")
    inp["mask"] = mask.to(torch.bfloat16)
    for causal in (False, True):
        o, lse = _run_fwd(A, inp, causal, 0.125)
        _, L = _check_fwd(o, lse, inp, causal, 0.125)
        assert np.isneginf(L[:, :, 17]).all()
        _check_bwd(_bwd_from_oracle_outputs(A, inp, causal, 0.125), inp, causal, 0.125)


def test_all_rows_masked(A):
    inp = {n: W.random_tensor((1, 1, 130, 64), 500 + i, torch.bfloat16) for i, n in enumerate(("q", "k", "v", "do"))}
    inp["mask"] = torch.full((1, 1, 130, 130), float("-inf"), dtype=torch.bfloat16)
    o, lse = _run_fwd(A, inp, False, 0.125)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    dq, dk, dv = _run_bwd(A, inp, False, 0.125, o, lse)
    assert torch.all(dq == 0) and torch.all(dk == 0) and torch.all(dv == 0)


def test_empty_problem(A):
    q = torch.empty((0, 2, 128, 64), dtype=torch.bfloat16, device="cuda")
    o, lse = A.attn_fwd(q, q, q)
    assert o.shape == q.shape and lse.shape == (0, 2, 128)


def test_deterministic_forward(A):
    inp = {n: W.random_tensor((2, 4, 700, 128), 600 + i, torch.bfloat16) for i, n in enumerate(("q", "k", "v"))}
    o1, l1 = _run_fwd(A, inp, True, 0.09)
    o2, l2 = _run_fwd(A, inp, True, 0.09)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_poisoned_outputs_fully_written(A):
    inp = {n: W.random_tensor((1, 3, 383, 64), 700 + i, torch.bfloat16) for i, n in enumerate(("q", "k", "v"))}
    q, k, v = (_dev(inp[n]) for n in ("q", "k", "v"))
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), device="cuda")
    A.attn_fwd(q, k, v, causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()


# ------------------------------------------------------ full size, sampled
def _sample_rows(N, count, seed):
    r = np.random.default_rng(seed)
    rows = set(r.choice(N, size=min(count, N), replace=False).tolist())
    rows.update({0, N - 1, min(N - 1, 127), min(N - 1, 128)})
    return np.array(sorted(rows))


@pytest.mark.parametrize("idx", [2, 3, 4, 5])
def test_full_size_forward_sampled(A, idx):
    w = W.WORKLOADS[idx]
    inp = W.make_inputs(w, with_grad=False)
    o, lse = _run_fwd(A, inp, w.causal, w.scale)
    heads = [(0, 0), (w.B - 1, w.H - 1), (w.B // 2, w.H // 2)]
    for b, h in heads:
        rows = _sample_rows(w.N, 48, 1000 * b + h)
        if w.mask:
            rows = np.union1d(rows, W.masked_rows(w, b).numpy()[:4])
        maskh = None if inp.get("mask") is None else to64(inp["mask"][b, 0])
        O, L = ref.forward_head(to64(inp["q"][b, h]), to64(inp["k"][b, h]), to64(inp["v"][b, h]), w.scale,
                                w.causal, maskh, rows=rows)
        assert_close_bf16(f"O[{b},{h}]", o[b, h, rows], O)
        assert_lse(lse[b, h, rows], L)
        assert_masked_rows_zero(o[b, h, rows], L)


@pytest.mark.parametrize("idx", [2, 4, 5])
def test_full_size_backward_whole_head(A, idx):
    """The full-size backward in the benchmark's launch configuration, one whole head compared
    element by element: first with that head's saved O and LSE taken from the oracle (the
    function the stored-output oracle defines), then chained on the kernel forward's own O and
    LSE, against the same oracle."""
    w = W.WORKLOADS[idx]
    inp = W.make_inputs(w)
    o, lse = _run_fwd(A, inp, w.causal, w.scale)
    b, h = w.B - 1, w.H // 2
    maskh = None if inp.get("mask") is None else to64(inp["mask"][b, 0])
    hargs = (to64(inp["q"][b, h]), to64(inp["k"][b, h]), to64(inp["v"][b, h]), to64(inp["do"][b, h]), w.scale,
             w.causal, maskh)
    stored = ref.backward_head(*hargs, o_storage="bf16")
    pure = ref.backward_head(*hargs)
    chained = _run_bwd(A, inp, w.causal, w.scale, o, lse)
    chained = [g[b, h].cpu() for g in chained]
    O, L = ref.forward_head(*hargs[:3], w.scale, w.causal, maskh)
    o[b, h] = torch.from_numpy(ref.round_bf16(O)).to(o.dtype).to(o.device)
    lse[b, h] = torch.from_numpy(L).to(torch.float32).to(lse.device)
    fed = _run_bwd(A, inp, w.causal, w.scale, o, lse)
    for t in fed:
        assert torch.isfinite(t).all()
    for label, grads in (("oracle-saved O, LSE", [g[b, h] for g in fed]), ("chained", chained)):
        for i, (name, g) in enumerate(zip(("dQ", "dK", "dV"), grads)):
            e = assert_grad(f"{label} {name}", g, stored[i], pure[i])
            print(f"[{w.name} b={b} h={h}] {label} {name}: stored max-abs {e['stored'][0]:.3e} rel-L2 "
                  f"{e['stored'][1]:.3e}; pure max-abs {e['pure'][0]:.3e} rel-L2 {e['pure'][1]:.3e}")


# ------------------------------------------------------------- IEEE half
@pytest.mark.parametrize("idx,shape", [
    (2, (2, 3, 300, 64)),
    (3, (1, 2, 1000, 128)),
    (4, (2, 2, 520, 128)),
    (5, (1, 2, 777, 128)),
])
def test_fp16_reduced_workloads(A, idx, shape):
    w = W.with_dtype(W.WORKLOADS[idx], "f16")
    inp = W.make_inputs(w, with_grad=True, shape=shape)
    o, lse = _run_fwd(A, inp, w.causal, w.scale)
    assert o.dtype == torch.float16
    _check_fwd(o, lse, inp, w.causal, w.scale)
    _check_bwd(_bwd_from_oracle_outputs(A, inp, w.causal, w.scale), inp, w.causal, w.scale)
    _check_bwd(_run_bwd(A, inp, w.causal, w.scale, o, lse), inp, w.causal, w.scale)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 129, 257])
@pytest.mark.parametrize("causal", [False, True])
def test_fp16_edge_lengths(A, d, N, causal):
    inp = {n: W.random_tensor((1, 2, N, d), 150 + i, torch.float16) for i, n in enumerate(("q", "k", "v", "do"))}
    scale = 1 / math.sqrt(d)
    o, lse = _run_fwd(A, inp, causal, scale)
    _check_fwd(o, lse, inp, causal, scale)
    _check_bwd(_bwd_from_oracle_outputs(A, inp, causal, scale), inp, causal, scale)


def test_fp16_additive_mask(A):
    B, H, N, d = 2, 2, 300, 64
    inp = {n: W.random_tensor((B, H, N, d), 450 + i, torch.float16) for i, n in enumerate(("q", "k", "v", "do"))}
    g = torch.Generator().manual_seed(8)
    mask = torch.randn(B, 1, N, N, generator=g) * 2
    mask[torch.rand(mask.shape, generator=g) < 0.2] = float("-inf")
    mask[:, :, 33, :] = float("-inf")
    inp["mask"] = mask.to(torch.float16)
    for causal in (False, True):
        o, lse = _run_fwd(A, inp, causal, 0.125)
        _check_fwd(o, lse, inp, causal, 0.125)
        _check_bwd(_bwd_from_oracle_outputs(A, inp, causal, 0.125), inp, causal, 0.125)


def test_fp16_benchmark_shape_sampled(A):
    w = W.F16_WORKLOADS[6]
    inp = W.make_inputs(w)
    o, lse = _run_fwd(A, inp, w.causal, w.scale)
    dq, dk, dv = _run_bwd(A, inp, w.causal, w.scale, o, lse)
    b, h = w.B - 1, w.H // 2
    rows = _sample_rows(w.N, 64, 99)
    O, L = ref.forward_head(to64(inp["q"][b, h]), to64(inp["k"][b, h]), to64(inp["v"][b, h]), w.scale, w.causal,
                            None, rows=rows)
    assert_close_bf16("O", o[b, h, rows], O)
    assert_lse(lse[b, h, rows], L)
    hargs = (to64(inp["q"][b, h]), to64(inp["k"][b, h]), to64(inp["v"][b, h]), to64(inp["do"][b, h]), w.scale,
             w.causal, None)
    pure = ref.backward_head(*hargs, q_rows=rows, k_rows=rows)
    stored = ref.backward_head(*hargs, q_rows=rows, k_rows=rows, o_storage="f16")
    for i, (name, g) in enumerate((("dQ", dq), ("dK", dk), ("dV", dv))):
        assert_grad(name, g[b, h, rows], stored[i], pure[i])
