"""The FP8 (E4M3) forward (head dims 128 and 256) against the fp64 oracle of the
values the codes stand for.

Tolerance, derived from the kernel's arithmetic (written out here, not fitted):
the scores are exact products of E4M3 values summed in fp32, and the softmax
runs in fp32 as in the 16-bit kernels; what is new is that each probability is
rounded to E4M3 before it multiplies V. With p_j = exp(s_j - m) <= 1 for the
row max m, the kernel holds p_j 2^k for some 0 <= k <= 8 (its reference max
sits up to 8 below m in log2 units), so the rounding error of p_j is at most
2^-4 p_j when p_j 2^k is a normal E4M3 value (>= 2^-6) and at most
2^-10 2^-k <= 2^-10 otherwise. O is divided by l, the sum of the unrounded
values, with its largest term p_* swapped for the rounded one: l~ = l + eps_*
(eps_j = p~_j - p_j; the common factor 2^k cancels). Then
    O_kernel - O = (sum_j eps_j v_j - eps_* O) / l~,
so per element, whichever largest term the kernel picked,
    |O_kernel - O| <= (sum_j e_j |v_jd| + e_max |O_d|) / (l - e_max),
    e_j = max(2^-4 p_j, 2^-10 [0 < p_j < 2^-6]),  e_max = max_j e_j,
plus the bf16 rounding of the output (2^-8 relative, with slack for fp32).
LSE comes from the unrounded l and keeps the 1e-3 bound.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import ref
from parity_util import assert_lse, assert_masked_rows_zero, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attn_fwd_03_gb300 as m
    return m


def _inputs(shape, seed, mult=1.0):
    out = {}
    for i, name in enumerate(("q", "k", "v")):
        x = W.random_tensor(shape, seed + i) * (mult if name != "v" else 1.0)
        out[name + "8"], out[name + "_ds"] = W.quantize_e4m3(x)
    return out


def _bound_and_ref(inp, scale, causal, mask, heads=None, rows=None):
    """Oracle O, LSE and the per-element error bound for the heads (b, h) given (all if None)."""
    B, H, N, _ = inp["q8"].shape
    heads = heads or [(b, h) for b in range(B) for h in range(H)]
    res = {}
    for b, h in heads:
        q, k, v = (ref.decode_e4m3(inp[n + "8"][b, h].numpy()) * inp[n + "_ds"] for n in ("q", "k", "v"))
        r = np.arange(N) if rows is None else rows
        maskh = None if mask is None else to64(mask[b if mask.shape[0] > 1 else 0, h if mask.shape[1] > 1 else 0])
        O, L = ref.forward_head(q, k, v, scale, causal, maskh, rows=r)
        s = ref.head_scores(q, k, r, scale, causal, maskh)
        m = s.max(axis=1, keepdims=True)
        empty = np.isneginf(m)
        p = np.where(empty, 0.0, np.exp(s - np.where(empty, 0.0, m)))
        lsum = p.sum(axis=1, keepdims=True)
        e = np.maximum(2.0 ** -4 * p, np.where((p > 0) & (p < 2.0 ** -6), 2.0 ** -10, 0.0))
        emax = e.max(axis=1, keepdims=True) if e.shape[1] else np.zeros_like(lsum)
        low = lsum - emax
        bound = (e @ np.abs(v) + emax * np.abs(O)) / np.where(low > 0, low, 1.0)
        res[(b, h)] = (O, L, bound)
    return res


def _check(o, lse, res, rows=None):
    for (b, h), (O, L, bound) in res.items():
        got = to64(o[b, h] if rows is None else o[b, h, rows])
        err = np.abs(got - O)
        allowed = bound + 2.0 ** -8 * np.abs(O) + 1e-6 * (np.abs(O).max() + 1e-30)
        worst = np.unravel_index(np.argmax(err - allowed), err.shape)
        assert np.all(err <= allowed), (f"O[{b},{h}] error {err[worst]:.3e} > bound {allowed[worst]:.3e} at {worst}")
        assert_lse(lse[b, h] if rows is None else lse[b, h, rows], L)
        assert_masked_rows_zero(got, L)
        # each probability is off by at most 2^-4 of itself, so the errors of a whole head, which
        # are sums of many independent roundings, stay below 2^-4 of O in the L2 norm (a broken
        # packing or layout of P gives errors of the size of O itself)
        if np.linalg.norm(O) > 0:
            assert np.linalg.norm(got - O) <= 2.0 ** -4 * np.linalg.norm(O), f"O[{b},{h}] rel-L2"


def _run(A, inp, causal, scale, mask=None):
    dev = lambda t: t.cuda().view(torch.float8_e4m3fn)  # noqa: E731
    o, lse = A.attn_fwd_fp8(dev(inp["q8"]), dev(inp["k8"]), dev(inp["v8"]), inp["q_ds"], inp["k_ds"], inp["v_ds"],
                            scale=scale, causal=causal, mask=None if mask is None else mask.cuda())
    torch.cuda.synchronize()
    assert A.attn_status() == A.ATTN_OK, A.last_error()
    return o, lse


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("N", [1, 2, 127, 128, 129, 255, 257, 600])
@pytest.mark.parametrize("causal", [False, True])
def test_edge_lengths(A, d, N, causal):
    inp = _inputs((1, 2, N, d), 4000 + N + d)
    o, lse = _run(A, inp, causal, 1 / math.sqrt(d))
    _check(o, lse, _bound_and_ref(inp, 1 / math.sqrt(d), causal, None))


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_several_units_per_cta(A, d, causal):
    inp = _inputs((2, 12, 700, d), 4100)
    o, lse = _run(A, inp, causal, 1 / math.sqrt(d))
    _check(o, lse, _bound_and_ref(inp, 1 / math.sqrt(d), causal, None, heads=[(0, 0), (1, 11), (0, 5)]))


@pytest.mark.parametrize("d", [128, 256])
def test_large_scores_rescale(A, d):
    inp = _inputs((1, 2, 500, d), 4200, mult=math.sqrt(30.0))
    o, lse = _run(A, inp, True, 1 / math.sqrt(d))
    _check(o, lse, _bound_and_ref(inp, 1 / math.sqrt(d), True, None))


@pytest.mark.parametrize("d", [128, 256])
def test_additive_mask_with_masked_rows(A, d):
    B, H, N = 2, 2, 264
    inp = _inputs((B, H, N, d), 4300)
    g = torch.Generator().manual_seed(43)
    mask = torch.randn(B, 1, N, N, generator=g) * 2
    mask[torch.rand(mask.shape, generator=g) < 0.2] = float("-inf")
    mask[:, :, 9, :] = float("-inf")
    mask = mask.to(torch.bfloat16)
    for causal in (False, True):
        o, lse = _run(A, inp, causal, 0.1, mask=mask)
        res = _bound_and_ref(inp, 0.1, causal, mask)
        _check(o, lse, res)
        assert np.isneginf(res[(0, 0)][1][9])


def test_same_bits_every_call(A):
    inp = _inputs((1, 4, 900, 128), 4400)
    a = _run(A, inp, True, 0.09)
    b = _run(A, inp, True, 0.09)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_close_to_the_bf16_forward_of_the_same_values(A):
    # E4M3 values (4 significant bits) are exact in bf16, so the 16-bit kernel, given the
    # decoded codes with the descales folded into the scale (q, k) and the output (v),
    # computes the same attention without rounding P: the two differ by the FP8 bound above
    inp = _inputs((1, 2, 1000, 128), 4500)
    o8, l8 = _run(A, inp, True, 0.09)
    raw = {n: ref.decode_e4m3(inp[n + "8"].numpy()) for n in ("q", "k", "v")}
    vals = {n: torch.from_numpy(x).to(torch.bfloat16) for n, x in raw.items()}
    assert all(np.array_equal(vals[n].double().numpy(), raw[n]) for n in raw)
    o16, l16 = A.attn_fwd(vals["q"].cuda(), vals["k"].cuda(), vals["v"].cuda(),
                          scale=0.09 * inp["q_ds"] * inp["k_ds"], causal=True)
    torch.cuda.synchronize()
    res = _bound_and_ref(inp, 0.09, True, None)
    for (b, h), (O, L, bound) in res.items():
        err = np.abs(to64(o8[b, h]) - inp["v_ds"] * to64(o16[b, h]))
        assert np.all(err <= bound + 2.0 ** -7 * np.abs(O) + 1e-3 * np.abs(O).max())
    assert torch.allclose(l8, l16, atol=1e-3)


def test_poisoned_outputs_fully_written(A):
    inp = _inputs((1, 3, 383, 128), 4600)
    dev = lambda t: t.cuda().view(torch.float8_e4m3fn)  # noqa: E731
    o = torch.full((1, 3, 383, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((1, 3, 383), float("nan"), device="cuda")
    A.attn_fwd_fp8(dev(inp["q8"]), dev(inp["k8"]), dev(inp["v8"]), inp["q_ds"], inp["k_ds"], inp["v_ds"],
                   causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()


@pytest.mark.parametrize("idx", sorted(W.FP8_WORKLOADS))
def test_full_size_sampled(A, idx):
    w = W.FP8_WORKLOADS[idx]
    inp = W.make_fp8_inputs(w)
    o, lse = _run(A, inp, w.causal, w.scale)
    r = np.random.default_rng(500 + idx)
    rows = np.array(sorted(set(r.choice(w.N, size=32, replace=False).tolist()) | {0, w.N - 1, 127, 128}))
    res = _bound_and_ref(inp, w.scale, w.causal, None, heads=[(0, 0), (w.B - 1, w.H - 1)], rows=rows)
    _check(o, lse, res, rows=rows)


def test_bnhd_strided_layout(A):
    inp = _inputs((2, 3, 300, 128), 4700)
    dev = lambda t: t.permute(0, 2, 1, 3).contiguous().cuda().permute(0, 2, 1, 3).view(torch.float8_e4m3fn)  # noqa: E731
    o = torch.empty((2, 300, 3, 128), dtype=torch.bfloat16, device="cuda").permute(0, 2, 1, 3)
    lse = torch.empty((2, 3, 300), dtype=torch.float32, device="cuda")
    A.attn_fwd_fp8(dev(inp["q8"]), dev(inp["k8"]), dev(inp["v8"]), inp["q_ds"], inp["k_ds"], inp["v_ds"],
                   scale=0.1, causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert A.attn_status() == A.ATTN_OK, A.last_error()
    _check(o, lse, _bound_and_ref(inp, 0.1, True, None))
