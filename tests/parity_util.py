"""Comparison helpers shared by the GPU parity tests.

Tolerances (written here once, used by every parity test):
  * bf16 inputs, fp32 accumulation: max-abs error <= 2e-2 and relative-L2
    error <= 5e-3 on O (gradients: the same two numbers, below).
  * fp32 inputs: max-abs <= 1e-4 on O and LSE.
  * LSE: max-abs <= 1e-3 on finite entries; -inf entries (fully masked rows)
    must sit at exactly the same positions, and those rows of O must be 0.
  * Gradients. The backward computes D = rowsum(dO * O) from the O the forward
    stored (bf16 or half), as the method prescribes: it recomputes from the
    stored output and the saved row statistics. The oracle for that method is
    the fp64 gradient with D taken from the oracle's own O rounded to the
    storage dtype (o_storage="bf16" / "f16"). Gradients are held to the same
    two numbers as O against it: rel-L2 <= 5e-3 and max-abs <= 2e-2 *
    max(1, max|ref|). The max-abs bound scales with the largest reference
    value because a bf16 number of magnitude M in [2^e, 2^(e+1)) is only
    representable to half a unit in the last place, 2^(e-8), which exceeds
    2e-2 once M > 5.12 (the large-score workload's dQ reaches ~21); at
    max|ref| <= 1 the bound is the plain 2e-2. The distance to the pure fp64
    gradient (D from the exact O) is returned for reporting, not asserted.
  * IEEE half inputs (an extension; no tolerance is stated for them). Half
    keeps 10 fraction bits against bf16's 7, so every rounding in the path
    (inputs, P, dS, O, dQ/dK/dV) is 8x finer; the bf16 bounds are scaled by
    1/8 and rounded up: max-abs <= 4e-3 and rel-L2 <= 1e-3 (gradients against
    the half-stored oracle, o_storage="f16").
"""
from __future__ import annotations

import numpy as np
import torch

BF16_ATOL = 2e-2
BF16_REL_L2 = 5e-3
F16_ATOL = 4e-3
F16_REL_L2 = 1e-3
F32_ATOL = 1e-4
LSE_ATOL = 1e-3


def to64(t) -> np.ndarray:
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().to("cpu").to(torch.float64).numpy()


def errors(got, want):
    got, want = to64(got), to64(want)
    diff = got - want
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    denom = float(np.linalg.norm(want))
    rel = float(np.linalg.norm(diff)) / denom if denom > 0 else float(np.linalg.norm(diff))
    return max_abs, rel


def _bounds(dtype):
    return (F16_ATOL, F16_REL_L2) if dtype == torch.float16 else (BF16_ATOL, BF16_REL_L2)


def assert_close_bf16(name, got, want, relative_max=False):
    """16-bit outputs: the bf16 bounds, or the half bounds when `got` is half."""
    atol, rtol = _bounds(got.dtype if isinstance(got, torch.Tensor) else None)
    g, w = to64(got), to64(want)
    max_abs, rel = errors(g, w)
    bound = atol * (max(1.0, float(np.max(np.abs(w)))) if (relative_max and w.size) else 1.0)
    assert max_abs <= bound and rel <= rtol, \
        f"{name}: max-abs {max_abs:.3e} (bound {bound:.3e}), rel-L2 {rel:.3e} (bound {rtol:.1e})"
    return max_abs, rel


def assert_close_f32(name, got, want):
    max_abs, rel = errors(got, want)
    assert max_abs <= F32_ATOL, f"{name}: max-abs {max_abs:.3e} > {F32_ATOL:.0e}"
    return max_abs, rel


def assert_lse(got, want, atol=LSE_ATOL):
    g, w = to64(got), to64(want)
    fin_g, fin_w = np.isfinite(g), np.isfinite(w)
    assert np.array_equal(fin_g, fin_w), "LSE: -inf rows differ"
    assert np.all(np.isneginf(g[~fin_g])), "LSE: non-finite entries must be -inf"
    if fin_w.any():
        err = float(np.max(np.abs(g[fin_w] - w[fin_w])))
        assert err <= atol, f"LSE: max-abs {err:.3e} > {atol:.0e}"
        return err
    return 0.0


def assert_masked_rows_zero(o, lse_ref):
    o = to64(o)
    dead = np.isneginf(to64(lse_ref))
    if dead.any():
        assert np.all(o[dead] == 0.0), "fully masked rows of O must be exactly 0"


def assert_grad(name, got, stored, pure=None):
    """Gradient check against the stored-output oracle, with the bounds above.

    Returns {"stored": (max_abs, rel_l2)} and, when `pure` is given, also
    {"pure": (max_abs, rel_l2)}: the distance to the gradient with D from the
    exact O, reported only."""
    atol, rtol = _bounds(got.dtype if isinstance(got, torch.Tensor) else None)
    g, w = to64(got), to64(stored)
    max_abs, rel = errors(g, w)
    bound_abs = atol * max(1.0, float(np.max(np.abs(w))) if w.size else 1.0)
    assert max_abs <= bound_abs and rel <= rtol, \
        f"{name}: max-abs {max_abs:.3e} (bound {bound_abs:.3e}), rel-L2 {rel:.3e} (bound {rtol:.1e})"
    out = {"stored": (max_abs, rel)}
    if pure is not None:
        out["pure"] = errors(g, to64(pure))
    return out


def stored_forward(inp, causal, scale, device="cuda"):
    """The oracle's O rounded to the input dtype (what a forward stores) and its LSE in
    fp32, as device tensors: the saved outputs a backward consumes, from the oracle
    alone. Feeding these to the CUDA backward makes it compute the very function the
    stored-output oracle defines."""
    from oracle import ref
    mask = inp.get("mask")
    O, L = ref.attention_forward(to64(inp["q"]), to64(inp["k"]), to64(inp["v"]), scale, causal,
                                 None if mask is None else to64(mask))
    dt = inp["q"].dtype
    rnd = ref.round_f16 if dt == torch.float16 else ref.round_bf16
    o = torch.from_numpy(rnd(O)).to(dt).to(device)
    lse = torch.from_numpy(L).to(torch.float32).to(device)
    return o, lse


def storage_of(dtype):
    return "f16" if dtype == torch.float16 else "bf16"


def padded_mask(mask: torch.Tensor, device=None) -> torch.Tensor:
    """The same values in storage whose rows are padded to a multiple of 8
    elements (16 bytes), which the TMA-fed kernels require."""
    n = mask.shape[-1]
    npad = (n + 7) // 8 * 8
    store = torch.zeros(*mask.shape[:-1], npad, dtype=mask.dtype, device=device or mask.device)
    store[..., :n] = mask.to(store.device)
    return store[..., :n]
