"""Comparison helpers shared by the GPU parity tests.

Tolerances (written here once, used by every parity test):
  * bf16 inputs, fp32 accumulation: max-abs error <= 2e-2 and relative-L2
    error <= 5e-3 on O; gradients use the same two numbers, with the max-abs
    bound taken relative to max(1, max |reference|) because a bf16 output of
    magnitude M cannot be closer than its own rounding step (M * 2^-9).
  * fp32 inputs: max-abs <= 1e-4 on O and LSE.
  * LSE: max-abs <= 1e-3 on finite entries; -inf entries (fully masked rows)
    must sit at exactly the same positions, and those rows of O must be 0.
  * Gradients. The backward computes D = rowsum(dO * O) from the O the forward
    stored in bf16, as the method prescribes (the backward recomputes from
    the stored output and statistics). Where dP - D cancels (tiny N, peaked
    P) that storage rounding alone moves dQ and dK by more than 5e-3 of their
    norm, so the bound is derived from it: against the pure fp64 gradient,
        rel-L2  <= 5e-3 + 2 * delta,   max-abs <= 2e-2 * max(1, max|ref|) + 2 * delta_abs,
    where delta / delta_abs are the relative-L2 / max-abs change the oracle
    itself sees when it takes D from its own bf16-rounded O instead of the
    exact one. Both come from the oracle alone; for non-degenerate shapes
    delta is ~1e-3.
  * IEEE half inputs (an extension; no tolerance is stated for them). Half
    keeps 10 fraction bits against bf16's 7, so every rounding in the path
    (inputs, P, dS, O, dQ/dK/dV) is 8x finer; the bf16 bounds are scaled by
    1/8 and rounded up: max-abs <= 4e-3 and rel-L2 <= 1e-3 (gradients: the
    same derived allowance, with delta taken from a half-rounded O).
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


def assert_grad(name, got, pure, stored):
    """Gradient check with the stored-output allowance described above."""
    atol, rtol = _bounds(got.dtype if isinstance(got, torch.Tensor) else None)
    g, w, st = to64(got), to64(pure), to64(stored)
    delta_abs, delta = errors(st, w)
    max_abs, rel = errors(g, w)
    bound_abs = atol * max(1.0, float(np.max(np.abs(w))) if w.size else 1.0) + 2 * delta_abs
    bound_rel = rtol + 2 * delta
    assert max_abs <= bound_abs and rel <= bound_rel, \
        f"{name}: max-abs {max_abs:.3e} (bound {bound_abs:.3e}), rel-L2 {rel:.3e} (bound {bound_rel:.3e})"
    return max_abs, rel


def padded_mask(mask: torch.Tensor, device=None) -> torch.Tensor:
    """The same values in storage whose rows are padded to a multiple of 8
    elements (16 bytes), which the TMA-fed kernels require."""
    n = mask.shape[-1]
    npad = (n + 7) // 8 * 8
    store = torch.zeros(*mask.shape[:-1], npad, dtype=mask.dtype, device=device or mask.device)
    store[..., :n] = mask.to(store.device)
    return store[..., :n]
