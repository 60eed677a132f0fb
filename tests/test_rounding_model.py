"""A CPU model of the kernels' rounding, and what it says about the gradient tolerance.

The backward takes D = rowsum(dO * O) from the O the forward stored in bf16. When the
softmax of a row is sharply peaked (the x30-score workload), dS = P (dP - D) is a small
difference of large terms, and an error of one bf16 step in a stored O element moves dQ
and dK of that row by far more than their own rounding. Chained on the kernel's forward,
the gradients therefore inherit the forward's O error; this model shows which rounding
dominates it and that the divisor the kernels use removes it.

The model repeats the kernels' arithmetic in fp64 with their roundings:
  forward: scores in the log2 domain; per 128-key tile a reference max that moves only
           when the tile max exceeds it by more than 8; p = 2^(s - m_ref) rounded to bf16
           for the P V product; l summed unrounded; LSE from l; O rounded to bf16;
  backward: P from the LSE, dS rounded to bf16 for dQ and dK, P rounded for dV, outputs
           rounded to bf16.
Two divisors of O are compared: l itself, and l with its largest term (p of the row max,
2^(m_row - m_ref) >= 1, generally not a bf16 number) swapped for the rounded value the
product used. It is test code only: it models the CUDA path and shares nothing with it.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import ref

rb = ref.round_bf16
LOG2E = math.log2(math.e)


def _forward_model(q, k, v, scale, mask, dominant_divisor):
    n = q.shape[0]
    c = scale * LOG2E
    o_out, lse = np.zeros_like(q), np.zeros(n)
    for c0 in range(0, n, 128):
        r = np.arange(c0, min(n, c0 + 128))
        s2 = (q[r] @ k.T) * c + mask[r] * LOG2E
        s2 = np.where(np.arange(n)[None, :] > r[:, None], -np.inf, s2)  # causal
        m_ref = np.full(len(r), -np.inf)
        m_row = np.full(len(r), -np.inf)
        l, o = np.zeros(len(r)), np.zeros((len(r), v.shape[1]))
        for j0 in range(0, c0 + 128, 128):
            t = s2[:, j0:j0 + 128]
            m_tile = t.max(axis=1)
            m_row = np.maximum(m_row, m_tile)
            m_new = np.where(m_tile > m_ref + 8.0, m_tile, m_ref)
            moved = m_new != m_ref
            with np.errstate(invalid="ignore"):
                alpha = np.where(moved, np.where(np.isneginf(m_ref), 0.0, np.exp2(m_ref - m_new)), 1.0)
            m_ref = m_new
            p = np.exp2(t - np.where(np.isneginf(m_ref), 0.0, m_ref)[:, None])
            l = l * alpha + p.sum(axis=1)
            o = o * alpha[:, None] + rb(p) @ v[j0:j0 + 128]
        den = l.copy()
        live = l > 0
        if dominant_divisor:
            pm = np.exp2(m_row[live] - m_ref[live])
            den[live] = l[live] + (rb(pm) - pm)
        o_out[r] = np.where(live[:, None], o / np.where(live, den, 1.0)[:, None], 0.0)
        lse[r] = np.where(live, (m_ref + np.log2(np.where(live, l, 1.0))) / LOG2E, -np.inf)
    return rb(o_out), lse.astype(np.float32).astype(np.float64)


def _backward_model(q, k, v, do, o, lse, scale, mask):
    n = q.shape[0]
    L = np.where(np.isneginf(lse), np.inf, lse)
    D = (do * o).sum(axis=1)
    s = scale * (q @ k.T) + mask
    s = np.where(np.arange(n)[None, :] > np.arange(n)[:, None], -np.inf, s)
    p = np.exp(s - L[:, None])
    ds = rb(p * (do @ v.T - D[:, None]))
    return rb(scale * ds @ k), rb(scale * ds.T @ q), rb(rb(p).T @ do)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.fixture(scope="module")
def peaked_head():
    # one head of the x30-score causal workload (Q and K scaled by sqrt(30)), shortened
    w = W.WORKLOADS[4]
    inp = W.make_inputs(w, shape=(1, 1, 2048, 128))
    f = lambda t: t[0, 0].to(torch.float64).numpy()  # noqa: E731
    q, k, v, do, mask = f(inp["q"]), f(inp["k"]), f(inp["v"]), f(inp["do"]), f(inp["mask"])
    stored = ref.backward_head(q, k, v, do, w.scale, True, mask, o_storage="bf16")
    return q, k, v, do, mask, w.scale, stored


def test_dominant_term_divisor_keeps_chained_gradients_within_tolerance(peaked_head):
    q, k, v, do, mask, scale, stored = peaked_head
    errs = {}
    for dom in (False, True):
        o, lse = _forward_model(q, k, v, scale, mask, dom)
        dq, dk, dv = _backward_model(q, k, v, do, o, lse, scale, mask)
        errs[dom] = (_rel(dq, stored[0]), _rel(dk, stored[1]), _rel(dv, stored[2]))
    # with the plain divisor the rounding of each row's largest p passes into O and, through D,
    # into dQ and dK; the swapped term removes most of that error
    assert errs[True][0] < 5e-3 and errs[True][1] < 5e-3 and errs[True][2] < 5e-3, errs
    assert errs[False][0] > 1.3 * errs[True][0] and errs[False][1] > 1.3 * errs[True][1], errs
    assert errs[False][2] == errs[True][2]  # dV does not depend on O


def test_gradients_from_stored_outputs_are_within_tolerance(peaked_head):
    # fed the oracle's own saved O and LSE, the modelled backward differs from the stored-output
    # oracle only by the rounding of P, dS and the outputs
    q, k, v, do, mask, scale, stored = peaked_head
    O, L = ref.forward_head(q, k, v, scale, True, mask)
    dq, dk, dv = _backward_model(q, k, v, do, rb(O), L.astype(np.float32).astype(np.float64), scale, mask)
    assert _rel(dq, stored[0]) < 5e-3 and _rel(dk, stored[1]) < 5e-3 and _rel(dv, stored[2]) < 5e-3
