"""The online-softmax recurrence itself, in plain fp64 Python/NumPy.

TEST INFRASTRUCTURE ONLY (see oracle/ref.py). A second, deliberately plainer
oracle: it walks the tiles one by one with the running state the pages
describe, so that the pages' worked examples can be replayed step by step and
the BLAS oracle in ref.py can be cross-checked on small inputs.

State per query row ("Explain FlashAttention and why it is IO-aware",
"Keep only the state needed for the final weighted average";
"What is FlashAttention?", Step 2):
    m  the largest score seen so far
    l  the sum of exp(score - m) over the scores seen so far
    o  the exp(score - m)-weighted sum of the value rows seen so far
A tile with scores s and value rows V_t updates it as
    m' = max(m, max s),  alpha = exp(m - m'),
    l  <- alpha l + sum exp(s - m'),   o <- alpha o + exp(s - m') V_t,
and after the last tile the row's output is o / l.

Empty-state policy ("Explain FlashAttention and why it is IO-aware",
"Executable recurrence, with an empty-state policy"): a tile whose scores
are all -inf changes nothing and is skipped before any subtraction, so
-inf - (-inf) is never evaluated; a row that never saw a finite score
returns zeros. Scores may be finite or -inf; NaN and +inf scores, non-finite
values and a tile width that is not a positive int are rejected with
ValueError, as that page's contract states.

`break_rescale` and `subtract_max=False` reproduce the two ways the
"FlashAttention" page ("Why it is allowed to be exact") breaks the
algorithm; they exist only for the tests that replay those experiments.
"""
from __future__ import annotations

import math
from typing import List, Optional, Tuple

import numpy as np


class RowState:
    """Running (m, l, o) of one query row."""

    def __init__(self, width: int, dtype=np.float64, subtract_max: bool = True,
                 break_rescale: bool = False):
        self.dtype = dtype
        self.m = dtype(-np.inf)
        self.l = dtype(0.0)
        self.o = np.zeros(width, dtype=dtype)
        self.subtract_max = subtract_max
        self.break_rescale = break_rescale

    def absorb(self, scores: np.ndarray, values: np.ndarray) -> None:
        scores = scores.astype(self.dtype)
        values = values.astype(self.dtype)
        tile_max = scores.max()
        if np.isneginf(tile_max):
            return  # all masked: nothing to add, and no -inf - (-inf)
        new_m = max(self.m, tile_max)
        if self.subtract_max:
            shift = new_m
            alpha = self.dtype(0.0) if np.isneginf(self.m) else np.exp(self.m - new_m)
        else:
            shift = self.dtype(0.0)
            alpha = self.dtype(1.0)
        if self.break_rescale:
            alpha = self.dtype(1.0)
        with np.errstate(over="ignore", invalid="ignore"):
            w = np.exp(scores - shift).astype(self.dtype)
            self.l = self.dtype(alpha * self.l + w.sum(dtype=self.dtype))
            self.o = (alpha * self.o + w @ values).astype(self.dtype)
        self.m = self.dtype(new_m)

    def result(self) -> np.ndarray:
        if self.l == 0:
            return np.zeros_like(self.o)
        with np.errstate(over="ignore", invalid="ignore"):
            return self.o / self.l


def merge_states(a: RowState, b: RowState) -> RowState:
    """The state of a row whose keys are those of `a` followed by those of `b`.

    Two partial states combine with the same rescaling that absorbs a tile
    ("Explain FlashAttention and why it is IO-aware", "Keep only the state
    needed for the final weighted average"): against the larger maximum m,
    each state's l and o are scaled by exp(m_own - m) and added. A state that
    saw no finite score (m = -inf, l = 0, o = 0) is the identity. This is the
    combine step of a split-key decode ("FlashAttention", "What it does not
    do")."""
    out = RowState(a.o.shape[0], dtype=a.dtype)
    if np.isneginf(a.m) and np.isneginf(b.m):
        return out
    m = max(a.m, b.m)
    wa = 0.0 if np.isneginf(a.m) else np.exp(a.m - m)
    wb = 0.0 if np.isneginf(b.m) else np.exp(b.m - m)
    out.m = a.dtype(m)
    out.l = a.dtype(wa * a.l + wb * b.l)
    out.o = (wa * a.o + wb * b.o).astype(a.dtype)
    return out


def _check_contract(scores: np.ndarray, values: np.ndarray, tile) -> None:
    if scores.ndim != 1 or values.ndim != 2 or scores.shape[0] != values.shape[0]:
        raise ValueError("need a 1-D score vector and one value row per score")
    if not isinstance(tile, int) or isinstance(tile, bool) or tile <= 0:
        raise ValueError("tile width must be a positive int")
    if np.isnan(scores).any() or np.isposinf(scores).any():
        raise ValueError("scores must be finite or -inf")
    if not np.isfinite(values).all():
        raise ValueError("values must be finite")


def online_row(scores, values, tile: int = 2) -> np.ndarray:
    """Output of one query row from precomputed scaled/masked scores, tile by tile."""
    scores = np.asarray(scores, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    _check_contract(scores, values, tile)
    st = RowState(values.shape[1])
    for start in range(0, scores.shape[0], tile):
        st.absorb(scores[start:start + tile], values[start:start + tile])
    return st.result()


def online_trace(scores, tile: int) -> List[Tuple[float, float]]:
    """(m, l) after each tile, for replaying the pages' worked examples."""
    scores = np.asarray(scores, dtype=np.float64)
    st = RowState(1)
    trace = []
    for start in range(0, scores.shape[0], tile):
        chunk = scores[start:start + tile]
        st.absorb(chunk, np.zeros((chunk.shape[0], 1)))
        trace.append((float(st.m), float(st.l)))
    return trace


def online_row_states(scores, values, tile: int) -> List[Tuple[float, float, np.ndarray]]:
    """(m, l, o) after each tile (unnormalised o)."""
    scores = np.asarray(scores, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    _check_contract(scores, values, tile)
    st = RowState(values.shape[1])
    out = []
    for start in range(0, scores.shape[0], tile):
        st.absorb(scores[start:start + tile], values[start:start + tile])
        out.append((float(st.m), float(st.l), st.o.copy()))
    return out


def online_row_variant(scores, values, tile: int, dtype=np.float64, subtract_max: bool = True,
                       break_rescale: bool = False) -> np.ndarray:
    """online_row in another precision, optionally broken on purpose."""
    scores = np.asarray(scores, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    _check_contract(scores, values, tile)
    st = RowState(values.shape[1], dtype=dtype, subtract_max=subtract_max,
                  break_rescale=break_rescale)
    for start in range(0, scores.shape[0], tile):
        st.absorb(scores[start:start + tile], values[start:start + tile])
    return st.result()


def tiled_attention(q, k, v, scale: float, block_q: int, block_k: int, causal: bool = False,
                    mask: Optional[np.ndarray] = None):
    """One head of attention in the FlashAttention-2 order, fp64.

    Query blocks in the outer loop keep their (m, l, o) resident; key/value
    blocks stream through the inner loop ("What is FlashAttention?", Step 3).
    Returns (O, LSE, largest number of scores held at once).
    """
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    n, n_k = q.shape[0], k.shape[0]
    out = np.zeros((n, v.shape[1]))
    lse = np.full(n, -np.inf)
    held = 0
    for q0 in range(0, n, block_q):
        rows = np.arange(q0, min(n, q0 + block_q))
        m = np.full(rows.shape[0], -np.inf)
        l = np.zeros(rows.shape[0])
        o = np.zeros((rows.shape[0], v.shape[1]))
        for k0 in range(0, n_k, block_k):
            cols = np.arange(k0, min(n_k, k0 + block_k))
            s = scale * (q[rows] @ k[cols].T)
            if mask is not None:
                s = s + mask[np.ix_(rows, cols)]
            if causal:
                s = np.where(cols[None, :] > rows[:, None], -np.inf, s)
            held = max(held, s.size)
            tile_max = s.max(axis=1)
            live = ~np.isneginf(tile_max)  # rows with at least one finite score here
            if not live.any():
                continue
            new_m = np.where(live, np.maximum(m, tile_max), m)
            seen = ~np.isneginf(m)
            alpha = np.ones_like(m)
            alpha[live & ~seen] = 0.0
            both = live & seen
            alpha[both] = np.exp(m[both] - new_m[both])
            shift = np.where(np.isneginf(new_m), 0.0, new_m)
            w = np.where(live[:, None], np.exp(s - shift[:, None]), 0.0)
            l = alpha * l + w.sum(axis=1)
            o = alpha[:, None] * o + w @ v[cols]
            m = new_m
        nz = l > 0
        out[rows[nz]] = o[nz] / l[nz, None]
        lse[rows[nz]] = m[nz] + np.log(l[nz])
    return out, lse, held


def exp_sum_one_shot(scores) -> Tuple[float, float]:
    """(max, sum exp(s - max)) of a whole row at once, with math.exp."""
    mx = max(scores)
    return mx, sum(math.exp(s - mx) for s in scores)
