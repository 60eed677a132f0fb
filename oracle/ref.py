"""fp64 CPU oracle for exact scaled-dot-product attention (forward and backward).

TEST INFRASTRUCTURE ONLY. Nothing in the library imports this module; only
the tests, the package smoke check and the benchmark's CPU-baseline leg do.
It shares no code with the CUDA path.

What it computes is the plain definition the explainer pages say the tiled
method reaches exactly, up to rounding ("What is FlashAttention?", "Common
mistakes"; "FlashAttention", "Why it is allowed to be exact"; "Explain
FlashAttention and why it is IO-aware", "Exact attention, finite precision and
backward"). There is no tiling and no online recurrence here: per query row
it forms every score, takes one stable softmax and one weighted sum of V.
Query rows are processed in chunks of 256 only so that no N x N matrix per
head is ever held; each chunk is computed independently and exactly as the
definition says.

Forward, per (batch b, head h, query row i)
("Explain FlashAttention and why it is IO-aware", "Keep only the state
needed for the final weighted average"):
    s_ij = scale * <q_i, k_j> + mask_ij          (mask_ij = 0 without a mask)
    s_ij = -inf if causal and j > i              (absolute positions, same
                                                  section of that page, on
                                                  causal attention)
    R_i  = { j : s_ij > -inf }
    R_i empty  ->  o_i = 0, LSE_i = -inf         (the page's all-masked-row
                                                  policy, "Executable
                                                  recurrence, with an
                                                  empty-state policy")
    otherwise  m_i = max_j s_ij, l_i = sum_j exp(s_ij - m_i),
               P_ij = exp(s_ij - m_i) / l_i, o_i = sum_j P_ij v_j,
               LSE_i = m_i + ln l_i

Backward. The pages say only that S and P are recomputed from Q, K, V and
the saved row statistics ("What is FlashAttention?", Step 4;
"FlashAttention", "What it does not do"). The oracle takes the textbook
softmax-attention gradient, which that recomputation implies:
    dV = P^T dO,   dP = dO V^T,   D_i = sum_j P_ij dP_ij  (= <dO_i, o_i>),
    dS = P * (dP - D),   dQ = scale * dS K,   dK = scale * dS^T Q.
No gradient flows into the additive mask. Rows with empty R_i contribute
nothing. D is computed both ways and the two must agree to fp64 rounding.

Inputs may be any float dtype (bf16 tensors are converted by the caller to
fp64 exactly); everything is computed in fp64.

Stored output. The backward consumes the O that the forward stored, and the
library stores O in the dtype of Q. `attention_backward(..., o_storage=
"bf16")` (or "f16") therefore also models that storage: the oracle rounds its
own fp64 O to fp32 and then to bf16 or half (round to nearest even, as the
kernels do from their fp32 accumulators) and takes D = rowsum(dO * O_stored)
from it. Nothing else
changes; with o_storage=None the result is the pure mathematical gradient.

Parity pins: every function here is pinned by tests/test_oracle.py against
the pages' worked numbers, closed forms, invariants, a scalar brute force,
torch's fp64 scaled_dot_product_attention on the masked/causal special cases
and finite differences for the gradients.
"""
from __future__ import annotations

from typing import Optional, Sequence, Tuple

import numpy as np

CHUNK = 256


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def round_bf16(x) -> np.ndarray:
    """fp64 -> fp32 -> bf16 (round to nearest, ties to even), returned as fp64."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    finite = np.isfinite(f)
    out = np.where(finite, r, u & 0xFFFF0000).astype(np.uint32)
    return out.view(np.float32).astype(np.float64)


def round_f16(x) -> np.ndarray:
    """fp64 -> fp32 -> IEEE half (round to nearest, ties to even; beyond the
    largest finite half, 65504, the result is infinite), returned as fp64."""
    with np.errstate(over="ignore"):
        return np.asarray(x, dtype=np.float32).astype(np.float16).astype(np.float64)


_STORAGE = {"bf16": round_bf16, "f16": round_f16}


def decode_e4m3(codes) -> np.ndarray:
    """8-bit E4M3 floating-point codes (the FP8 format of an FP8 forward pass, "What is
    FlashAttention?", FAQ on FlashAttention-3) -> fp64, from the format's definition:
    bit 7 sign, bits 6..3 a biased exponent (bias 7), bits 2..0 the fraction.
      exponent 0:        (fraction / 8) * 2^-6            (zero and subnormals)
      exponent 1..15:    (1 + fraction / 8) * 2^(e - 7)   (largest finite: 448)
      exponent 15 with fraction 7: not a number; the format has no infinities."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    e = (c >> 3) & 0xF
    f = (c & 7).astype(np.float64)
    mag = np.where(e == 0, f / 8.0 * 2.0 ** -6, (1.0 + f / 8.0) * np.exp2((e - 7).astype(np.float64)))
    mag = np.where((e == 15) & (c & 7 == 7), np.nan, mag)
    return np.where((c & 0x80) != 0, -mag, mag)


def _mask_for_head(mask: Optional[np.ndarray], b: int, h: int) -> Optional[np.ndarray]:
    """mask has shape (Bm, Hm, N, N) with Bm in {1, B} and Hm in {1, H}."""
    if mask is None:
        return None
    bm = b if mask.shape[0] > 1 else 0
    hm = h if mask.shape[1] > 1 else 0
    return mask[bm, hm]


def head_scores(qh: np.ndarray, kh: np.ndarray, rows: np.ndarray, scale: float,
                causal: bool, maskh: Optional[np.ndarray]) -> np.ndarray:
    """Scaled, masked scores s_ij for the query rows `rows` of one head, fp64."""
    s = scale * (qh[rows] @ kh.T)
    if maskh is not None:
        s = s + maskh[rows]
    if causal:
        keys = np.arange(kh.shape[0])
        s = np.where(keys[None, :] > rows[:, None], -np.inf, s)
    return s


def row_softmax(s: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Stable softmax of each row of s and its natural-log LSE.

    A row whose scores are all -inf gets P = 0 and LSE = -inf.
    """
    if s.shape[1] == 0:
        return np.zeros_like(s), np.full(s.shape[0], -np.inf)
    m = s.max(axis=1)
    empty = np.isneginf(m)
    shift = np.where(empty, 0.0, m)
    e = np.exp(s - shift[:, None])  # exp(-inf) = 0, never -inf - (-inf)
    l = e.sum(axis=1)
    safe_l = np.where(empty, 1.0, l)
    p = np.where(empty[:, None], 0.0, e / safe_l[:, None])
    lse = np.where(empty, -np.inf, shift + np.log(safe_l))
    return p, lse


def forward_head(qh, kh, vh, scale: float, causal: bool = False, maskh=None,
                 rows: Optional[Sequence[int]] = None) -> Tuple[np.ndarray, np.ndarray]:
    """O and LSE for the query rows `rows` (all rows if None) of one head."""
    qh, kh, vh = _f64(qh), _f64(kh), _f64(vh)
    maskh = None if maskh is None else _f64(maskh)
    n = qh.shape[0]
    rows = np.arange(n) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.zeros((rows.shape[0], vh.shape[1]))
    lse = np.full(rows.shape[0], -np.inf)
    for c0 in range(0, rows.shape[0], CHUNK):
        r = rows[c0:c0 + CHUNK]
        p, l = row_softmax(head_scores(qh, kh, r, scale, causal, maskh))
        out[c0:c0 + CHUNK] = p @ vh
        lse[c0:c0 + CHUNK] = l
    return out, lse


def attention_forward(q, k, v, scale: float, causal: bool = False, mask=None):
    """O [B,H,N,d] and LSE [B,H,N] in fp64 for inputs [B,H,N,d]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    mask = None if mask is None else _f64(mask)
    B, H, N, d = q.shape
    o = np.zeros((B, H, N, v.shape[3]))
    lse = np.full((B, H, N), -np.inf)
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = forward_head(q[b, h], k[b, h], v[b, h], scale, causal,
                                              _mask_for_head(mask, b, h))
    return o, lse


def attention_forward_fp8(q8, k8, v8, q_descale: float, k_descale: float, v_descale: float, scale: float,
                          causal: bool = False, mask=None):
    """FP8 forward: Q, K, V arrive as E4M3 codes (uint8) with one descale factor per tensor, and
    the values they stand for are code value x descale. What the forward computes is the plain
    attention of those values ("What is FlashAttention?", FAQ: FlashAttention-3's FP8 forward
    computes the same attention at lower precision), so this is attention_forward on the
    decoded, descaled inputs, in fp64."""
    q = decode_e4m3(q8) * float(q_descale)
    k = decode_e4m3(k8) * float(k_descale)
    v = decode_e4m3(v8) * float(v_descale)
    return attention_forward(q, k, v, scale, causal, mask)


def decode_forward(q, k, v, scale: float, causal: bool = False):
    """Decode: O [B,H,nq,d] and LSE [B,H,nq] for nq query rows against nk keys,
    fp64, by the plain definition. With causal the queries are the last nq
    positions: query i sits at position nk - nq + i and sees the keys j with
    j <= nk - nq + i ("FlashAttention", "What it does not do": at decode the
    query is the newest row against the whole cache). A query that sees no
    key gets O = 0 and LSE = -inf, the all-masked policy of the forward."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, nq, _ = q.shape
    nk = k.shape[2]
    o = np.zeros((B, H, nq, v.shape[3]))
    lse = np.full((B, H, nq), -np.inf)
    for b in range(B):
        for h in range(H):
            s = scale * (q[b, h] @ k[b, h].T)
            if causal:
                limit = nk - nq + np.arange(nq)
                s = np.where(np.arange(nk)[None, :] > limit[:, None], -np.inf, s)
            p, lse[b, h] = row_softmax(s)
            o[b, h] = p @ v[b, h]
    return o, lse


def backward_head(qh, kh, vh, doh, scale: float, causal: bool = False, maskh=None,
                  q_rows: Optional[Sequence[int]] = None,
                  k_rows: Optional[Sequence[int]] = None, o_storage: Optional[str] = None):
    """Gradients of one head, by the closed form in the module docstring.

    Returns (dq[q_rows], dk[k_rows], dv[k_rows], D, D_from_o) where D and
    D_from_o cover every query row. With o_storage="bf16" (or "f16"), D is
    taken from the bf16- (or half-) rounded O (the stored output) instead of
    from P and dP.
    dK and dV of a key need every query row, so the whole head is always
    swept; `q_rows` / `k_rows` only select which gradient rows are returned
    (None = all).
    """
    qh, kh, vh, doh = _f64(qh), _f64(kh), _f64(vh), _f64(doh)
    maskh = None if maskh is None else _f64(maskh)
    n, d = qh.shape
    q_sel = np.arange(n) if q_rows is None else np.asarray(q_rows, dtype=np.int64)
    k_sel = np.arange(kh.shape[0]) if k_rows is None else np.asarray(k_rows, dtype=np.int64)
    q_pos = np.full(n, -1)
    q_pos[q_sel] = np.arange(q_sel.shape[0])
    dq = np.zeros((q_sel.shape[0], d))
    dk = np.zeros((k_sel.shape[0], d))
    dv = np.zeros((k_sel.shape[0], vh.shape[1]))
    D = np.zeros(n)
    D_o = np.zeros(n)
    for c0 in range(0, n, CHUNK):
        r = np.arange(c0, min(n, c0 + CHUNK))
        p, _ = row_softmax(head_scores(qh, kh, r, scale, causal, maskh))
        o_rows = p @ vh
        dp = doh[r] @ vh.T
        D_o[r] = (doh[r] * o_rows).sum(axis=1)
        if o_storage in _STORAGE:
            d_rows = (doh[r] * _STORAGE[o_storage](o_rows)).sum(axis=1)
        elif o_storage is None:
            d_rows = (p * dp).sum(axis=1)
        else:
            raise ValueError(f"unknown o_storage {o_storage!r}")
        D[r] = d_rows
        ds = p * (dp - d_rows[:, None])
        want = q_pos[r] >= 0
        if want.any():
            dq[q_pos[r][want]] = scale * (ds[want] @ kh)
        dk += scale * (ds[:, k_sel].T @ qh[r])
        dv += p[:, k_sel].T @ doh[r]
    return dq, dk, dv, D, D_o


def attention_backward(q, k, v, do, scale: float, causal: bool = False, mask=None,
                       o_storage: Optional[str] = None):
    """dQ, dK, dV [B,H,N,d] and D [B,H,N] in fp64 (D checked both ways when
    o_storage is None)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    mask = None if mask is None else _f64(mask)
    B, H, N, d = q.shape
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    D = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h], dv[b, h], D[b, h], D_o = backward_head(
                q[b, h], k[b, h], v[b, h], do[b, h], scale, causal, _mask_for_head(mask, b, h),
                o_storage=o_storage)
            scale_ref = max(1.0, float(np.abs(D[b, h]).max(initial=0.0)))
            if o_storage is None and not np.allclose(D[b, h], D_o, rtol=0.0, atol=1e-10 * scale_ref):
                raise AssertionError("D = rowsum(P * dP) and D = rowsum(dO * O) disagree")
    return dq, dk, dv, D
