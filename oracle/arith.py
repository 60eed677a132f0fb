"""Size, traffic and work arithmetic the pages print, written out plainly.

TEST INFRASTRUCTURE ONLY (see oracle/ref.py). Every function is a direct
count of bytes, elements or operations; tests/test_oracle.py checks each one
against the figure the pages print for it.
"""
from __future__ import annotations

import math

MiB = 1 << 20
GiB = 1 << 30


def score_matrix_bytes(n: int, heads: int = 1, elem: int = 2) -> int:
    """One N x N score (or probability) matrix per head
    ("What is FlashAttention?", Step 1 and "Worked example")."""
    return heads * n * n * elem


def score_row_bytes(n: int, elem: int = 2) -> int:
    """One row of the score matrix ("Explain FlashAttention and why it is
    IO-aware", "A strong answer")."""
    return n * elem


def materialising_bytes(n: int, d: int, elem: int = 2):
    """Logical HBM bytes of the deliberately materialising one-head baseline:
    scores written, read, probabilities written, read, plus one read of Q, K,
    V and one write of O ("Explain FlashAttention and why it is IO-aware",
    "What the byte arithmetic does and does not say").
    Returns (score transfers, Q/K/V/O minimum, total)."""
    scores = 4 * n * n * elem
    io = 4 * n * d * elem
    return scores, io, scores + io


def bandwidth_floor_seconds(nbytes: int, bytes_per_second: float) -> float:
    return nbytes / bytes_per_second


def matmul_flops(n: int, d: int) -> float:
    """The two matrix products of one head, 2 N^2 d each."""
    return 4.0 * n * n * d


def attention_flops(batch: int, heads: int, n: int, d: int, causal: bool = False,
                    backward: bool = False) -> float:
    """Useful attention FLOPs: 4 N^2 d per head, halved for causal
    ("FlashAttention", "Checking it on a real system"); the backward counts
    2.5 times the forward (its five N^2 d products against the forward's two)."""
    f = matmul_flops(n, d) * batch * heads
    if causal:
        f /= 2.0
    if backward:
        f *= 2.5
    return f


def row_stats_bytes(n: int, elem: int = 4) -> int:
    """m and l per row in fp32 ("What is FlashAttention?", Step 4)."""
    return 2 * n * elem


def algorithm1_blocks(sram_elems: int, d: int):
    """Key block ceil(M / 4d) and query block min(that, d)
    ("What is FlashAttention?", Step 3)."""
    bc = math.ceil(sram_elems / (4 * d))
    return bc, min(bc, d)


def theorem2_ratio(n: int, d: int, sram_elems: int) -> float:
    """(N d + N^2) / (N^2 d^2 / M): standard over tiled HBM-access leading
    terms ("What is FlashAttention?", Step 3)."""
    return (n * d + n * n) / (n * n * d * d / sram_elems)


def panel_standard_traffic(n: int, heads: int, d: int, elem: int = 2):
    """Per-layer HBM traffic of the three-pass kernel in the "FlashAttention"
    page's byte-accounting panel: the score matrices cross the bus four times
    and Q, K, V, O once each. Returns (score bytes, Q/K/V/O bytes, total)."""
    scores = 4 * score_matrix_bytes(n, heads, elem)
    io = 4 * heads * n * d * elem
    return scores, io, scores + io


def panel_peak_intermediate(n: int, heads: int, d: int, flash: bool, elem: int = 2,
                            stat_elem: int = 4) -> int:
    """Peak intermediate bytes in the same panel: one layer of score matrices
    for the standard kernel; the output plus one fp32 statistic per row for
    the tiled kernel (the reading that reproduces both printed figures)."""
    if not flash:
        return score_matrix_bytes(n, heads, elem)
    return heads * n * d * elem + heads * n * stat_elem
