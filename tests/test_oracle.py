"""Pins for the fp64 oracle: page-printed values, closed forms, invariants,
a scalar brute force, torch's fp64 SDPA on the special cases it covers, and
finite differences for the gradients. CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import arith, online, ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- brute force
def brute_attention(q, k, v, scale, causal=False, mask=None):
    """Scalar triple loop with math.exp: the definition, one number at a time."""
    B, H, N, d = q.shape
    dv = v.shape[3]
    O = np.zeros((B, H, N, dv))
    L = np.full((B, H, N), -np.inf)
    for b in range(B):
        for h in range(H):
            for i in range(N):
                s = []
                for j in range(N):
                    if causal and j > i:
                        s.append(-math.inf)
                        continue
                    acc = 0.0
                    for t in range(d):
                        acc += float(q[b, h, i, t]) * float(k[b, h, j, t])
                    extra = 0.0
                    if mask is not None:
                        extra = float(mask[b if mask.shape[0] > 1 else 0, h if mask.shape[1] > 1 else 0, i, j])
                    s.append(scale * acc + extra)
                finite = [x for x in s if x != -math.inf]
                if not finite:
                    continue
                mx = max(finite)
                w = [0.0 if x == -math.inf else math.exp(x - mx) for x in s]
                tot = sum(w)
                for c in range(dv):
                    O[b, h, i, c] = sum(w[j] * float(v[b, h, j, c]) for j in range(N)) / tot
                L[b, h, i] = mx + math.log(tot)
    return O, L


# ------------------------------------------------- "What is FlashAttention?"
def test_six_scores_running_stats():
    g = _golden("six_scores.json")
    trace = online.online_trace(g["scores"], g["block"])
    tol = 0.5 * 10 ** -g["printed_decimals"]
    assert trace[0][0] == g["after_block_1"]["m"]
    assert abs(trace[0][1] - g["after_block_1"]["l"]) <= tol
    assert trace[1][0] == g["final"]["m"]
    assert abs(trace[1][1] - g["final"]["l"]) <= tol
    mx, one_shot = online.exp_sum_one_shot(g["scores"])
    assert mx == trace[1][0]
    assert abs(one_shot - trace[1][1]) <= 1e-15


def test_six_scores_with_value_vectors():
    g = _golden("six_scores.json")
    s = np.array(g["scores"])
    vals = _rng(1).standard_normal((6, 8))
    got = online.online_row(s, vals, g["block"])
    p, _ = ref.row_softmax(s[None, :])
    want = (p @ vals)[0]
    # the page saw ~5.6e-17, i.e. fp64 rounding
    assert np.max(np.abs(got - want)) <= 1e-15


def test_two_tile_toy():
    g = _golden("two_tile_toy.json")
    states = online.online_row_states(g["scores"], g["values"], g["tile"])
    for (m, l, o), want in zip(states, g["states"]):
        assert abs(m - want["m"]) <= 1e-15
        assert abs(l - want["l"]) <= 1e-14
        assert abs(o[0] - want["o"]) <= 1e-13
    assert abs(math.exp(states[0][0] - states[1][0]) - g["states"][1]["alpha"]) <= 1e-15
    got = online.online_row(g["scores"], g["values"], g["tile"])
    assert abs(got[0] - 50.0 / 3.0) <= 1e-13
    assert abs(got[0] - g["result"]) <= 1e-13


@pytest.mark.parametrize("tile", [1, 2, 3, 4, 6])
def test_tile_width_independence_six_scores(tile):
    s = np.array(_golden("six_scores.json")["scores"])
    vals = _rng(2).standard_normal((6, 5))
    want = online.online_row(s, vals, 6)
    assert np.max(np.abs(online.online_row(s, vals, tile) - want)) <= 1e-15


@pytest.mark.parametrize("tile", [16, 32, 64, 128, 256])
def test_tile_width_independence_fp32(tile):
    # "FlashAttention": moving the tile width does not move the result in any
    # digit float32 can represent.
    r = _rng(3)
    s = r.standard_normal(256) * 3
    vals = r.standard_normal((256, 4))
    got = online.online_row_variant(s, vals, tile, dtype=np.float32)
    want = online.online_row_variant(s, vals, 256, dtype=np.float32)
    truth = online.online_row(s, vals, 256)
    assert np.max(np.abs(got.astype(np.float64) - truth)) <= 1e-5
    assert np.max(np.abs(got - want)) <= 8 * np.finfo(np.float32).eps * np.max(np.abs(truth))


def test_break_rescale_gives_wrong_answer():
    s = np.array(_golden("six_scores.json")["scores"])
    vals = _rng(4).standard_normal((6, 3))
    good = online.online_row(s, vals, 3)
    bad = online.online_row_variant(s, vals, 3, break_rescale=True)
    assert np.max(np.abs(bad - good)) > 1e-3


def test_break_max_subtraction_fp32():
    # largest base score 3, so x6 -> 18 and x30 -> 90; exp(90) ~ 1.2e39 > fp32 max
    base = np.array([1.0, 3.0, -2.0])
    vals = _rng(5).standard_normal((3, 2))
    for mult, finite in ((6.0, True), (30.0, False)):
        s = base * mult
        got = online.online_row_variant(s, vals, 1, dtype=np.float32, subtract_max=False)
        safe = online.online_row_variant(s, vals, 1, dtype=np.float32, subtract_max=True)
        truth = online.online_row(s, vals, 1)
        assert np.all(np.isfinite(safe))
        assert np.max(np.abs(safe - truth)) <= 1e-5
        if finite:
            assert np.max(np.abs(got - truth)) <= 1e-5
        else:
            assert not np.all(np.isfinite(got))
    assert math.exp(90.0) > float(np.finfo(np.float32).max)


def test_tiled_run_n256_d16():
    g = _golden("size_figures.json")["tiled_run"]
    r = _rng(6)
    n, d, blk = g["N"], g["d"], g["block"]
    q, k, v = (r.standard_normal((n, d)) for _ in range(3))
    scale = 1 / math.sqrt(d)
    o_t, lse_t, held = online.tiled_attention(q, k, v, scale, blk, blk)
    o, lse = ref.forward_head(q, k, v, scale)
    assert np.max(np.abs(o_t - o)) <= 1e-14
    assert np.max(np.abs(lse_t - lse)) <= 1e-13
    assert held == g["scores_per_tile"]
    assert n * n == g["scores_standard"]


# ------------------------------------------------------------ invariants etc.
def test_rows_sum_to_one_and_convex_hull():
    r = _rng(7)
    s = r.standard_normal((64, 200)) * 4
    s[3, :] = -np.inf
    s[5, ::2] = -np.inf
    p, lse = ref.row_softmax(s)
    assert np.all(p >= 0)
    sums = p.sum(axis=1)
    assert np.all(np.abs(sums[np.arange(64) != 3] - 1) <= 1e-14)
    assert sums[3] == 0 and np.isneginf(lse[3])
    q, k, v = (r.standard_normal((1, 1, 50, 8)) for _ in range(3))
    o, _ = ref.attention_forward(q, k, v, 0.3, causal=True)
    assert np.all(o[0, 0] <= v[0, 0].max(axis=0) + 1e-12)
    assert np.all(o[0, 0] >= v[0, 0].min(axis=0) - 1e-12)


def _tiny_case(seed, B, H, N, d, causal, masked):
    r = _rng(seed)
    q, k, v = (r.standard_normal((B, H, N, d)) for _ in range(3))
    mask = None
    if masked:
        mask = r.standard_normal((B, 1, N, N))
        mask[r.random((B, 1, N, N)) < 0.25] = -np.inf
        mask[0, 0, N // 2, :] = -np.inf  # one all-masked row
    return q, k, v, mask


@pytest.mark.parametrize("shape", [(1, 1, 1, 1), (1, 1, 5, 3), (2, 2, 8, 4), (1, 3, 7, 2)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("masked", [False, True])
def test_brute_force_tiny(shape, causal, masked):
    B, H, N, d = shape
    q, k, v, mask = _tiny_case(hash((shape, causal, masked)) % 2**31, B, H, N, d, causal, masked)
    scale = 0.7
    o, lse = ref.attention_forward(q, k, v, scale, causal, mask)
    o_b, lse_b = brute_attention(q, k, v, scale, causal, mask)
    assert np.max(np.abs(o - o_b)) <= 1e-12
    fin = np.isfinite(lse_b)
    assert np.array_equal(fin, np.isfinite(lse))
    assert np.max(np.abs(lse[fin] - lse_b[fin]), initial=0.0) <= 1e-12
    assert np.all(o[~fin] == 0)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("masked", [False, True])
def test_against_torch_sdpa_fp64(causal, masked):
    r = _rng(11)
    B, H, N, d = 2, 3, 37, 16
    q, k, v = (r.standard_normal((B, H, N, d)) for _ in range(3))
    mask = r.standard_normal((B, 1, N, N)) * 2 if masked else None
    scale = 1 / math.sqrt(d)
    o, lse = ref.attention_forward(q, k, v, scale, causal, mask)
    tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
    am = None
    if masked or causal:
        am = torch.zeros(B, 1, N, N, dtype=torch.float64)
        if masked:
            am = am + torch.from_numpy(mask)
        if causal:
            am = am.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    want = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=am, scale=scale)
    assert np.max(np.abs(o - want.numpy())) <= 1e-12
    s = torch.einsum("bhid,bhjd->bhij", tq, tk) * scale
    if am is not None:
        s = s + am
    assert np.max(np.abs(lse - torch.logsumexp(s, dim=-1).numpy())) <= 1e-12


@pytest.mark.parametrize("shift", [-1e4, 1e4])
def test_shift_invariance(shift):
    r = _rng(12)
    q, k, v = (r.standard_normal((1, 1, 40, 8)) for _ in range(3))
    base = np.zeros((1, 1, 40, 40))
    moved = base.copy()
    moved[0, 0, 7, :] += shift
    o0, l0 = ref.attention_forward(q, k, v, 0.5, False, base)
    o1, l1 = ref.attention_forward(q, k, v, 0.5, False, moved)
    assert np.max(np.abs(o1 - o0)) <= 1e-9
    assert abs((l1[0, 0, 7] - l0[0, 0, 7]) - shift) <= 1e-9
    assert np.max(np.abs(np.delete(l1 - l0, 7, axis=2))) == 0


def test_special_cases():
    r = _rng(13)
    # one key: o = v_0, LSE = s_00
    q, k, v = (r.standard_normal((1, 1, 1, 6)) for _ in range(3))
    o, lse = ref.attention_forward(q, k, v, 0.4)
    assert np.array_equal(o[0, 0, 0], v[0, 0, 0])
    assert abs(lse[0, 0, 0] - 0.4 * float(q[0, 0, 0] @ k[0, 0, 0])) <= 1e-15
    # equal scores: o = mean of v, LSE = s + ln N
    n = 9
    q = r.standard_normal((1, 1, n, 4))
    k = np.zeros((1, 1, n, 4))
    v = r.standard_normal((1, 1, n, 4))
    o, lse = ref.attention_forward(q, k, v, 1.0)
    assert np.max(np.abs(o[0, 0] - v[0, 0].mean(axis=0))) <= 1e-15
    assert np.max(np.abs(lse - math.log(n))) <= 1e-15
    # causal row 0 sees only key 0
    q, k, v = (r.standard_normal((1, 1, n, 4)) for _ in range(3))
    o, lse = ref.attention_forward(q, k, v, 0.5, causal=True)
    assert np.array_equal(o[0, 0, 0], v[0, 0, 0])
    assert abs(lse[0, 0, 0] - 0.5 * float(q[0, 0, 0] @ k[0, 0, 0])) <= 1e-15


def test_mask_broadcast_equals_expanded():
    r = _rng(14)
    q, k, v = (r.standard_normal((2, 3, 10, 4)) for _ in range(3))
    m = r.standard_normal((1, 1, 10, 10))
    o1, l1 = ref.attention_forward(q, k, v, 0.5, True, m)
    o2, l2 = ref.attention_forward(q, k, v, 0.5, True, np.broadcast_to(m, (2, 3, 10, 10)).copy())
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_empty_inputs():
    for shape in ((0, 2, 5, 4), (2, 0, 5, 4), (1, 1, 0, 4)):
        q = np.zeros(shape)
        o, lse = ref.attention_forward(q, q, q, 1.0, True)
        assert o.shape == shape and lse.shape == shape[:3]
        dq, dk, dv, D = ref.attention_backward(q, q, q, q, 1.0, True)
        assert dq.shape == shape and D.shape == shape[:3]


def test_chunked_equals_single_chunk(monkeypatch):
    r = _rng(15)
    q, k, v = (r.standard_normal((1, 1, 600, 8)) for _ in range(3))
    o1, l1 = ref.attention_forward(q, k, v, 0.3, True)
    monkeypatch.setattr(ref, "CHUNK", 10_000)
    o2, l2 = ref.attention_forward(q, k, v, 0.3, True)
    assert np.max(np.abs(o1 - o2)) <= 1e-14 and np.max(np.abs(l1 - l2)) <= 1e-13


# ------------------------------------------------------- online_row contract
def test_online_row_contract():
    vals = np.ones((3, 2))
    with pytest.raises(ValueError):
        online.online_row([1.0, np.nan, 0.0], vals)
    with pytest.raises(ValueError):
        online.online_row([1.0, np.inf, 0.0], vals)
    with pytest.raises(ValueError):
        online.online_row([1.0, 2.0, 0.0], np.array([[1.0, 2.0], [np.inf, 0], [0, 0]]))
    for bad in (0, -1, 2.0, True):
        with pytest.raises(ValueError):
            online.online_row([1.0, 2.0, 0.0], vals, bad)
    with pytest.raises(ValueError):
        online.online_row([1.0, 2.0], vals)
    assert np.array_equal(online.online_row(np.zeros(0), np.zeros((0, 2))), np.zeros(2))
    assert np.array_equal(online.online_row([-np.inf] * 3, vals), np.zeros(2))
    out = online.online_row([-np.inf, -np.inf, 1.0, 2.0], np.arange(8.0).reshape(4, 2), 2)
    assert np.all(np.isfinite(out))


@pytest.mark.parametrize("tile", [1, 2, 5, 16])
def test_online_row_matches_ref(tile):
    r = _rng(16 + tile)
    for _ in range(5):
        s = r.standard_normal(37) * 5
        s[r.random(37) < 0.3] = -np.inf
        vals = r.standard_normal((37, 3))
        p, _ = ref.row_softmax(s[None, :])
        assert np.max(np.abs(online.online_row(s, vals, tile) - (p @ vals)[0])) <= 1e-14


def test_tiled_attention_masks_and_causal():
    q, k, v, mask = _tiny_case(17, 1, 1, 40, 4, True, True)
    o_t, l_t, _ = online.tiled_attention(q[0, 0], k[0, 0], v[0, 0], 0.5, 16, 8, True, mask[0, 0])
    o, l = ref.forward_head(q[0, 0], k[0, 0], v[0, 0], 0.5, True, mask[0, 0])
    assert np.max(np.abs(o_t - o)) <= 1e-14
    assert np.array_equal(np.isfinite(l_t), np.isfinite(l))


# ------------------------------------------------------------------ backward
def _loss(q, k, v, do, scale, causal, mask):
    o, _ = ref.attention_forward(q, k, v, scale, causal, mask)
    return float((o * do).sum())


@pytest.mark.parametrize("causal,masked", [(False, False), (True, False), (True, True)])
def test_backward_finite_differences(causal, masked):
    q, k, v, mask = _tiny_case(21 + causal + 2 * masked, 1, 2, 6, 3, causal, masked)
    do = _rng(22).standard_normal(q.shape)
    scale = 0.8
    dq, dk, dv, _ = ref.attention_backward(q, k, v, do, scale, causal, mask)
    h = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + h
            up = _loss(q, k, v, do, scale, causal, mask)
            x[idx] = old - h
            dn = _loss(q, k, v, do, scale, causal, mask)
            x[idx] = old
            num[idx] = (up - dn) / (2 * h)
        assert np.max(np.abs(num - g)) <= 1e-7


def test_backward_invariants():
    q, k, v, mask = _tiny_case(23, 2, 2, 33, 5, True, True)
    do = _rng(24).standard_normal(q.shape)
    dq, dk, dv, D = ref.attention_backward(q, k, v, do, 0.6, True, mask)
    assert np.max(np.abs(dk.sum(axis=2))) <= 1e-12
    _, lse = ref.attention_forward(q, k, v, 0.6, True, mask)
    live = np.isfinite(lse)
    want = np.where(live[..., None], do, 0.0).sum(axis=2)
    assert np.max(np.abs(dv.sum(axis=2) - want)) <= 1e-12
    dead = ~live
    assert dead.any()
    assert np.all(dq[dead] == 0) and np.all(D[dead] == 0)


def test_backward_head_sampling_matches_full():
    q, k, v, mask = _tiny_case(25, 1, 1, 300, 6, True, True)
    do = _rng(26).standard_normal(q.shape)
    dq, dk, dv, D = ref.attention_backward(q, k, v, do, 0.4, True, mask)
    qr, kr = [3, 150, 299], [0, 7, 298]
    sq, sk, sv, sD, _ = ref.backward_head(q[0, 0], k[0, 0], v[0, 0], do[0, 0], 0.4, True, mask[0, 0], qr, kr)
    assert np.max(np.abs(sq - dq[0, 0, qr])) <= 1e-13
    assert np.max(np.abs(sk - dk[0, 0, kr])) <= 1e-13
    assert np.max(np.abs(sv - dv[0, 0, kr])) <= 1e-13
    assert np.max(np.abs(sD - D[0, 0])) <= 1e-13
    o, l = ref.forward_head(q[0, 0], k[0, 0], v[0, 0], 0.4, True, mask[0, 0], rows=qr)
    of, lf = ref.attention_forward(q, k, v, 0.4, True, mask)
    assert np.array_equal(o, of[0, 0, qr]) and np.array_equal(l, lf[0, 0, qr])


# --------------------------------------------------- planted oracle mistakes
def _wrong_causal(qh, kh, rows, scale, causal, maskh):
    s = scale * (qh[rows] @ kh.T)
    if maskh is not None:
        s = s + maskh[rows]
    if causal:
        keys = np.arange(kh.shape[0])
        s = np.where(keys[None, :] >= rows[:, None], -np.inf, s)  # off by one
    return s


def _no_scale(qh, kh, rows, scale, causal, maskh):
    s = qh[rows] @ kh.T
    if maskh is not None:
        s = s + maskh[rows]
    if causal:
        keys = np.arange(kh.shape[0])
        s = np.where(keys[None, :] > rows[:, None], -np.inf, s)
    return s


def _transposed(qh, kh, rows, scale, causal, maskh):
    s = scale * (kh[rows] @ qh.T)
    if maskh is not None:
        s = s + maskh[rows]
    if causal:
        keys = np.arange(kh.shape[0])
        s = np.where(keys[None, :] > rows[:, None], -np.inf, s)
    return s


def _mask_sign(qh, kh, rows, scale, causal, maskh):
    s = scale * (qh[rows] @ kh.T)
    if maskh is not None:
        s = s - np.where(np.isneginf(maskh[rows]), np.inf, maskh[rows])
    if causal:
        keys = np.arange(kh.shape[0])
        s = np.where(keys[None, :] > rows[:, None], -np.inf, s)
    return s


@pytest.mark.parametrize("mutant", [_wrong_causal, _no_scale, _transposed, _mask_sign])
def test_planted_mistakes_are_caught(monkeypatch, mutant):
    q, k, v, mask = _tiny_case(27, 1, 2, 7, 3, True, True)
    o_b, _ = brute_attention(q, k, v, 0.7, True, mask)
    monkeypatch.setattr(ref, "head_scores", mutant)
    o, _ = ref.attention_forward(q, k, v, 0.7, True, mask)
    assert np.max(np.abs(o - o_b)) > 1e-6


def test_dropped_D_term_is_caught():
    q, k, v, mask = _tiny_case(28, 1, 1, 5, 3, True, False)
    do = _rng(29).standard_normal(q.shape)
    good = ref.attention_backward(q, k, v, do, 0.8, True)[0]
    # a backward whose dS drops the -D term no longer matches finite differences
    h = 1e-6
    idx = (0, 0, 3, 1)
    x = q.copy()
    x[idx] += h
    up = _loss(x, k, v, do, 0.8, True, None)
    x[idx] -= 2 * h
    dn = _loss(x, k, v, do, 0.8, True, None)
    num = (up - dn) / (2 * h)
    assert abs(num - good[idx]) <= 1e-7
    p, _ = ref.row_softmax(ref.head_scores(q[0, 0], k[0, 0], np.arange(5), 0.8, True, None))
    dp = do[0, 0] @ v[0, 0].T
    wrong = 0.8 * ((p * dp) @ k[0, 0])
    assert abs(num - wrong[3, 1]) > 1e-4


# ----------------------------------------------------------- page arithmetic
def test_byte_accounting():
    g = _golden("byte_accounting.json")
    sc, io, tot = arith.materialising_bytes(g["N"], g["d"], g["elem_bytes"])
    assert sc == g["score_transfers_bytes"]
    assert io == g["qkvo_min_bytes"]
    assert tot == g["total_bytes"]
    assert tot == g["total_mib"] * arith.MiB
    assert round(arith.bandwidth_floor_seconds(tot, g["bandwidth_bytes_per_s"]), 6) == g["floor_seconds_printed"]
    assert tot // io == g["ratio_to_io_min_printed"]
    assert round(arith.matmul_flops(g["N"], g["d"]) / 1e9, 2) == g["matmul_gflops_printed"]


def test_size_figures():
    g = _golden("size_figures.json")
    assert arith.score_matrix_bytes(8192) == g["score_matrix_8192_fp16_mib"] * arith.MiB
    assert arith.score_matrix_bytes(8192, 32) == g["score_matrix_8192_x32_heads_gib"] * arith.GiB
    assert arith.score_matrix_bytes(131072) == g["score_matrix_131072_gib"] * arith.GiB
    assert arith.score_matrix_bytes(8192, elem=1) == g["score_elements_8192"]
    assert arith.score_row_bytes(8192) == g["score_row_8192_kib"] * 1024
    assert arith.score_matrix_bytes(4 * 8192) == 16 * arith.score_matrix_bytes(8192)
    assert arith.row_stats_bytes(8192) == g["row_stats_8192_fp32_bytes"]
    bc, br = arith.algorithm1_blocks(g["algorithm1_M"], g["algorithm1_d"])
    assert (bc, br) == (g["algorithm1_key_block"], g["algorithm1_query_block"])
    assert round(arith.theorem2_ratio(8192, 128, g["algorithm1_M"]), 1) == g["theorem2_ratio_printed"]


def test_panel_reading():
    p = _golden("size_figures.json")["panel"]
    sc, io, tot = arith.panel_standard_traffic(p["N"], p["heads"], p["d"])
    # 16.25 GiB, printed to one decimal rounding half up
    assert abs(tot / arith.GiB - p["standard_traffic_gib_printed"]) <= 0.05 + 1e-12
    assert round(sc / arith.GiB, 1) == p["score_traffic_gib_printed"]
    assert io == p["qkvo_mib_printed"] * arith.MiB
    assert arith.panel_peak_intermediate(p["N"], p["heads"], p["d"], False) == p["peak_standard_gib_printed"] * arith.GiB
    assert round(arith.panel_peak_intermediate(p["N"], p["heads"], p["d"], True) / arith.MiB, 1) == p["peak_flash_mib_printed"]
    n2 = p["N_long"]
    assert arith.panel_peak_intermediate(n2, p["heads"], p["d"], False) == p["peak_standard_long_gib_printed"] * arith.GiB
    assert arith.panel_peak_intermediate(n2, p["heads"], p["d"], True) == p["peak_flash_long_mib_printed"] * arith.MiB


def test_flops_formula():
    assert arith.attention_flops(1, 1, 8192, 128) == 4 * 8192**2 * 128
    assert arith.attention_flops(2, 32, 8192, 128, causal=True) == 2 * 32 * 8192**2 * 128 * 2
    assert arith.attention_flops(1, 1, 8, 2, causal=True, backward=True) == 2.5 * 4 * 64 * 2 / 2


# ------------------------------------------------------ stored-output model
def test_round_bf16_matches_torch():
    r = _rng(31)
    x = np.concatenate([r.standard_normal(20000) * 10.0 ** r.integers(-6, 6, 20000),
                        [0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, np.inf, -np.inf]])
    # exact ties in fp32 (low 16 bits == 0x8000) must round to even
    ties = (np.arange(1, 200, dtype=np.uint32) << 16) | 0x3F800000 | 0x8000
    x = np.concatenate([x, ties.view(np.float32).astype(np.float64)])
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    got = ref.round_bf16(x)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


def test_backward_with_stored_bf16_output():
    q, k, v, mask = _tiny_case(32, 1, 2, 40, 8, True, True)
    do = _rng(33).standard_normal(q.shape)
    dq, dk, dv, D = ref.attention_backward(q, k, v, do, 0.5, True, mask)
    dq2, dk2, dv2, D2 = ref.attention_backward(q, k, v, do, 0.5, True, mask, o_storage="bf16")
    o, _ = ref.attention_forward(q, k, v, 0.5, True, mask)
    assert np.allclose(D2, (do * ref.round_bf16(o)).sum(-1), rtol=0, atol=1e-12)
    assert np.array_equal(dv, dv2)  # dV does not involve D
    # dQ and dK move by the D perturbation only: dS changes by -P * (D2 - D)
    assert 0 < np.max(np.abs(dq2 - dq)) < 0.05 * np.max(np.abs(dq))
    with pytest.raises(ValueError):
        ref.attention_backward(q, k, v, do, 0.5, True, mask, o_storage="fp8")


def test_round_f16_ties_overflow_and_subnormals():
    # IEEE half: 10 fraction bits, largest finite 65504, smallest subnormal 2^-24
    u = 2.0 ** -10  # spacing just above 1
    cases = [
        (1.0 + u / 2, 1.0),                    # tie between 1 and 1+u: to even (1)
        (1.0 + 3 * u / 2, 1.0 + 2 * u),        # tie between 1+u and 1+2u: to even (1+2u)
        (1.0 + u / 2 + 2.0 ** -20, 1.0 + u),   # just above the tie: up
        (65504.0, 65504.0),
        (65519.0, 65504.0),                    # below the midpoint to 65536: stays finite
        (65520.0, np.inf),                     # the midpoint rounds to even, i.e. overflows
        (-70000.0, -np.inf),
        (2.0 ** -25, 0.0),                     # tie between 0 and 2^-24: to even (0)
        (3 * 2.0 ** -25, 2.0 ** -23),          # tie between 2^-24 and 2^-23: to even (2^-23)
        (2.0 ** -24, 2.0 ** -24),
        (0.1, 1638.0 / 16384.0),               # 0.1 = 1.6 * 2^-4 -> 1.599609375 * 2^-4
    ]
    x = np.array([c[0] for c in cases])
    want = np.array([c[1] for c in cases])
    assert np.array_equal(ref.round_f16(x), want)


def test_backward_with_stored_f16_output():
    q, k, v, mask = _tiny_case(34, 1, 2, 40, 8, True, True)
    do = _rng(35).standard_normal(q.shape)
    dq, dk, dv, D = ref.attention_backward(q, k, v, do, 0.5, True, mask)
    dq2, dk2, dv2, D2 = ref.attention_backward(q, k, v, do, 0.5, True, mask, o_storage="f16")
    o, _ = ref.attention_forward(q, k, v, 0.5, True, mask)
    assert np.allclose(D2, (do * ref.round_f16(o)).sum(-1), rtol=0, atol=1e-12)
    assert np.array_equal(dv, dv2)
    # half keeps 3 more fraction bits than bf16: the D perturbation is about 8x smaller
    _, _, _, D3 = ref.attention_backward(q, k, v, do, 0.5, True, mask, o_storage="bf16")
    assert np.max(np.abs(D2 - D)) < np.max(np.abs(D3 - D))


# ------------------------------------------------------------------ decode
def test_decode_square_causal_is_the_causal_forward():
    # with nq = nk the bottom-right causal alignment is the ordinary one
    q, k, v, _ = _tiny_case(40, 2, 2, 24, 8, False, False)
    o1, l1 = ref.decode_forward(q, k, v, 0.3, causal=True)
    o2, l2 = ref.attention_forward(q, k, v, 0.3, causal=True)
    assert np.allclose(o1, o2, rtol=0, atol=1e-14) and np.allclose(l1, l2, rtol=0, atol=1e-14)


def test_decode_rows_are_the_last_rows_of_a_causal_forward():
    # nq query rows appended to a prefix: decode of those rows = the last rows of the causal
    # forward over prefix + rows
    r = _rng(41)
    B, H, nk, nq, d = 1, 2, 37, 5, 8
    qf = r.standard_normal((B, H, nk, d))
    k = r.standard_normal((B, H, nk, d))
    v = r.standard_normal((B, H, nk, d))
    o_full, l_full = ref.attention_forward(qf, k, v, 0.4, causal=True)
    o, l = ref.decode_forward(qf[:, :, nk - nq:], k, v, 0.4, causal=True)
    assert np.allclose(o, o_full[:, :, nk - nq:], rtol=0, atol=1e-14)
    assert np.allclose(l, l_full[:, :, nk - nq:], rtol=0, atol=1e-14)


def test_decode_brute_force_and_unseen_rows():
    r = _rng(42)
    nq, nk, d = 6, 4, 3
    q, k, v = r.standard_normal((1, 1, nq, d)), r.standard_normal((1, 1, nk, d)), r.standard_normal((1, 1, nk, d))
    for causal in (False, True):
        o, lse = ref.decode_forward(q, k, v, 0.7, causal)
        for i in range(nq):
            keys = [j for j in range(nk) if not causal or j <= nk - nq + i]
            if not keys:  # nq > nk: the first rows see no key
                assert np.all(o[0, 0, i] == 0) and np.isneginf(lse[0, 0, i])
                continue
            s = [0.7 * sum(q[0, 0, i, t] * k[0, 0, j, t] for t in range(d)) for j in keys]
            mx = max(s)
            w = [math.exp(x - mx) for x in s]
            want = [sum(w[a] * v[0, 0, j, t] for a, j in enumerate(keys)) / sum(w) for t in range(d)]
            assert np.allclose(o[0, 0, i], want, rtol=0, atol=1e-13)
            assert abs(lse[0, 0, i] - (mx + math.log(sum(w)))) < 1e-13


def test_merged_states_equal_the_whole_row():
    r = _rng(43)
    s = r.standard_normal(50) * 3
    s[10:14] = -np.inf
    vals = r.standard_normal((50, 4))
    whole = online.RowState(4)
    whole.absorb(s, vals)
    for cut in (0, 1, 13, 25, 49, 50):
        a, b = online.RowState(4), online.RowState(4)
        if cut > 0:
            a.absorb(s[:cut], vals[:cut])
        if cut < 50:
            b.absorb(s[cut:], vals[cut:])
        m = online.merge_states(a, b)
        assert abs(m.m - whole.m) == 0
        assert abs(m.l - whole.l) < 1e-12 * whole.l
        assert np.allclose(m.result(), whole.result(), rtol=0, atol=1e-14)
    empty = online.RowState(4)
    e = online.merge_states(empty, online.RowState(4))
    assert np.isneginf(e.m) and e.l == 0 and np.all(e.result() == 0)


# ------------------------------------------------------------------ FP8 (E4M3) forward
def test_decode_e4m3_matches_torch_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    got = ref.decode_e4m3(codes)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_decode_e4m3_closed_forms():
    d = lambda c: float(ref.decode_e4m3(np.array([c], dtype=np.uint8))[0])  # noqa: E731
    assert d(0x00) == 0.0 and math.copysign(1.0, d(0x80)) == -1.0
    assert d(0x01) == 2.0 ** -9 and d(0x07) == 7 * 2.0 ** -9  # subnormals
    assert d(0x08) == 2.0 ** -6  # smallest normal
    assert d(0x38) == 1.0 and d(0x3C) == 1.5 and d(0x40) == 2.0 and d(0xB8) == -1.0
    assert d(0x7E) == 448.0 and d(0xFE) == -448.0 and d(0x77) == 240.0
    assert math.isnan(d(0x7F)) and math.isnan(d(0xFF))


def test_fp8_forward_is_attention_of_the_values_the_codes_stand_for():
    # codes 0x30..0x47 stand for 0.5 .. 3.75 in steps the bf16 format holds exactly, so the
    # FP8 forward must equal the plain forward of those values times the descales
    rng = np.random.default_rng(5)
    shape = (1, 2, 37, 8)
    q8, k8, v8 = (rng.integers(0x30, 0x48, size=shape).astype(np.uint8) for _ in range(3))
    signs = [np.where(rng.random(shape) < 0.5, 0x80, 0).astype(np.uint8) for _ in range(3)]
    q8, k8, v8 = q8 | signs[0], k8 | signs[1], v8 | signs[2]
    qd, kd, vd = 0.25, 0.5, 2.0
    for causal in (False, True):
        o, lse = ref.attention_forward_fp8(q8, k8, v8, qd, kd, vd, 0.3, causal)
        qv = torch.from_numpy(q8).view(torch.float8_e4m3fn).double() * qd
        kv = torch.from_numpy(k8).view(torch.float8_e4m3fn).double() * kd
        vv = torch.from_numpy(v8).view(torch.float8_e4m3fn).double() * vd
        want = torch.nn.functional.scaled_dot_product_attention(qv, kv, vv, scale=0.3, is_causal=causal)
        assert np.allclose(o, want.numpy(), rtol=0, atol=1e-13)
        # a single key: O is that key's value row
    o1, _ = ref.attention_forward_fp8(q8[:, :, :1], k8[:, :, :1], v8[:, :, :1], qd, kd, vd, 0.3)
    assert np.array_equal(o1, ref.decode_e4m3(v8[:, :, :1]) * vd)
