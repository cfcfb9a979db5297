"""Pins of the CPU oracle to things other than itself (CPU only).

Each test checks the oracle against what the pages or the mathematics fix:
brute-force enumeration of the rank definition, exact rational arithmetic on
integer data, closed forms, special cases that reduce to a library routine
(torch's scaled_dot_product_attention in float64), and the worked examples the
pages print (tests/golden). A plausible slip in the oracle — a dropped scale,
a flipped tie-break, an off-by-one causal edge, a transposed operand, a missing
max-subtraction — fails at least one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from workloads import WORKLOADS, make_scorer_inputs, plant_groups, plant_positions, small
from workloads.gen import PLANT_DIMS, PLANT_GROUPS

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_int(shape, seed):
    g = np.random.default_rng(seed)
    return g.integers(-4, 5, size=shape).astype(np.float64)


def _brute_topk(S, valid, k):
    """Rank definition: key j's rank is the number of valid keys beating it
    (higher score, or equal score and lower index). Selected iff rank < k;
    output slot = rank. Returns idx [k] padded with -1."""
    n = len(S)
    out = [-1] * k
    for j in range(n):
        if not valid[j]:
            continue
        rank = 0
        for jj in range(n):
            if valid[jj] and (S[jj] > S[j] or (S[jj] == S[j] and jj < j)):
                rank += 1
        if rank < k:
            out[rank] = j
    return out


@pytest.mark.parametrize("Tq,Tk,P,k,causal", [
    (9, 9, 16, 4, False), (13, 13, 16, 5, True), (7, 20, 32, 6, True),
    (20, 7, 16, 3, True), (16, 16, 64, 16, False), (31, 48, 16, 48, True),
])
def test_topk_brute_force_integer(Tq, Tk, P, k, causal):
    """Exact: integer data, scores as Fractions, selection by the rank definition."""
    q = _rand_int((Tq, P), 1 + Tq)
    kl = _rand_int((Tk, P), 2 + Tk)
    idx, sc = oracle.topk_rows(q, np.arange(Tq), kl, k, Tq, causal)
    r = math.isqrt(P)
    for i in range(Tq):
        dots = [int(np.dot(q[i].astype(np.int64), kl[j].astype(np.int64))) for j in range(Tk)]
        if r * r == P:   # scale 1/r is exact: scores are exact rationals
            S = [Fraction(d, r) for d in dots]
        else:            # scale rounded to fp32, product rounded to fp32
            S = [Fraction(float(np.float32(d) * np.float32(1.0 / math.sqrt(P)))) for d in dots]
        valid = [(not causal) or (j <= i + (Tk - Tq)) for j in range(Tk)]
        want = _brute_topk(S, valid, k)
        assert list(idx[i]) == want, (i, list(idx[i]), want)
        for t, j in enumerate(want):
            if j >= 0:
                assert Fraction(float(sc[i, t])) == S[j]
            else:
                assert sc[i, t] == -np.inf


def test_topk_brute_force_float():
    """Continuous data: selection matches the rank definition on scores formed
    by a library matmul (fp64), rounded to fp32 and scaled in fp32."""
    g = np.random.default_rng(7)
    Tq, Tk, P, k = 24, 40, 32, 10
    q = g.standard_normal((Tq, P))
    kl = g.standard_normal((Tk, P))
    idx, sc = oracle.topk_rows(q, np.arange(Tq), kl, k, Tq, True)
    S = (q @ kl.T).astype(np.float32) * np.float32(1.0 / math.sqrt(P))
    for i in range(Tq):
        valid = [j <= i + (Tk - Tq) for j in range(Tk)]
        assert list(idx[i]) == _brute_topk(list(S[i]), valid, k)


def test_topk_scale_and_order_invariants():
    w = small("topk_f32_t1024_k32", Tq=64, Tk=300, k=40)
    q, kl = make_scorer_inputs(w)
    idx, sc = oracle.score_topk(q, kl, w.k, causal=False)
    qd, kd = q.double().numpy(), kl.double().numpy()
    for h in range(w.H):
        for i in range(w.Tq):
            S = (qd[0, h, i] @ kd[0, h].T) / 4.0   # P = 16: scale exactly 1/4
            ids = idx[0, h, i]
            assert len(set(ids.tolist())) == w.k
            np.testing.assert_array_equal(sc[0, h, i], S[ids].astype(np.float32))
            # sorted (score desc, index asc)
            for a, b in zip(ids[:-1], ids[1:]):
                assert S[a] > S[b] or (S[a] == S[b] and a < b)
            # every unselected key is beaten by the last selected one
            last = ids[-1]
            rest = np.setdiff1d(np.arange(w.Tk), ids)
            assert np.all((S[rest] < S[last]) | ((S[rest] == S[last]) & (rest > last)))


def test_topk_second_routine_on_the_fp32_workload():
    """A second, independent selection on the whole fp32 workload
    (B1 H2 T1024, d_proj 16, k 32, integer data): int64 dot products by a
    library matmul, then a stable lexicographic sort on (-score, index). The
    scale 16^-0.5 = 1/4 is exact, so ranking the integer dots is ranking the
    scores; the oracle must agree bit for bit, scores included."""
    w = WORKLOADS["topk_f32_t1024_k32"]
    q, kl = make_scorer_inputs(w)
    idx, sc = oracle.score_topk(q, kl, w.k, w.causal)
    qi = q.numpy().astype(np.int64)
    ki = kl.numpy().astype(np.int64)
    assert np.array_equal(qi, q.numpy()) and np.array_equal(ki, kl.numpy())   # integer data
    for b in range(w.B):
        for h in range(w.H):
            dots = qi[b, h] @ ki[b, h].T                     # [Tq, Tk], exact
            j = np.arange(w.Tk)
            for i in range(w.Tq):
                order = np.lexsort((j, -dots[i]))            # last key is primary
                top = order[:w.k]
                np.testing.assert_array_equal(idx[b, h, i], top.astype(np.int32))
                np.testing.assert_array_equal(sc[b, h, i], (dots[i, top] / 4.0).astype(np.float32))


def test_topk_all_ties_lower_index_wins():
    Tq, Tk, k = 10, 50, 7
    q = np.zeros((Tq, 16))
    kl = _rand_int((Tk, 16), 3)
    idx, sc = oracle.topk_rows(q, np.arange(Tq), kl, k, Tq, False)
    assert (idx == np.arange(k)[None, :]).all()
    assert (sc == 0).all()
    idx, _ = oracle.topk_rows(q, np.arange(Tq), kl, k, Tq, True)   # causal, Tq < Tk
    for i in range(Tq):
        nv = min(i + (Tk - Tq) + 1, Tk)
        want = list(range(min(k, nv))) + [-1] * max(0, k - nv)
        assert list(idx[i]) == want


def test_topk_k_exceeds_valid_pads():
    Tq = Tk = 12
    q = _rand_int((Tq, 16), 4)
    kl = _rand_int((Tk, 16), 5)
    k = 20
    idx, sc = oracle.topk_rows(q, np.arange(Tq), kl, k, Tq, True)
    for i in range(Tq):
        sel = idx[i][idx[i] >= 0]
        assert sorted(sel.tolist()) == list(range(i + 1))      # every valid key, nothing else
        assert (idx[i][i + 1:] == -1).all() and np.isneginf(sc[i][i + 1:]).all()


def test_topk_rows_with_no_valid_key():
    """Causal with Tq > Tk: the first Tq - Tk queries see no key at all."""
    Tq, Tk = 8, 5
    q = _rand_int((Tq, 16), 6)
    kl = _rand_int((Tk, 16), 7)
    idx, _ = oracle.topk_rows(q, np.arange(Tq), kl, 3, Tq, True)
    assert (idx[:Tq - Tk] == -1).all()
    assert idx[Tq - Tk][0] == 0 and (idx[Tq - Tk][1:] == -1).all()


def test_planted_keys_boost_exactly_64():
    w = WORKLOADS["topk_causal_bf16_t128k_k512_planted"].with_(H=2, Tq=2048, Tk=2048, planted=16)
    q, kl = make_scorer_inputs(w)
    grp = plant_groups(w)
    pos = plant_positions(w)
    base = w.P - PLANT_GROUPS * PLANT_DIMS
    qd, kd = q.double(), kl.double()
    for h in range(w.H):
        for i in [0, 5, 1000, 2047]:
            g = int(grp[0, h, i])
            full = kd[0, h] @ qd[0, h, i]
            rand = kd[0, h, :, :base] @ qd[0, h, i, :base]
            boost = full - rand
            planted = set(pos[0, h, g].tolist())
            for j in range(w.Tk):
                assert boost[j] == (64.0 if j in planted else 0.0)
    # integer range of every element
    assert q.abs().max() <= 4 and kl.abs().max() <= 4


def _sdpa(Q, K, V, mask=None, scale=None, causal=False):
    """torch's scaled_dot_product_attention in float64 (library routine)."""
    return F.scaled_dot_product_attention(
        torch.as_tensor(Q, dtype=torch.float64)[None, None],
        torch.as_tensor(K, dtype=torch.float64)[None, None],
        torch.as_tensor(V, dtype=torch.float64)[None, None],
        attn_mask=None if mask is None else torch.as_tensor(mask)[None, None],
        is_causal=causal, scale=scale)[0, 0].numpy()


def test_attn_full_selection_equals_dense_sdpa():
    g = np.random.default_rng(11)
    T, D = 37, 64
    Q, K, V = (g.standard_normal((T, D)) for _ in range(3))
    idx = np.tile(np.arange(T, dtype=np.int32), (T, 1))
    O, bad = oracle.attn_rows(Q, K, V, idx)
    assert bad == 0
    np.testing.assert_allclose(O, _sdpa(Q, K, V), rtol=0, atol=1e-12)


def test_attn_causal_full_topk_equals_causal_sdpa():
    g = np.random.default_rng(12)
    T, D = 29, 32
    Q, K, V = (g.standard_normal((T, D)) for _ in range(3))
    ql, kl = _rand_int((T, 16), 8), _rand_int((T, 16), 9)
    idx, _ = oracle.topk_rows(ql, np.arange(T), kl, T, T, True)
    O, _ = oracle.attn_rows(Q, K, V, idx)
    np.testing.assert_allclose(O, _sdpa(Q, K, V, causal=True), rtol=0, atol=1e-12)


def test_attn_equals_masked_dense():
    """Sparse attention over idx equals dense attention under the boolean mask built from idx."""
    g = np.random.default_rng(13)
    Tq, Tk, D, k = 16, 64, 32, 9
    Q = g.standard_normal((Tq, D))
    K, V = g.standard_normal((Tk, D)), g.standard_normal((Tk, D))
    idx = np.stack([g.choice(Tk, size=k, replace=False) for _ in range(Tq)]).astype(np.int32)
    mask = np.zeros((Tq, Tk), dtype=bool)
    for i in range(Tq):
        mask[i, idx[i]] = True
    O, _ = oracle.attn_rows(Q, K, V, idx)
    np.testing.assert_allclose(O, _sdpa(Q, K, V, mask=mask), rtol=0, atol=1e-12)


def test_attn_closed_forms():
    g = np.random.default_rng(14)
    Tk, D = 40, 16
    Q = g.standard_normal((5, D)) * 3
    K, V = g.standard_normal((Tk, D)), g.standard_normal((Tk, D))
    # k = 1: the single selected value row, exactly
    idx1 = np.array([[3], [0], [39], [17], [17]], dtype=np.int32)
    O, _ = oracle.attn_rows(Q, K, V, idx1)
    np.testing.assert_array_equal(O, V[idx1[:, 0]])
    # constant V rows: output is that constant
    Vc = np.tile(g.standard_normal(D), (Tk, 1))
    idx = np.stack([g.choice(Tk, 8, replace=False) for _ in range(5)]).astype(np.int32)
    O, _ = oracle.attn_rows(Q, K, Vc, idx)
    np.testing.assert_allclose(O, np.tile(Vc[0], (5, 1)), rtol=0, atol=1e-14)
    # identical keys: uniform weights, output is the mean of the selected values
    Ke = np.tile(g.standard_normal(D), (Tk, 1))
    O, _ = oracle.attn_rows(Q, Ke, V, idx)
    np.testing.assert_allclose(O, np.stack([V[r].mean(0) for r in idx]), rtol=0, atol=1e-14)
    # permutation of the list changes nothing beyond rounding
    perm = idx[:, ::-1].copy()
    O1, _ = oracle.attn_rows(Q, K, V, idx)
    O2, _ = oracle.attn_rows(Q, K, V, perm)
    np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-13)


def test_attn_hand_example_and_list_semantics():
    # D = 1, scale 1: logits 0 and ln 3 -> weights 1/4 and 3/4
    K = np.array([[0.0], [math.log(3.0)], [5.0]])
    V = np.array([[2.0], [10.0], [-7.0]])
    q = np.array([[1.0]])
    O, _ = oracle.attn_rows(q, K, V, np.array([[0, 1]], np.int32), scale=1.0)
    assert abs(O[0, 0] - (0.25 * 2.0 + 0.75 * 10.0)) < 1e-14
    # -1 entries are skipped
    O2, _ = oracle.attn_rows(q, K, V, np.array([[0, -1, 1, -1]], np.int32), scale=1.0)
    assert O2[0, 0] == O[0, 0]
    # a repeated entry counts once per occurrence: weights 1:1:3 -> (2 + 2 + 30) / 5
    O3, _ = oracle.attn_rows(q, K, V, np.array([[0, 0, 1]], np.int32), scale=1.0)
    assert abs(O3[0, 0] - (2.0 + 2.0 + 3.0 * 10.0) / 5.0) < 1e-14
    # no valid entry: zeros; out-of-range entries are counted and skipped
    O4, bad = oracle.attn_rows(q, K, V, np.array([[-1, 7]], np.int32), scale=1.0)
    assert O4[0, 0] == 0.0 and bad == 1
    # default scale is head_dim^-0.5: D = 4 -> 1/2
    K4, V4 = np.array([[0.0] * 4, [1.0] * 4]), np.array([[0.0] * 4, [1.0] * 4])
    O5, _ = oracle.attn_rows(np.array([[1.0] * 4]), K4, V4, np.array([[0, 1]], np.int32))
    w1 = math.exp(2.0) / (1.0 + math.exp(2.0))   # logit 4 * 1/2 = 2
    np.testing.assert_allclose(O5[0], [w1] * 4, rtol=0, atol=1e-14)


def test_attn_large_logits_stable():
    """Max-subtraction: logits of order 1e3 must not overflow."""
    K = np.array([[1000.0], [999.0]])
    V = np.array([[1.0], [0.0]])
    O, _ = oracle.attn_rows(np.array([[1.0]]), K, V, np.array([[0, 1]], np.int32), scale=1.0)
    assert abs(O[0, 0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-14


@pytest.mark.parametrize("T,w", [(50, 3), (50, 0), (20, 25), (64, 7)])
def test_window_equals_band_masked_sdpa(T, w):
    g = np.random.default_rng(15 + T + w)
    D = 16
    Q, K, V = (g.standard_normal((T, D)) for _ in range(3))
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    mask = np.abs(i - j) <= w
    O = oracle.window_rows(Q, np.arange(T), K, V, w, w)
    np.testing.assert_allclose(O, _sdpa(Q, K, V, mask=mask), rtol=0, atol=1e-12)
    if w == 0:
        np.testing.assert_array_equal(O, V)
    if w >= T:
        np.testing.assert_allclose(O, _sdpa(Q, K, V), rtol=0, atol=1e-12)


def test_window_equals_sparse_band():
    g = np.random.default_rng(16)
    T, D, w = 40, 8, 4
    Q, K, V = (g.standard_normal((T, D)) for _ in range(3))
    Ow = oracle.window_rows(Q, np.arange(T), K, V, w, w)
    for i in range(T):
        band = np.arange(max(0, i - w), min(T - 1, i + w) + 1, dtype=np.int32)
        Os, _ = oracle.attn_rows(Q[i:i + 1], K, V, band[None, :])
        np.testing.assert_allclose(Ow[i], Os[0], rtol=0, atol=1e-14)


def test_golden_window_radius_example():
    """Worked example: radius 5 around token 100 covers positions 95..105."""
    gold = json.load(open(os.path.join(GOLDEN, "window_radius.json")))
    ex = gold["radius_example"]
    T, w, i = 400, ex["w"], ex["i"]
    # zero query: uniform weights; V_j = j and j^2 recover the key set's mean and second moment
    K = np.random.default_rng(17).standard_normal((T, 2))
    V = np.stack([np.arange(T, dtype=np.float64), np.arange(T, dtype=np.float64) ** 2], 1)
    Q = np.zeros((T, 2))
    O = oracle.window_rows(Q[i:i + 1], [i], K, V, w, w)
    keys = np.arange(ex["first_key"], ex["last_key"] + 1)
    assert len(keys) == 2 * w + 1
    np.testing.assert_allclose(O[0], [keys.mean(), (keys ** 2).mean()], rtol=1e-15)
    fx = gold["fraction_example"]
    assert round(100.0 * (2 * fx["w"] + 1) / fx["n"], 1) == fx["percent_one_decimal"]


def test_golden_selection_fraction_at_128k():
    """k = 512 of n = 128K keys is 0.4% of the dense row: the oracle's last row selects exactly k."""
    gold = json.load(open(os.path.join(GOLDEN, "selection_fraction.json")))
    w = WORKLOADS["topk_causal_bf16_t128k_k512_planted"].with_(H=1)
    assert (w.Tk, w.k) == (gold["n"], gold["k"])
    q, kl = make_scorer_inputs(w)
    i = w.Tq - 1
    idx, _ = oracle.topk_rows(q[0, 0, i:i + 1], [i], kl[0, 0], w.k, w.Tq, True)
    assert (idx >= 0).sum() == gold["k"]
    assert round(100.0 * (idx >= 0).sum() / gold["n"], 1) == gold["percent_one_decimal"]


# ------------------------------------------------------------ scorer alone

@pytest.mark.parametrize("Tq,Tk,P,causal,scale", [
    (9, 9, 16, False, 0.0), (7, 20, 64, True, 0.0), (20, 7, 64, True, 0.0),
    (12, 12, 32, True, 0.5),
])
def test_scores_equal_exact_integer_product(Tq, Tk, P, causal, scale):
    """Integer data: every score is an integer dot product (exact in int64)
    times a power-of-two scale, so the oracle must reproduce it exactly; keys
    outside the bottom-right causal band hold -inf."""
    q = _rand_int((Tq, P), 5 + Tq)
    kl = _rand_int((Tk, P), 6 + Tk)
    S = oracle.scores_rows(q, np.arange(Tq), kl, Tq, causal, scale)
    dots = q.astype(np.int64) @ kl.astype(np.int64).T
    sc = scale if scale > 0 else 1.0 / math.isqrt(P)     # P = 16, 64: exact powers of two
    for i in range(Tq):
        for j in range(Tk):
            if causal and j > i + (Tk - Tq):
                assert S[i, j] == -np.inf
            else:
                assert S[i, j] == dots[i, j] * sc


def test_scores_rank_like_the_selection():
    """The selection is the top of each score row: sorting a row of
    oracle.scores by (score desc, index asc) gives oracle.topk_rows."""
    Tq, Tk, P, k = 30, 50, 16, 12
    q = _rand_int((Tq, P), 11)
    kl = _rand_int((Tk, P), 12)
    S = oracle.scores_rows(q, np.arange(Tq), kl, Tq, True)
    idx, sc = oracle.topk_rows(q, np.arange(Tq), kl, k, Tq, True)
    for i in range(Tq):
        order = sorted((j for j in range(Tk) if S[i, j] > -np.inf), key=lambda j: (-S[i, j], j))
        want = (order + [-1] * k)[:k]
        assert list(idx[i]) == want


# ------------------------------------------------------ scorer projection
# The scorer's q_low / k_low come from bias-free linear layers d_model ->
# d_proj (mhpq.cn/news/1098205, section 2.2): out = x W^T with W in a linear
# layer's [d_proj][d_model] layout.

def test_project_selects_and_scales_columns():
    """Rows of W that are unit vectors (times a power of two) copy one column
    of x exactly; a transposed W or a wrong index would pick other columns."""
    rng = np.random.default_rng(11)
    x = rng.standard_normal((7, 64))
    perm = rng.permutation(64)[:40]
    W = np.zeros((40, 64))
    for p, c in enumerate(perm):
        W[p, c] = 2.0 ** (p % 5 - 2)
    out = oracle.lowrank_project(x, W)
    for p, c in enumerate(perm):
        assert np.array_equal(out[:, p], x[:, c] * 2.0 ** (p % 5 - 2))


def test_project_is_linear_in_the_weight_exactly():
    """Integer-valued inputs: every product and sum is exact in fp64, so
    x (W1 + W2)^T equals x W1^T + x W2^T to the last bit."""
    rng = np.random.default_rng(12)
    x = rng.integers(-4, 5, (9, 128)).astype(np.float64)
    W1 = rng.integers(-4, 5, (64, 128)).astype(np.float64)
    W2 = rng.integers(-4, 5, (64, 128)).astype(np.float64)
    assert np.array_equal(oracle.lowrank_project(x, W1 + W2),
                          oracle.lowrank_project(x, W1) + oracle.lowrank_project(x, W2))


def test_project_feeds_the_scorer_reassociated():
    """(x Wq^T)(x Wk^T)^T equals x (Wq^T Wk) x^T, computed in the other
    association by numpy on exact integers: pins the projection's layout
    (rows of W are output features) against an independent product, and its
    output against the scorer oracle that consumes it."""
    rng = np.random.default_rng(13)
    T, dm, P = 40, 64, 16
    x = rng.integers(-2, 3, (T, dm)).astype(np.float64)
    Wq = rng.integers(-2, 3, (P, dm)).astype(np.float64)
    Wk = rng.integers(-2, 3, (P, dm)).astype(np.float64)
    ql = oracle.lowrank_project(x, Wq)
    kl = oracle.lowrank_project(x, Wk)
    S_other = x @ (Wq.T @ Wk) @ x.T
    assert np.array_equal(ql @ kl.T, S_other)
    # the scorer oracle on these projections: fp64 dot rounded to fp32, times 1
    S = oracle.scores(torch.from_numpy(ql)[None, None], torch.from_numpy(kl)[None, None],
                      causal=False, scale=1.0)
    assert np.array_equal(np.asarray(S)[0, 0], S_other.astype(np.float32).astype(np.float64))


def test_round_bf16_nearest_even():
    """bf16 keeps 8 significant bits; ties go to the even significand."""
    v = [1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 0.75 * 2 ** -7, 257.0, 259.0, -3.0 - 2 ** -7,
         2 ** -100, 65504.0]
    want = [1.0, 1.0, 1.0 + 2 ** -6, 1.0 + 2 ** -7, 256.0, 260.0, -3.0, 2 ** -100, 65536.0]
    assert np.array_equal(oracle.round_bf16(v), np.array(want))
    # agrees with torch's own float64 -> bfloat16 conversion
    rng = np.random.default_rng(14)
    r = rng.standard_normal(4096) * 10.0 ** rng.integers(-6, 6, 4096)
    ref = torch.from_numpy(r).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.round_bf16(r), ref)


# ------------------------------------------------- selection variants
# mhpq.cn/news/1098205, section 4.2: a temperature divides the scores before
# the selection; boundary smoothing also selects the (k+1)-th key when it is
# within a threshold of the k-th.

def test_temperature_is_a_scale_and_keeps_the_selection():
    """scores / T with T > 0 is the scorer's scale times 1/T: on exact
    (integer) scores the selection is unchanged and the scores scale."""
    q = torch.from_numpy(_rand_int((1, 2, 64, 16), 77))
    kl = torch.from_numpy(_rand_int((1, 2, 300, 16), 78))
    i1, s1 = oracle.score_topk(q, kl, 24, True, scale=0.25)
    i2, s2 = oracle.score_topk(q, kl, 24, True, scale=2.5)   # the same with temperature 0.1
    assert np.array_equal(i1, i2)
    fin = np.isfinite(s1)
    assert np.array_equal(s2[fin], (s1[fin] * np.float32(10.0)).astype(np.float32))


def test_boundary_smoothing_hand_example():
    """Scores 5, 4, 3.95, 1 with k = 2: the third key joins when the gap
    0.05 is below the threshold, and not otherwise; equal scores always join
    for a positive threshold; a missing (k+1)-th key stays missing."""
    idx = np.array([[7, 3, 9, 1]], np.int32)[:, :3]
    sc = np.array([[5.0, 4.0, 3.95, 1.0]], np.float32)[:, :3]
    i, s = oracle.smooth_boundary(idx, sc, 2, 0.1)
    assert i.tolist() == [[7, 3, 9]] and s[0, 2] == np.float32(3.95)
    i, s = oracle.smooth_boundary(idx, sc, 2, 0.01)
    assert i.tolist() == [[7, 3, -1]] and s[0, 2] == -np.inf
    i, _ = oracle.smooth_boundary(np.array([[1, 2, 3]], np.int32),
                                  np.array([[2.0, 1.5, 1.5]], np.float32), 2, 1e-30)
    assert i.tolist() == [[1, 2, 3]]
    i, _ = oracle.smooth_boundary(np.array([[1, 2, -1]], np.int32),
                                  np.array([[2.0, 1.5, -np.inf]], np.float32), 2, 10.0)
    assert i.tolist() == [[1, 2, -1]]
    i, _ = oracle.smooth_boundary(idx, sc, 2, 0.0)   # threshold 0: the plain top-k
    assert i.tolist() == [[7, 3, -1]]


def test_boundary_smoothing_against_brute_force():
    """On exact integer scores the smoothed selection equals a direct
    enumeration: the top k by (score desc, index asc), plus the next key when
    its score is within delta of the k-th."""
    q = torch.from_numpy(_rand_int((1, 1, 20, 8), 79))
    kl = torch.from_numpy(_rand_int((1, 1, 60, 8), 80))
    k, delta = 5, 2.5
    i, s = oracle.score_topk(q, kl, k + 1, False, scale=1.0)
    i, s = oracle.smooth_boundary(i, s, k, delta)
    qn, kn = q.numpy()[0, 0], kl.numpy()[0, 0]
    for r in range(20):
        sc = qn[r] @ kn.T
        order = sorted(range(60), key=lambda j: (-sc[j], j))
        want = order[:k] + ([order[k]] if sc[order[k - 1]] - sc[order[k]] < delta else [])
        got = [int(j) for j in i[0, 0, r] if j >= 0]
        assert got == want
