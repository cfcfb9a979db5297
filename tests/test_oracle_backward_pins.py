"""Pins of the oracle's backward (straight-through estimator) to things other
than itself (CPU only).

The backward formulas in oracle.c are checked against:
- central finite differences of the forward oracle, which is pinned on its
  own in test_oracle_pins.py;
- torch autograd through float64 scaled_dot_product_attention, where the
  selection is every key (dense) or the causal prefix;
- the estimator's definition. A selected pair's score acts on the loss as a
  bias on that pair's attention logit. The bias is built from the forward
  oracle by widening Q and K with one extra column.
A dropped scale, a missing softmax-centering term, a transposed operand, a
duplicate key counted once or a gradient leaking to unselected keys each
fails one of them.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def _case(n, Tk, D, k, seed, pad=True, dup=True):
    g = np.random.default_rng(seed)
    Q = g.standard_normal((n, D))
    K = g.standard_normal((Tk, D))
    V = g.standard_normal((Tk, D))
    dO = g.standard_normal((n, D))
    idx = np.stack([g.choice(Tk, size=k, replace=False) for _ in range(n)]).astype(np.int32)
    if pad:
        idx[0, k - 1] = -1          # a padded slot
        idx[1, 1:] = -1             # a row with one key
        idx[2, :] = -1              # a row with none
    if dup:
        idx[3, 1] = idx[3, 0]       # a repeated key counts once per entry
    return Q, K, V, dO, idx


def _loss(Q, K, V, idx, dO, scale):
    """sum(O * dO) from the forward oracle. When Q and K carry extra columns
    (a logit bias), V gets zero columns to match and they are dropped from O."""
    D = dO.shape[1]
    if Q.shape[1] > D:
        V = np.hstack([V, np.zeros((V.shape[0], Q.shape[1] - D))])
    O, _ = oracle.attn_rows(Q, K, V, idx, scale, nthreads=1)
    return float(np.sum(O[:, :D] * dO))


def _fd(f, X, h=1e-6):
    """Central differences of the scalar f over every entry of X (modified in place, restored)."""
    G = np.zeros_like(X)
    for e in np.ndindex(X.shape):
        x0 = X[e]
        X[e] = x0 + h
        fp = f()
        X[e] = x0 - h
        fm = f()
        X[e] = x0
        G[e] = (fp - fm) / (2 * h)
    return G


@pytest.mark.parametrize("scale", [0.0, 0.37])
def test_attn_bwd_matches_finite_differences(scale):
    Q, K, V, dO, idx = _case(6, 9, 4, 5, seed=11)
    c = scale if scale > 0 else 4 ** -0.5
    dQ, dK, dV, dS, bad = oracle.attn_bwd_rows(Q, K, V, idx, dO, scale, nthreads=2)
    assert bad == 0
    f = lambda: _loss(Q, K, V, idx, dO, c)  # noqa: E731
    np.testing.assert_allclose(dQ, _fd(f, Q), atol=1e-7, rtol=1e-6)
    np.testing.assert_allclose(dK, _fd(f, K), atol=1e-7, rtol=1e-6)
    np.testing.assert_allclose(dV, _fd(f, V), atol=1e-7, rtol=1e-6)


def test_pair_gradient_is_the_logit_gradient():
    """dS[i][t] summed over the slots that hold key j is the derivative of the
    loss with respect to a bias on the logit of the pair (i, j). The bias is
    c * eps, entering through an extra column: eps on row i of Q and 1 on key j
    of K."""
    n, Tk, D, k = 6, 9, 4, 5
    Q, K, V, dO, idx = _case(n, Tk, D, k, seed=12)
    c = 0.41
    _, _, _, dS, _ = oracle.attn_bwd_rows(Q, K, V, idx, dO, c, nthreads=1)
    for i in range(n):
        for j in range(Tk):
            u = np.zeros((Tk, 1))
            u[j] = 1.0
            Kx = np.hstack([K, u])

            def f(eps):
                Qx = np.hstack([Q, np.zeros((n, 1))])
                Qx[i, D] = eps
                return _loss(Qx, Kx, V, idx, dO, c)

            h = 1e-6
            fd = (f(h) - f(-h)) / (2 * h) / c
            want = sum(dS[i, t] for t in range(k) if idx[i, t] == j)
            assert abs(fd - want) < 1e-7 + 1e-6 * abs(want), (i, j, fd, want)


def test_scorer_bwd_is_the_gradient_of_a_score_bias():
    """The straight-through estimator, end to end: adding
    S = sigma * q_low . k_low to the logits of the selected pairs (one extra
    block of columns in Q and K) and differentiating at zero perturbation
    gives the scorer's gradients."""
    n, Tk, D, k, P = 6, 9, 4, 5, 3
    Q, K, V, dO, idx = _case(n, Tk, D, k, seed=13)
    g = np.random.default_rng(14)
    ql = g.standard_normal((n, P))
    kl = g.standard_normal((Tk, P))
    c, sigma = 0.5, 0.3
    _, _, _, dS, _ = oracle.attn_bwd_rows(Q, K, V, idx, dO, c, nthreads=1)
    dq, dk = oracle.scorer_bwd_rows(ql, kl, idx, dS, sigma)
    # q_low perturbed: Q' = [Q, (sigma / c) * dq_pert], K' = [K, k_low]
    dqp = np.zeros((n, P))
    Kx = np.hstack([K, kl])
    f = lambda: _loss(np.hstack([Q, (sigma / c) * dqp]), Kx, V, idx, dO, c)  # noqa: E731
    np.testing.assert_allclose(dq, _fd(f, dqp), atol=1e-7, rtol=1e-6)
    # k_low perturbed: Q' = [Q, (sigma / c) * q_low], K' = [K, dk_pert]
    dkp = np.zeros((Tk, P))
    Qx = np.hstack([Q, (sigma / c) * ql])
    f = lambda: _loss(Qx, np.hstack([K, dkp]), V, idx, dO, c)  # noqa: E731
    np.testing.assert_allclose(dk, _fd(f, dkp), atol=1e-7, rtol=1e-6)


def _sdpa_grads(Q, K, V, dO, causal):
    q, kk, v = (torch.tensor(x[None, None], dtype=torch.float64, requires_grad=True)
                for x in (Q, K, V))
    o = F.scaled_dot_product_attention(q, kk, v, is_causal=causal)
    o.backward(torch.tensor(dO[None, None], dtype=torch.float64))
    return (t.grad[0, 0].numpy() for t in (q, kk, v))


@pytest.mark.parametrize("causal", [False, True])
def test_full_selection_equals_dense_autograd(causal):
    """Selecting every admissible key (all of them, or the causal prefix) is
    dense attention: the gradients equal autograd through float64 SDPA."""
    T, D = 24, 8
    g = np.random.default_rng(15)
    Q, K, V, dO = (g.standard_normal((T, D)) for _ in range(4))
    if causal:
        idx = np.full((T, T), -1, np.int32)
        for i in range(T):
            idx[i, :i + 1] = np.arange(i + 1)[::-1]   # any order: the sum is the same
    else:
        idx = np.tile(np.arange(T, dtype=np.int32), (T, 1))
    dQ, dK, dV, _, _ = oracle.attn_bwd_rows(Q, K, V, idx, dO, 0.0, nthreads=3)
    wQ, wK, wV = _sdpa_grads(Q, K, V, dO, causal)
    np.testing.assert_allclose(dQ, wQ, atol=1e-12, rtol=1e-10)
    np.testing.assert_allclose(dK, wK, atol=1e-12, rtol=1e-10)
    np.testing.assert_allclose(dV, wV, atol=1e-12, rtol=1e-10)


def test_scorer_bwd_equals_autograd_of_the_selected_scores():
    """sum over selected pairs of dS * S, S = sigma * q_low . k_low, through
    torch autograd (repeated entries count per entry; -1 slots not at all)."""
    n, Tk, P, k = 7, 11, 16, 4
    g = np.random.default_rng(16)
    ql, kl = g.standard_normal((n, P)), g.standard_normal((Tk, P))
    idx = np.stack([g.choice(Tk, size=k, replace=False) for _ in range(n)]).astype(np.int32)
    idx[0, 3] = -1
    idx[1, 2] = idx[1, 0]
    dS = g.standard_normal((n, k))
    dq, dk = oracle.scorer_bwd_rows(ql, kl, idx, dS)
    sigma = float(np.float32(P ** -0.5))
    q = torch.tensor(ql, requires_grad=True)
    kk = torch.tensor(kl, requires_grad=True)
    S = sigma * q @ kk.T
    ix = torch.tensor(np.where(idx < 0, 0, idx), dtype=torch.long)
    w = torch.tensor(np.where(idx < 0, 0.0, dS))
    (torch.gather(S, 1, ix) * w).sum().backward()
    np.testing.assert_allclose(dq, q.grad.numpy(), atol=1e-12, rtol=1e-12)
    np.testing.assert_allclose(dk, kk.grad.numpy(), atol=1e-12, rtol=1e-12)


def test_backward_invariants():
    """Softmax shift invariance: the pair gradients of a row sum to zero. The
    weights of a row sum to one, so sum_j dV_j = sum over rows with a key of
    dO_i. Keys never selected and padded slots get nothing. A one-key row
    passes no gradient to Q, K or its score."""
    n, Tk, D, k = 40, 64, 8, 12
    Q, K, V, dO, idx = _case(n, Tk, D, k, seed=17)
    dQ, dK, dV, dS, bad = oracle.attn_bwd_rows(Q, K, V, idx, dO, 0.0, nthreads=4)
    assert bad == 0
    np.testing.assert_allclose(dS.sum(axis=1), 0.0, atol=1e-12)
    has_key = (idx >= 0).any(axis=1)
    np.testing.assert_allclose(dV.sum(axis=0), dO[has_key].sum(axis=0), atol=1e-12)
    assert np.all(dS[idx < 0] == 0.0)
    unused = np.setdiff1d(np.arange(Tk), idx[idx >= 0])
    assert np.all(dK[unused] == 0.0) and np.all(dV[unused] == 0.0)
    assert np.all(dQ[1] == 0.0) and np.all(dS[1] == 0.0)        # the one-key row
    assert np.all(dQ[2] == 0.0)                                  # the empty row


def test_single_key_selection():
    """k = 1: O_i = V_{j_i}, so dV_j = sum of dO_i over the rows choosing j and
    nothing reaches Q, K or the scores."""
    n, Tk, D = 10, 6, 4
    g = np.random.default_rng(18)
    Q, dO = g.standard_normal((n, D)), g.standard_normal((n, D))
    K, V = g.standard_normal((Tk, D)), g.standard_normal((Tk, D))
    idx = g.integers(0, Tk, size=(n, 1)).astype(np.int32)
    dQ, dK, dV, dS, _ = oracle.attn_bwd_rows(Q, K, V, idx, dO)
    want = np.zeros((Tk, D))
    for i in range(n):
        want[idx[i, 0]] += dO[i]
    np.testing.assert_array_equal(dV, want)
    assert np.all(dQ == 0) and np.all(dK == 0) and np.all(dS == 0)


def test_out_of_range_entries_are_skipped_and_counted():
    n, Tk, D, k = 4, 8, 4, 3
    Q, K, V, dO, idx = _case(n, Tk, D, k, seed=19, pad=False, dup=False)
    ref = oracle.attn_bwd_rows(Q, K, V, np.where(np.arange(k) == 2, -1, idx).astype(np.int32),
                               dO)
    bad_idx = idx.copy()
    bad_idx[:, 2] = [Tk, Tk + 5, -2, -7]
    out = oracle.attn_bwd_rows(Q, K, V, bad_idx, dO)
    assert out[4] == 4 and ref[4] == 0
    for a, b in zip(out[:4], ref[:4]):
        np.testing.assert_array_equal(a, b)


def test_whole_tensor_calls_match_per_head():
    B, H, T, D, P, k = 2, 2, 10, 4, 8, 3
    g = np.random.default_rng(20)
    Q, K, V, dO = (g.standard_normal((B, H, T, D)) for _ in range(4))
    ql, kl = g.standard_normal((B, H, T, P)), g.standard_normal((B, H, T, P))
    idx = np.stack([[np.stack([g.choice(T, size=k, replace=False) for _ in range(T)])
                     for _ in range(H)] for _ in range(B)]).astype(np.int32)
    dQ, dK, dV, dS = oracle.sparse_attn_bwd(Q, K, V, idx, dO)
    dq, dk = oracle.scorer_bwd(ql, kl, idx, dS)
    for b in range(B):
        for h in range(H):
            r = oracle.attn_bwd_rows(Q[b, h], K[b, h], V[b, h], idx[b, h], dO[b, h])
            for a, w in zip((dQ[b, h], dK[b, h], dV[b, h], dS[b, h]), r[:4]):
                np.testing.assert_array_equal(a, w)
            s = oracle.scorer_bwd_rows(ql[b, h], kl[b, h], idx[b, h], dS[b, h])
            np.testing.assert_array_equal(dq[b, h], s[0])
            np.testing.assert_array_equal(dk[b, h], s[1])


def _grouped_case(seed, B=1, H=4, H_kv=2, H_idx=1, Tq=5, Tk=7, D=3, k=3):
    g = np.random.default_rng(seed)
    Q = g.standard_normal((B, H, Tq, D))
    dO = g.standard_normal((B, H, Tq, D))
    K = g.standard_normal((B, H_kv, Tk, D))
    V = g.standard_normal((B, H_kv, Tk, D))
    idx = np.stack([[np.stack([g.choice(Tk, size=k, replace=False) for _ in range(Tq)])
                     for _ in range(H_idx)] for _ in range(B)]).astype(np.int32)
    idx[0, 0, 1, 2] = -1
    return Q, K, V, dO, idx


def _grouped_loss(Q, K, V, dO, idx, scale):
    """sum over query heads of O_h . dO_h, each head through the forward
    oracle with its shared key/value head and index list."""
    B, H = Q.shape[:2]
    gk, gi = H // K.shape[1], H // idx.shape[1]
    tot = 0.0
    for b in range(B):
        for h in range(H):
            O, _ = oracle.attn_rows(Q[b, h], K[b, h // gk], V[b, h // gk], idx[b, h // gi], scale,
                                    nthreads=1)
            tot += float(np.sum(O * dO[b, h]))
    return tot


@pytest.mark.parametrize("H,H_kv,H_idx", [(4, 2, 1), (4, 1, 2), (2, 2, 2)])
def test_grouped_bwd_matches_finite_differences(H, H_kv, H_idx):
    """A shared key/value head's gradient sums over the query heads reading it:
    central differences of the forward oracle with shared K and V."""
    Q, K, V, dO, idx = _grouped_case(30 + H_kv + 3 * H_idx, H=H, H_kv=H_kv, H_idx=H_idx)
    c = 0.45
    dQ, dK, dV, dS = oracle.sparse_attn_grouped_bwd(Q, K, V, idx, dO, c)
    f = lambda: _grouped_loss(Q, K, V, dO, idx, c)  # noqa: E731
    np.testing.assert_allclose(dQ, _fd(f, Q), atol=1e-7, rtol=1e-6)
    np.testing.assert_allclose(dK, _fd(f, K), atol=1e-7, rtol=1e-6)
    np.testing.assert_allclose(dV, _fd(f, V), atol=1e-7, rtol=1e-6)
    if H_kv == H_idx == H:   # the plain layout is the plain routine
        r = oracle.sparse_attn_bwd(Q, K, V, idx, dO, c)
        for a, w in zip((dQ, dK, dV, dS), r):
            np.testing.assert_array_equal(a, w)


def test_shared_scorer_bwd_is_the_gradient_of_a_score_bias():
    """One scorer head shared by all query heads (the layout of
    mhpq.cn/news/1098205, section 3.2): a perturbation of the shared q_low or
    k_low moves the selected logits of every head by sigma * dq . k_low (or
    q_low . dk); the finite difference equals the grouped scorer gradient."""
    B, H, H_kv, H_idx, Tq, Tk, D, P = 1, 3, 3, 1, 5, 7, 3, 2
    Q, K, V, dO, idx = _grouped_case(41, B, H, H_kv, H_idx, Tq, Tk, D)
    g = np.random.default_rng(42)
    ql = g.standard_normal((B, H_idx, Tq, P))
    kl = g.standard_normal((B, H_idx, Tk, P))
    c, sigma = 0.5, 0.3
    _, _, _, dS = oracle.sparse_attn_grouped_bwd(Q, K, V, idx, dO, c)
    dq, dk = oracle.scorer_grouped_bwd(ql, kl, idx, dS, sigma)

    def loss_with(qx, kx):
        """Forward loss with Q' = [Q, (sigma / c) qx] and K' = [K, kx]: the
        logits gain sigma * qx . kx (qx, kx of the one scorer head, shared by
        every query head and every key/value head)."""
        Qx = np.concatenate([Q, np.broadcast_to((sigma / c) * qx, (B, H, Tq, P))], axis=-1)
        Kx = np.concatenate([K, np.broadcast_to(kx, (B, H_kv, Tk, P))], axis=-1)
        Vx = np.concatenate([V, np.zeros((B, H_kv, Tk, P))], axis=-1)
        dOx = np.concatenate([dO, np.zeros((B, H, Tq, P))], axis=-1)
        return _grouped_loss(Qx, Kx, Vx, dOx, idx, c)

    dqp = np.zeros((B, H_idx, Tq, P))   # perturbation of q_low around a bias-free forward
    np.testing.assert_allclose(dq, _fd(lambda: loss_with(dqp, kl), dqp), atol=1e-7, rtol=1e-6)
    dkp = np.zeros((B, H_idx, Tk, P))
    np.testing.assert_allclose(dk, _fd(lambda: loss_with(ql, dkp), dkp), atol=1e-7, rtol=1e-6)
