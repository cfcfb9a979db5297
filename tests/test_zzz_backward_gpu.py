"""GPU parity of the backward under the straight-through estimator (B300).

ssa_sparse_attn_bwd and ssa_scorer_bwd against the fp64 oracle
(oracle.sparse_attn_bwd / scorer_bwd, pinned on the CPU). Inputs are exact in
fp32 (bf16 or fp32 data) and every sum runs in fp32, so both dtypes share one
tolerance: a relative bound per tensor, TOL x the tensor's largest magnitude.
The sums have at most k terms (query side) or a key's pair count (key side),
each of about that magnitude. 2e-5 covers the rounding of a few hundred such
terms: k * 2^-24 is 3e-5 at k = 512, and the rounding errors rarely all add
up. The same kernels run under host emulation in
tests/test_backward_emulated.py. This file is collected last, after the
no-allocation tests, so that a run stopping at its first failure has already
run every other test.
"""
import numpy as np
import pytest
import torch

import dynamic_top_sparse_rank_b300 as ssa
import oracle
from workloads import WORKLOADS, make_attn_inputs, make_grad_output, make_scorer_inputs

pytestmark = pytest.mark.gpu

TOL = 2e-5


def _close(gpu, ref, what, tol=TOL):
    gpu = gpu.detach().cpu().double().numpy() if isinstance(gpu, torch.Tensor) else gpu
    ref = np.asarray(ref, np.float64)
    bound = tol * max(1.0, float(np.abs(ref).max(initial=0.0)))
    err = np.abs(gpu - ref)
    assert err.max(initial=0.0) <= bound, "%s: max err %.3g > %.3g" % (what, err.max(), bound)


def _inputs(B, H, Tq, Tk, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    mk = lambda T: torch.randn(B, H, T, D, generator=g).to(dtype)  # noqa: E731
    return mk(Tq), mk(Tk), mk(Tk), mk(Tq)


def _idx(B, H, Tq, Tk, k, seed):
    g = np.random.default_rng(seed)
    idx = g.integers(0, Tk, size=(B, H, Tq, k)).astype(np.int32)   # repeats allowed
    if k > 1:
        idx[..., -1] = -1                                           # a padded slot
    idx[0, 0, 0, :] = -1                                            # an empty row
    return idx


CASES = [
    # B, H, Tq, Tk, D, k, dtype
    (1, 2, 100, 300, 128, 7, torch.bfloat16),
    (2, 1, 129, 1000, 64, 33, torch.bfloat16),
    (1, 1, 50, 2000, 128, 512, torch.bfloat16),
    (1, 2, 77, 400, 64, 40, torch.float32),
    (1, 1, 31, 700, 128, 96, torch.float32),
    (1, 1, 40, 64, 64, 1, torch.bfloat16),
]


@pytest.mark.parametrize("B,H,Tq,Tk,D,k,dtype", CASES)
def test_sparse_attn_bwd_matches_oracle(cuda_dev, B, H, Tq, Tk, D, k, dtype):
    Q, K, V, dO = _inputs(B, H, Tq, Tk, D, dtype, seed=300 + k)
    idx = _idx(B, H, Tq, Tk, k, seed=k)
    rQ, rK, rV, rS = oracle.sparse_attn_bwd(Q, K, V, idx, dO)
    dev = [t.to(cuda_dev) for t in (Q, K, V, torch.from_numpy(idx), dO)]
    dQ, dK, dV, dS, p = ssa.ssa_sparse_attn_bwd(*dev, with_prob=True)
    _close(dQ, rQ, "dQ")
    _close(dK, rK, "dK")
    _close(dV, rV, "dV")
    _close(dS, rS, "dS")
    assert (dS[0, 0, 0] == 0).all() and (dQ[0, 0, 0] == 0).all()   # the empty row
    pn = p.cpu().numpy()
    live = idx >= 0
    assert (pn[~live] == 0).all()
    np.testing.assert_allclose(pn.sum(-1)[live.any(-1)], 1.0, atol=1e-5)


@pytest.mark.parametrize("P,dtype", [(64, torch.bfloat16), (16, torch.float32),
                                     (128, torch.bfloat16)])
def test_scorer_bwd_matches_oracle(cuda_dev, P, dtype):
    B, H, Tq, Tk, k = 1, 2, 90, 500, 24
    g = torch.Generator().manual_seed(P)
    ql = torch.randn(B, H, Tq, P, generator=g).to(dtype)
    kl = torch.randn(B, H, Tk, P, generator=g).to(dtype)
    idx = _idx(B, H, Tq, Tk, k, seed=P)
    dS = torch.randn(B, H, Tq, k, generator=g)
    rq, rk = oracle.scorer_bwd(ql, kl, idx, dS.numpy())
    dq, dk = ssa.ssa_scorer_bwd(ql.to(cuda_dev), kl.to(cuda_dev),
                                torch.from_numpy(idx).to(cuda_dev), dS.to(cuda_dev))
    _close(dq, rq, "dq_low")
    _close(dk, rk, "dk_low")


@pytest.mark.parametrize("B,H,Tq,Tk,D,P,k,dtype", [
    (1, 2, 100, 300, 128, 64, 7, torch.bfloat16),
    (2, 1, 60, 900, 64, 16, 33, torch.float32),
])
def test_fused_attn_scorer_bwd_matches_oracle(cuda_dev, B, H, Tq, Tk, D, P, k, dtype):
    """ssa_sparse_attn_scorer_bwd (one build of the key-major lists for both
    key sides) against the oracle's attention and scorer gradients."""
    Q, K, V, dO = _inputs(B, H, Tq, Tk, D, dtype, seed=500 + k)
    g = torch.Generator().manual_seed(P + k)
    ql = torch.randn(B, H, Tq, P, generator=g).to(dtype)
    kl = torch.randn(B, H, Tk, P, generator=g).to(dtype)
    idx = _idx(B, H, Tq, Tk, k, seed=k + 1)
    rQ, rK, rV, rS = oracle.sparse_attn_bwd(Q, K, V, idx, dO)
    rq, rk = oracle.scorer_bwd(ql, kl, idx, rS)
    dv = [t.to(cuda_dev) for t in (Q, K, V, dO, ql, kl, torch.from_numpy(idx))]
    dQ, dK, dV, dS, dq, dk = ssa.ssa_sparse_attn_scorer_bwd(*dv)
    for a, r, n in ((dQ, rQ, "dQ"), (dK, rK, "dK"), (dV, rV, "dV"), (dS, rS, "dS"),
                    (dq, rq, "dq_low"), (dk, rk, "dk_low")):
        _close(a, r, n)


def test_backward_of_the_exact_selection(cuda_dev):
    """The path end to end: the GPU top-k feeds the backward; the oracle's
    top-k (bit-identical on integer scorer data) feeds the oracle's."""
    B, H, T, P, D, k = 1, 2, 300, 64, 128, 32
    g = torch.Generator().manual_seed(7)
    ql = torch.randint(-4, 5, (B, H, T, P), generator=g).to(torch.bfloat16)
    kl = torch.randint(-4, 5, (B, H, T, P), generator=g).to(torch.bfloat16)
    Q, K, V, dO = _inputs(B, H, T, T, D, torch.bfloat16, seed=8)
    dv = [t.to(cuda_dev) for t in (ql, kl, Q, K, V, dO)]
    idx = ssa.ssa_score_topk(dv[0], dv[1], k, True)
    ref_idx, _ = oracle.score_topk(ql, kl, k, True)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    dQ, dK, dV, dS = ssa.ssa_sparse_attn_bwd(dv[2], dv[3], dv[4], idx, dv[5])
    dq, dk = ssa.ssa_scorer_bwd(dv[0], dv[1], idx, dS)
    rQ, rK, rV, rS = oracle.sparse_attn_bwd(Q, K, V, ref_idx, dO)
    rq, rk = oracle.scorer_bwd(ql, kl, ref_idx, rS)
    for a, b, n in ((dQ, rQ, "dQ"), (dK, rK, "dK"), (dV, rV, "dV"), (dS, rS, "dS"),
                    (dq, rq, "dq_low"), (dk, rk, "dk_low")):
        _close(a, b, n)


def test_bwd_reports_bad_index(cuda_dev):
    B, H, Tq, Tk, D, k = 1, 1, 8, 16, 64, 4
    Q, K, V, dO = (t.to(cuda_dev) for t in _inputs(B, H, Tq, Tk, D, torch.bfloat16, seed=1))
    idx = torch.zeros(B, H, Tq, k, dtype=torch.int32)
    idx[0, 0, 3, 1] = Tk + 3
    st = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    dQ, dK, dV, dS = ssa.ssa_sparse_attn_bwd(Q, K, V, idx.to(cuda_dev), dO, dev_status=st)
    assert int(st.item()) & 0x1
    assert float(dS[0, 0, 3, 1]) == 0.0


def test_bwd_without_query_rows_zeroes_key_gradients(cuda_dev):
    B, H, Tk, D, k = 1, 2, 40, 64, 4
    Q = torch.zeros(B, H, 0, D, dtype=torch.bfloat16, device=cuda_dev)
    K = torch.randn(B, H, Tk, D, device=cuda_dev).to(torch.bfloat16)
    idx = torch.zeros(B, H, 0, k, dtype=torch.int32, device=cuda_dev)
    dQ, dK, dV, dS = ssa.ssa_sparse_attn_bwd(Q, K, K.clone(), idx, Q.clone())
    torch.cuda.synchronize()
    assert (dK == 0).all() and (dV == 0).all()


GROUPED_CASES = [
    # B, H, H_kv, H_idx, Tq, Tk, D, k, dtype
    (2, 4, 2, 1, 150, 400, 64, 24, torch.bfloat16),    # grouped-query heads, one shared scorer
    (1, 4, 1, 2, 110, 300, 128, 40, torch.float32),    # one key/value head, two index heads
    (1, 8, 8, 1, 130, 500, 128, 64, torch.bfloat16),   # the pages' layout: a shared scorer only
]


@pytest.mark.parametrize("B,H,H_kv,H_idx,Tq,Tk,D,k,dtype", GROUPED_CASES)
def test_grouped_bwd_matches_oracle(cuda_dev, B, H, H_kv, H_idx, Tq, Tk, D, k, dtype):
    g = torch.Generator().manual_seed(H * 10 + H_kv)
    Q = torch.randn(B, H, Tq, D, generator=g).to(dtype)
    dO = torch.randn(B, H, Tq, D, generator=g).to(dtype)
    K = torch.randn(B, H_kv, Tk, D, generator=g).to(dtype)
    V = torch.randn(B, H_kv, Tk, D, generator=g).to(dtype)
    ql = torch.randn(B, H_idx, Tq, 64, generator=g).to(dtype)
    kl = torch.randn(B, H_idx, Tk, 64, generator=g).to(dtype)
    rng = np.random.default_rng(H_idx + 7 * k)
    idx = rng.integers(0, Tk, size=(B, H_idx, Tq, k)).astype(np.int32)
    idx[..., -1] = -1
    idx[0, 0, 0, :] = -1
    dv = [t.to(cuda_dev) for t in (Q, K, V, torch.from_numpy(idx), dO, ql, kl)]
    dQ, dK, dV, dS = ssa.ssa_sparse_attn_grouped_bwd(*dv[:5])
    dq, dk = ssa.ssa_scorer_grouped_bwd(dv[5], dv[6], dv[3], dS)
    rQ, rK, rV, rS = oracle.sparse_attn_grouped_bwd(Q, K, V, idx, dO)
    rq, rk = oracle.scorer_grouped_bwd(ql, kl, idx, rS)
    for a, r, n in ((dQ, rQ, "dQ"), (dK, rK, "dK"), (dV, rV, "dV"), (dS, rS, "dS"),
                    (dq, rq, "dq_low"), (dk, rk, "dk_low")):
        _close(a, r, n)


# ------------------------------------------------- full-size sampled parity

FULL_TOL = 1e-4   # keys chosen by thousands of rows sum that many fp32 terms


def check_backward_sampled(w, dev, idx, n_rows=24, seed=0):
    """The backward workload's launch at full size, checked on samples. Each
    sampled row's dQ, dS and dq_low come from the oracle on that row alone.
    Each sampled key's dK, dV and dk_low come from the oracle on exactly the
    rows that chose it (their full index lists), so every term of the key's
    sum is included. idx is the forward's index lists on `dev`."""
    q_low, k_low = make_scorer_inputs(w, dev)
    Q, K, V = make_attn_inputs(w, dev)
    dO = make_grad_output(w, dev)
    # the bench's call: both backward passes, the key-major lists built once
    dQ, dK, dV, dS, dq, dk = ssa.ssa_sparse_attn_scorer_bwd(Q, K, V, dO, q_low, k_low, idx)
    g = np.random.default_rng(seed)
    heads = sorted({0, w.B * w.H - 1})
    for bh in heads:
        b, h = divmod(bh, w.H)
        ix = idx[b, h].cpu().numpy()
        host = [t[b, h].cpu() for t in (Q, K, V, dO, q_low, k_low)]
        Qh, Kh, Vh, dOh, qh, kh = host
        rows = np.unique(np.concatenate([[0, w.Tq - 1], g.choice(w.Tq, n_rows, replace=False)]))
        rQ, _, _, rS, _ = oracle.attn_bwd_rows(Qh[rows], Kh, Vh, ix[rows], dOh[rows])
        rq, _ = oracle.scorer_bwd_rows(qh[rows], kh, ix[rows], rS)
        sel = torch.from_numpy(rows).to(dev)
        _close(dQ[b, h][sel], rQ, "dQ rows of head %d" % bh, FULL_TOL)
        _close(dS[b, h][sel], rS, "dS rows of head %d" % bh, FULL_TOL)
        _close(dq[b, h][sel], rq, "dq_low rows of head %d" % bh, FULL_TOL)
        # the head's most chosen key (a planted key: its sums are the longest)
        top = int(np.bincount(ix[ix >= 0].ravel(), minlength=w.Tk).argmax())
        for j in sorted({0, w.Tk // 2, w.Tk - 1, int(g.integers(0, w.Tk)), top}):
            who = np.unique(np.nonzero(ix == j)[0])
            if len(who) == 0:
                assert float(dK[b, h, j].abs().max()) == 0.0 and float(dV[b, h, j].abs().max()) == 0.0
                continue
            _, rK, rV, rSj, _ = oracle.attn_bwd_rows(Qh[who], Kh, Vh, ix[who], dOh[who])
            _, rk = oracle.scorer_bwd_rows(qh[who], kh, ix[who], rSj)
            _close(dK[b, h, j], rK[j], "dK key %d of head %d (%d rows)" % (j, bh, len(who)),
                   FULL_TOL)
            _close(dV[b, h, j], rV[j], "dV key %d of head %d" % (j, bh), FULL_TOL)
            _close(dk[b, h, j], rk[j], "dk_low key %d of head %d" % (j, bh), FULL_TOL)


def test_backward_full_size_sampled(cuda_dev):
    """The 128K workload (B1 H8, k 512, D 128) in the bench's launch
    configuration, on sampled rows and keys."""
    w = WORKLOADS["topk_causal_bf16_t128k_k512_planted"]
    q_low, k_low = make_scorer_inputs(w, cuda_dev)
    idx = ssa.ssa_score_topk(q_low, k_low, w.k, w.causal)
    del q_low, k_low
    check_backward_sampled(w, cuda_dev, idx)
