"""The tensor-core score path against the oracle (needs a B300).

ssa_lowrank_scores runs the tcgen05 contraction alone and must reproduce the
oracle's scores bit for bit on integer data. ssa_score_topk on bf16 inputs
with d_proj 64 or 128, k <= 512 and at least 64 query rows runs the
tensor-core selection (group maxima -> per-row bound -> candidates -> sort,
rows that overflow their candidate list redone row-wise); these cases cover
every group size, several 128-row tiles with ragged tails, Tq != Tk, rows
whose candidates overflow, and heavy ties (equal scores everywhere, few
distinct scores, ties above the truncated bound).
"""
import numpy as np
import pytest
import torch

import dynamic_top_sparse_rank_b300 as ssa
import oracle
from workloads import fill

pytestmark = pytest.mark.gpu


def _int_inputs(B, H, Tq, Tk, P, seed, lo=-4, hi=4):
    q = fill((B, H, Tq, P), "int", seed, 1, torch.bfloat16, "cpu")
    k = fill((B, H, Tk, P), "int", seed, 2, torch.bfloat16, "cpu")
    if (lo, hi) != (-4, 4):
        q, k = torch.clamp(q, lo, hi), torch.clamp(k, lo, hi)
    return q, k


@pytest.mark.parametrize("B,H,Tq,Tk,P,causal", [
    (1, 2, 300, 500, 64, True),      # ragged query and key tiles, bottom-right causal
    (2, 1, 129, 1000, 128, False),   # two K atoms per row
    (1, 1, 256, 256, 64, True),      # exact tiles
    (1, 1, 500, 200, 64, True),      # Tq > Tk: leading rows see no key
])
def test_lowrank_scores_exact(cuda_dev, B, H, Tq, Tk, P, causal):
    q, kl = _int_inputs(B, H, Tq, Tk, P, seed=30 + Tq)
    S = ssa.ssa_lowrank_scores(q.to(cuda_dev), kl.to(cuda_dev), causal)
    torch.cuda.synchronize()
    ref = oracle.scores(q, kl, causal)
    np.testing.assert_array_equal(S.cpu().numpy(), ref)


TILE_CASES = [
    # B, H, Tq, Tk, P, k, causal
    (1, 1, 2048, 2048, 64, 64, True),     # group sizes 1..16 across the tiles
    (1, 2, 4096, 4096, 64, 512, True),    # k = 512, groups of 1..2
    (1, 1, 8192, 8192, 64, 32, False),    # group size 128, every row full
    (1, 1, 1000, 3000, 128, 100, True),   # d_proj 128, Tq < Tk
    (1, 1, 3000, 1000, 64, 50, True),     # Tq > Tk: 2000 empty rows
    (2, 3, 333, 777, 64, 17, False),      # ragged everything, small k
    (1, 1, 640, 640, 64, 512, False),     # k close to Tk
    (1, 1, 96, 96, 64, 1, True),          # k = 1
]


@pytest.mark.parametrize("B,H,Tq,Tk,P,k,causal", TILE_CASES)
def test_tile_topk_matches_oracle(cuda_dev, B, H, Tq, Tk, P, k, causal):
    q, kl = _int_inputs(B, H, Tq, Tk, P, seed=40 + Tq + k)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    idx, sc = ssa.ssa_score_topk(q.to(cuda_dev), kl.to(cuda_dev), k, causal, with_score=True,
                                 dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & ~ssa.SSA_DEV_OVERFLOW == 0   # rows redone row-wise are informational
    ref_idx, ref_sc = oracle.score_topk(q, kl, k, causal)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    np.testing.assert_array_equal(sc.cpu().numpy(), ref_sc)


def test_tile_topk_heavy_ties_overflow(cuda_dev):
    """Values in {-1, 0, 1}: few distinct scores, so many rows hold more tied
    candidates than their lists; ties at the bound are dropped once a list is
    full, and rows where a key above the bound finds no slot are redone
    row-wise."""
    B, H, Tq, Tk, P, k = 1, 2, 700, 2500, 64, 64
    q, kl = _int_inputs(B, H, Tq, Tk, P, seed=77, lo=-1, hi=1)
    idx, sc = ssa.ssa_score_topk(q.to(cuda_dev), kl.to(cuda_dev), k, True, with_score=True)
    ref_idx, ref_sc = oracle.score_topk(q, kl, k, True)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    np.testing.assert_array_equal(sc.cpu().numpy(), ref_sc)


ALL_TIES_CASES = [
    # B, H, Tq, Tk, P, k, causal
    (1, 2, 2048, 2048, 64, 512, True),    # the headline k: 1024-entry lists, 512 ties selected
    (1, 1, 1000, 5000, 128, 100, False),  # d_proj 128, every row full
    (2, 1, 700, 3000, 64, 64, True),      # Tq < Tk, small lists
]


@pytest.mark.parametrize("B,H,Tq,Tk,P,k,causal", ALL_TIES_CASES)
def test_tile_topk_all_equal_scores(cuda_dev, B, H, Tq, Tk, P, k, causal):
    """q_low = 0: every score is 0, so every row's answer is its first k_eff
    valid keys. Each row's lists fill with ties at the bound, the later ties
    are dropped, and the sort ranks more than 256 ties by index."""
    q = torch.zeros((B, H, Tq, P), dtype=torch.bfloat16)
    kl = fill((B, H, Tk, P), "int", 61 + k, 2, torch.bfloat16, "cpu")
    st = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    idx, sc = ssa.ssa_score_topk(q.to(cuda_dev), kl.to(cuda_dev), k, causal, with_score=True,
                                 dev_status=st)
    assert int(st.item()) == 0   # no row is redone row-wise: ties at the bound are dropped
    idx, sc = idx.cpu().numpy(), sc.cpu().numpy()
    i = np.arange(Tq)[:, None]
    j = np.arange(k)[None, :]
    n = np.clip(i + (Tk - Tq) + 1, 0, Tk) if causal else np.full_like(i, Tk)
    want = np.where(j < n, j, -1).astype(np.int32)
    np.testing.assert_array_equal(idx, np.broadcast_to(want, idx.shape))
    np.testing.assert_array_equal(sc, np.broadcast_to(np.where(j < n, 0.0, -np.inf).astype(np.float32),
                                                      sc.shape))
    ref_idx, ref_sc = oracle.score_topk(q[:, :1], kl[:, :1], k, causal)
    np.testing.assert_array_equal(idx[:, :1], ref_idx)
    np.testing.assert_array_equal(sc[:, :1], ref_sc)


def test_tile_topk_few_distinct_scores(cuda_dev):
    """One-hot q_low, k_low in {0, 1, 2}: three distinct scores, the top one
    held by about a third of the keys, so the lists fill with ties at the
    bound (which is exact here)."""
    B, H, Tq, Tk, P, k = 1, 2, 1024, 4096, 64, 256
    g = np.random.default_rng(71)
    q = np.zeros((B, H, Tq, P), np.float32)
    q[0, np.arange(H)[:, None], np.arange(Tq)[None, :], g.integers(0, P, size=(H, Tq))] = 1.0
    kl = g.integers(0, 3, size=(B, H, Tk, P)).astype(np.float32)
    q, kl = torch.from_numpy(q).to(torch.bfloat16), torch.from_numpy(kl).to(torch.bfloat16)
    idx, sc = ssa.ssa_score_topk(q.to(cuda_dev), kl.to(cuda_dev), k, True, with_score=True)
    ref_idx, ref_sc = oracle.score_topk(q, kl, k, True)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    np.testing.assert_array_equal(sc.cpu().numpy(), ref_sc)


def test_tile_topk_ties_above_the_bound(cuda_dev):
    """Scores 128.25 (a third of the keys) and 128.5 (twelve late keys): after
    scaling by 1/8 the two share their 16-bit truncated order key, so the
    bound sits below both. The lists fill with 128.25 ties; the late 128.5
    keys lie above the bound and find no slot, so their rows are redone
    row-wise and must still match the oracle."""
    B, H, Tq, Tk, P, k = 1, 1, 512, 3000, 64, 40
    g = np.random.default_rng(72)
    q = np.zeros((B, H, Tq, P), np.float32)
    q[..., 0] = 1.0
    q[..., 1] = 1.0
    kl = np.zeros((B, H, Tk, P), np.float32)
    top = g.random(Tk) < 0.3
    kl[0, 0, :, 0] = np.where(top, 128.0, g.integers(0, 100, size=Tk))
    kl[0, 0, :, 1] = np.where(top, 0.25, 0.0)
    late = g.choice(np.arange(Tk // 4, Tk), size=12, replace=False)
    kl[0, 0, late, 0] = 128.0
    kl[0, 0, late, 1] = 0.5
    q, kl = torch.from_numpy(q).to(torch.bfloat16), torch.from_numpy(kl).to(torch.bfloat16)
    for causal in (False, True):
        st = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
        idx, sc = ssa.ssa_score_topk(q.to(cuda_dev), kl.to(cuda_dev), k, causal, with_score=True,
                                     dev_status=st)
        assert int(st.item()) == ssa.SSA_DEV_OVERFLOW   # rows redone row-wise, reported
        ref_idx, ref_sc = oracle.score_topk(q, kl, k, causal)
        np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
        np.testing.assert_array_equal(sc.cpu().numpy(), ref_sc)


def test_tile_topk_two_calls_one_workspace(cuda_dev):
    """Back-to-back calls on one workspace (stale bounds, counts and
    candidates from the first call must not leak into the second)."""
    B, H, Tq, Tk, P, k = 1, 2, 1500, 1500, 64, 128
    q1, k1 = _int_inputs(B, H, Tq, Tk, P, seed=91)
    q2, k2 = _int_inputs(B, H, Tq, Tk, P, seed=92)
    ws = torch.full((ssa.score_topk_workspace_size(B, H, Tq, Tk, P, k, 1),), 0x5A,
                    dtype=torch.uint8, device=cuda_dev)
    a = ssa.ssa_score_topk(q1.to(cuda_dev), k1.to(cuda_dev), k, True, workspace=ws).cpu()
    b = ssa.ssa_score_topk(q2.to(cuda_dev), k2.to(cuda_dev), k, True, workspace=ws).cpu()
    np.testing.assert_array_equal(a.numpy(), oracle.score_topk(q1, k1, k, True)[0])
    np.testing.assert_array_equal(b.numpy(), oracle.score_topk(q2, k2, k, True)[0])


def test_tile_topk_continuous_scores_are_consistent(cuda_dev):
    """Non-integer bf16 inputs: the selection must be exactly the top of the
    scores the same contraction produces (ssa_lowrank_scores), under the
    (score desc, index asc) order."""
    B, H, Tq, Tk, P, k = 1, 1, 384, 900, 64, 40
    q = fill((B, H, Tq, P), "normal", 5, 1, torch.bfloat16, "cpu")
    kl = fill((B, H, Tk, P), "normal", 5, 2, torch.bfloat16, "cpu")
    qd, kd = q.to(cuda_dev), kl.to(cuda_dev)
    idx, sc = ssa.ssa_score_topk(qd, kd, k, True, with_score=True)
    S = ssa.ssa_lowrank_scores(qd, kd, True).cpu().numpy()
    idx, sc = idx.cpu().numpy(), sc.cpu().numpy()
    for i in range(Tq):
        row = S[0, 0, i]
        order = sorted((j for j in range(Tk) if row[j] > -np.inf), key=lambda j: (-row[j], j))
        want = (order + [-1] * k)[:k]
        assert list(idx[0, 0, i]) == want
        got = sc[0, 0, i][: min(k, len(order))]
        np.testing.assert_array_equal(got, row[want[: len(got)]])


# ------------------------------------------------ boundary smoothing
# mhpq.cn/news/1098205, section 4.2: the (k+1)-th key joins when its score is
# within a threshold of the k-th.

@pytest.mark.parametrize("Tq,Tk,k,causal,delta,dtype,P", [
    (300, 300, 20, True, 3.0, torch.bfloat16, 64),
    (1000, 1000, 64, True, 0.5, torch.bfloat16, 64),
    (129, 700, 31, False, 1e-6, torch.bfloat16, 64),   # only exact ties join
    (1000, 1000, 64, False, 0.0, torch.bfloat16, 64),  # the plain top-k
    (200, 500, 32, True, 1.0, torch.float32, 16),      # the row-wise path
])
def test_score_topk_smooth_matches_oracle(cuda_dev, Tq, Tk, k, causal, delta, dtype, P):
    q = fill((1, 2, Tq, P), "int", Tq + k, 1, dtype, "cpu")
    kl = fill((1, 2, Tk, P), "int", Tq + k, 2, dtype, "cpu")
    idx, sc = ssa.ssa_score_topk_smooth(q.to(cuda_dev), kl.to(cuda_dev), k, causal, delta,
                                        with_score=True)
    ri, rs = oracle.score_topk(q, kl, k + 1, causal)
    ri, rs = oracle.smooth_boundary(ri, rs, k, delta)
    assert np.array_equal(idx.cpu().numpy(), ri)
    assert np.array_equal(sc.cpu().numpy(), rs)
    if delta <= 0:
        assert (idx[..., k] == -1).all()
