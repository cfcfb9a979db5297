"""Parity of the scorer's low-rank projection (ssa_lowrank_project, tcgen05)
with the oracle: out = x W^T, bias-free (mhpq.cn/news/1098205, section 2.2).

Integer-valued inputs have exact fp32 sums, so the bf16 result must equal the
oracle's exact sum rounded to bf16 bit for bit; normal inputs may differ by
the fp32 summation error of the tensor cores' order plus the final bf16
rounding.
"""
import numpy as np
import pytest
import torch

import dynamic_top_sparse_rank_b300 as ssa
import oracle
from workloads import fill

pytestmark = pytest.mark.gpu

SHAPES = [(1, 64, 64), (127, 128, 64), (300, 1024, 64), (257, 256, 128), (4096, 64, 128),
          (1000, 4096, 64)]


def _inputs(rows, dm, P, kind, seed):
    x = fill((rows, dm), kind, seed, 21, torch.bfloat16, "cpu")
    W = fill((P, dm), kind, seed, 22, torch.bfloat16, "cpu")
    return x, W


@pytest.mark.parametrize("rows,dm,P", SHAPES)
def test_project_integer_inputs_exact(cuda_dev, rows, dm, P):
    x, W = _inputs(rows, dm, P, "int", rows + dm + P)
    ssa.trace_begin()
    out = ssa.ssa_lowrank_project(x.to(cuda_dev), W.to(cuda_dev))
    torch.cuda.synchronize()
    assert [n for n, _ in ssa.trace_end()] == ["lowrank_project"]
    ref = oracle.round_bf16(oracle.lowrank_project(x, W))
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("rows,dm,P", SHAPES)
def test_project_normal_inputs_within_bound(cuda_dev, rows, dm, P):
    """Normal inputs: the fp32 sum in the tensor cores' order may differ from
    the exact one by at most 2 * d_model * 2^-24 * sum_c |x_c W_pc| (a rounded
    sum of d_model exact products), and the result is then rounded once to
    bf16 (at most one bf16 unit in the last place of the result). Where the
    sum nearly cancels, the first term is larger than a bf16 ulp."""
    x, W = _inputs(rows, dm, P, "normal", 3 * rows + dm)
    out = ssa.ssa_lowrank_project(x.to(cuda_dev), W.to(cuda_dev))
    ref = oracle.round_bf16(oracle.lowrank_project(x, W))
    mag = oracle.lowrank_project(x.float().abs(), W.float().abs())
    got = out.float().cpu().numpy().astype(np.float64)
    _, e = np.frexp(np.maximum(np.abs(ref), 1e-30))
    ulp = np.ldexp(1.0, e - 8)   # bf16 spacing at |ref|
    bound = ulp + 2.0 * dm * 2.0 ** -24 * mag
    err = np.abs(got - ref)
    assert (err <= bound).all(), "max err / bound %.3g" % float((err / bound).max())
    # and most results are the correctly rounded value
    assert (err == 0).mean() > 0.9


def test_project_feeds_score_topk(cuda_dev):
    """Projected queries and keys go straight into the tensor-core top-k: with
    integer inputs the projections are exact in bf16, so the indices equal the
    oracle's top-k of the oracle's projections."""
    B, H, T, dm, P, k = 1, 2, 1000, 128, 64, 64
    x = fill((B, H, T, dm), "int", 5, 23, torch.bfloat16, "cpu")
    x = torch.clamp(x, -1, 1)
    Wq = torch.clamp(fill((P, dm), "int", 5, 24, torch.bfloat16, "cpu"), -1, 1)
    Wk = torch.clamp(fill((P, dm), "int", 5, 25, torch.bfloat16, "cpu"), -1, 1)
    dx = x.to(cuda_dev)
    ql = ssa.ssa_lowrank_project(dx, Wq.to(cuda_dev))
    kl = ssa.ssa_lowrank_project(dx, Wk.to(cuda_dev))
    assert tuple(ql.shape) == (B, H, T, P)
    idx = ssa.ssa_score_topk(ql, kl, k, True)
    qo = oracle.lowrank_project(x, Wq)
    ko = oracle.lowrank_project(x, Wk)
    assert np.array_equal(ql.float().cpu().numpy(), qo)   # |q_low| <= 128: exact in bf16
    ref_idx, _ = oracle.score_topk(torch.from_numpy(qo), torch.from_numpy(ko), k, True)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)


def test_project_rejects_unsupported(cuda_dev):
    x = torch.zeros((4, 100), dtype=torch.bfloat16, device=cuda_dev)
    W = torch.zeros((64, 100), dtype=torch.bfloat16, device=cuda_dev)
    with pytest.raises(ssa.SSAError):
        ssa.ssa_lowrank_project(x, W)              # d_model not a multiple of 64
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device=cuda_dev)
    with pytest.raises(ssa.SSAError):
        ssa.ssa_lowrank_project(x, torch.zeros((32, 64), dtype=torch.bfloat16, device=cuda_dev))
    with pytest.raises(ssa.SSAError):
        ssa.ssa_lowrank_project(x.float(), torch.zeros((64, 64), dtype=torch.float32, device=cuda_dev))
    out = ssa.ssa_lowrank_project(x[:0], torch.zeros((64, 64), dtype=torch.bfloat16, device=cuda_dev))
    assert out.shape == (0, 64)
