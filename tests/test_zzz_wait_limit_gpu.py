"""Failure detection without a GPU fault (B300): a bounded device wait that
runs out reports SSA_DEV_WAIT_LIMIT and returns, and the context stays
usable. ssa_selftest_wait_limit waits, with the tensor-core kernels' own wait
helper, on an mbarrier that nothing completes. Collected last."""
import time

import numpy as np
import pytest
import torch

import dynamic_top_sparse_rank_b300 as ssa
import oracle

pytestmark = pytest.mark.gpu


def test_wait_runs_out_reports_and_the_context_stays_usable(cuda_dev):
    st = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ssa.ssa_selftest_wait_limit(st, limit_ns=2_000_000)   # 2 ms
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(st.item()) == ssa.SSA_DEV_WAIT_LIMIT
    assert 0.002 <= waited < 5.0
    # the host end of the rule: the wait that ran out reads as SSA_ERR_TIMEOUT
    assert ssa.device_status(st) == (ssa.SSA_ERR_TIMEOUT, ssa.SSA_DEV_WAIT_LIMIT)
    st.zero_()
    assert ssa.device_status(st) == (0, 0)
    # the context still runs the path: a small exact top-k against the oracle
    g = np.random.default_rng(0)
    q = torch.from_numpy(g.integers(-4, 5, size=(1, 2, 200, 64)).astype(np.float32)).to(torch.bfloat16)
    k = torch.from_numpy(g.integers(-4, 5, size=(1, 2, 200, 64)).astype(np.float32)).to(torch.bfloat16)
    idx = ssa.ssa_score_topk(q.to(cuda_dev), k.to(cuda_dev), 16, True)
    ref, _ = oracle.score_topk(q, k, 16, True)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref)
