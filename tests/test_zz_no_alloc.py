"""ssa_score_topk_noalloc against ssa_score_topk (needs a B300).

The no-allocation entry point serves callers that may not allocate device
memory where they run the op (an engine plugin confined to a pre-sized arena,
a latency-critical loop that must never call cudaMalloc). It must give the
same answer as the workspace entry point, bit for bit, call after call on the
library's one shared scratch array. This file is collected after the forward
path's tests (only the backward's come later) so that a run stopping at its
first failure has already run them.
"""
import ctypes

import pytest
import torch

import dynamic_top_sparse_rank_b300 as ssa
from dynamic_top_sparse_rank_b300 import _native
from workloads import fill

pytestmark = pytest.mark.gpu


def _inputs(B, H, Tq, Tk, P, dtype, seed):
    q = fill((B, H, Tq, P), "int", seed, 1, dtype, "cpu")
    k = fill((B, H, Tk, P), "int", seed, 2, dtype, "cpu")
    return q, k


CASES = [
    # B, H, Tq, Tk, P, k, causal, dtype
    (1, 2, 300, 5000, 64, 128, True, torch.bfloat16),
    (4, 2, 1, 65536, 64, 512, False, torch.bfloat16),
    (1, 1, 1500, 1500, 16, 32, False, torch.float32),
]


def test_noalloc_matches_workspace_entry_point_two_calls_in_a_row(cuda_dev):
    # two consecutive no-allocation calls per case (the scratch keeps the
    # previous call's contents), each compared with the workspace entry point
    for n, (B, H, Tq, Tk, P, k, causal, dtype) in enumerate(CASES):
        q, kl = _inputs(B, H, Tq, Tk, P, dtype, seed=900 + n)
        qd, kd = q.to(cuda_dev), kl.to(cuda_dev)
        ref_idx, ref_sc = ssa.ssa_score_topk(qd, kd, k, causal, with_score=True)
        for _ in range(2):
            idx, sc = ssa.ssa_score_topk_noalloc(qd, kd, k, causal, with_score=True)
            torch.cuda.synchronize()
            assert torch.equal(idx, ref_idx)
            assert torch.equal(sc, ref_sc)


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_dev):
    lib = ssa.load()
    buf = torch.zeros(1024, dtype=torch.bfloat16, device=cuda_dev)
    out = torch.zeros(64, dtype=torch.int32, device=cuda_dev)
    p = ctypes.c_void_p(buf.data_ptr())
    too_long = _native.NOALLOC_MAX_TK + 1
    rc = lib.ssa_score_topk_noalloc(p, p, _native.SSA_BF16, 1, 1, 1, too_long, 64, 4, 0, 0.0,
                                    ctypes.c_void_p(out.data_ptr()), None, None, None)
    assert rc == _native.SSA_ERR_UNSUPPORTED
    # an empty problem at the largest accepted Tk is accepted (and is a no-op)
    rc = lib.ssa_score_topk_noalloc(p, p, _native.SSA_BF16, 1, 1, 0, _native.NOALLOC_MAX_TK, 64,
                                    4, 0, 0.0, ctypes.c_void_p(out.data_ptr()), None, None, None)
    assert rc == _native.SSA_OK
