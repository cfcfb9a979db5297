"""ssa_score_topk_noalloc on a B300: against the oracle and against ssa_score_topk.

The no-allocation entry point serves callers that may not allocate device
memory where they run the op (an engine plugin confined to a pre-sized arena,
a latency-critical loop that must never call cudaMalloc). It must give the
oracle's answer bit for bit, the same answer as the workspace entry point,
call after call on the library's one shared scratch array, and it must not
change the device's free memory. This file is collected after the forward
path's tests (only the backward's and the wait-limit self-test come later) so
that a run stopping at its first failure has already run them.
"""
import ctypes

import numpy as np
import pytest
import torch

import dynamic_top_sparse_rank_b300 as ssa
import oracle
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


def _raw_call(lib, qd, kd, k, causal, idx, sc):
    B, H, Tq, P = qd.shape
    Tk = kd.shape[2]
    dt = _native.SSA_BF16 if qd.dtype == torch.bfloat16 else _native.SSA_F32
    return lib.ssa_score_topk_noalloc(
        ctypes.c_void_p(qd.data_ptr()), ctypes.c_void_p(kd.data_ptr()), dt, B, H, Tq, Tk, P, k,
        int(causal), 0.0, ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(sc.data_ptr()), None,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_oracle_and_workspace_entry_point_two_calls_in_a_row(cuda_dev):
    # two consecutive no-allocation calls per case (the scratch keeps the
    # previous call's contents), each compared with the oracle and with the
    # workspace entry point
    lib = ssa.load()
    for n, (B, H, Tq, Tk, P, k, causal, dtype) in enumerate(CASES):
        q, kl = _inputs(B, H, Tq, Tk, P, dtype, seed=900 + n)
        ref_idx, ref_sc = oracle.score_topk(q, kl, k, causal)
        qd, kd = q.to(cuda_dev), kl.to(cuda_dev)
        ws_idx, ws_sc = ssa.ssa_score_topk(qd, kd, k, causal, with_score=True)
        idx = torch.empty((B, H, Tq, k), dtype=torch.int32, device=cuda_dev)
        sc = torch.empty((B, H, Tq, k), dtype=torch.float32, device=cuda_dev)
        for _ in range(2):
            idx.fill_(-7)
            sc.fill_(0.5)
            assert _raw_call(lib, qd, kd, k, causal, idx, sc) == _native.SSA_OK
            torch.cuda.synchronize()
            np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
            np.testing.assert_array_equal(sc.cpu().numpy(), ref_sc)
            assert torch.equal(idx, ws_idx)
            assert torch.equal(sc, ws_sc)


def test_noalloc_leaves_free_device_memory_unchanged(cuda_dev):
    # outputs and inputs exist before the calls; the first call may load the
    # library's module (which holds the fixed array), so the measurement
    # starts after it
    lib = ssa.load()
    B, H, Tq, Tk, P, k, causal, dtype = CASES[0]
    q, kl = _inputs(B, H, Tq, Tk, P, dtype, seed=950)
    qd, kd = q.to(cuda_dev), kl.to(cuda_dev)
    idx = torch.empty((B, H, Tq, k), dtype=torch.int32, device=cuda_dev)
    sc = torch.empty((B, H, Tq, k), dtype=torch.float32, device=cuda_dev)
    assert _raw_call(lib, qd, kd, k, causal, idx, sc) == _native.SSA_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(cuda_dev)
    for _ in range(3):
        assert _raw_call(lib, qd, kd, k, causal, idx, sc) == _native.SSA_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(cuda_dev)
    assert free1 == free0


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
    # a misaligned dev_status is refused like every other call's
    rc = lib.ssa_score_topk_noalloc(p, p, _native.SSA_BF16, 1, 1, 1, 64, 64, 4, 0, 0.0,
                                    ctypes.c_void_p(out.data_ptr()), None,
                                    ctypes.c_void_p(out.data_ptr() + 2), None)
    assert rc == _native.SSA_ERR_INVALID
