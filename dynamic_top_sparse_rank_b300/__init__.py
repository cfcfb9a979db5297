"""Dynamic top-k sparse attention on NVIDIA B300 (sm_103a).

The path's calls, each hand-written CUDA kernels behind the C ABI of
libssa.so (include/ssa.h):

  ssa_score_topk       low-rank scorer fused with exact per-query top-k,
  ssa_sparse_attn      softmax attention over the selected keys only,
  ssa_window_attn      sliding-window attention (the fixed-index special case),
  ssa_sparse_attn_bwd, ssa_scorer_bwd
                       their gradients under the straight-through estimator,
and the projections, selection variants and grouped heads around them.

The binding is marshalling only; there is no CPU fallback.
"""
from ._native import (EXPORTS, SSA_BF16, SSA_DEV_BAD_INDEX, SSA_DEV_OVERFLOW, SSA_DEV_WAIT_LIMIT,
                      SSA_F32, SSAError, load, score_topk_workspace_size, ssa_lowrank_project,
                      ssa_lowrank_scores, ssa_score_topk, ssa_score_topk_smooth,
                      score_topk_smooth_workspace_size, trace_begin, trace_end,
                      ssa_score_topk_noalloc, ssa_scorer_bwd, ssa_sparse_attn, ssa_sparse_attn_bwd,
                      ssa_sparse_attn_grouped, ssa_window_attn, status_string,
                      sparse_attn_bwd_workspace_size, scorer_bwd_workspace_size,
                      ssa_sparse_attn_grouped_bwd, ssa_scorer_grouped_bwd,
                      ssa_selftest_wait_limit, device_status, SSA_ERR_TIMEOUT,
                      ssa_sparse_attn_scorer_bwd, sparse_attn_scorer_bwd_workspace_size)

__all__ = ["EXPORTS", "SSA_BF16", "SSA_DEV_BAD_INDEX", "SSA_DEV_OVERFLOW", "SSA_DEV_WAIT_LIMIT",
           "SSA_F32", "SSAError", "load", "score_topk_workspace_size", "ssa_lowrank_project",
           "ssa_lowrank_scores", "ssa_score_topk_smooth", "score_topk_smooth_workspace_size",
           "ssa_score_topk", "trace_begin", "trace_end",
           "ssa_score_topk_noalloc", "ssa_scorer_bwd", "ssa_sparse_attn", "ssa_sparse_attn_bwd",
           "ssa_sparse_attn_grouped", "ssa_window_attn", "status_string",
           "sparse_attn_bwd_workspace_size", "scorer_bwd_workspace_size",
           "ssa_sparse_attn_grouped_bwd", "ssa_scorer_grouped_bwd", "ssa_selftest_wait_limit",
           "device_status", "SSA_ERR_TIMEOUT", "ssa_sparse_attn_scorer_bwd",
           "sparse_attn_scorer_bwd_workspace_size"]
