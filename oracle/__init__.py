"""CPU oracle for dynamic top-k sparse attention (test infrastructure only)."""
from .oracle import (attn_bwd_rows, attn_rows, build, default_threads, lowrank_project, round_bf16,
                     score_topk, scorer_bwd, scorer_bwd_rows, scorer_grouped_bwd, scores,
                     scores_rows, smooth_boundary, sparse_attn, sparse_attn_bwd,
                     sparse_attn_grouped_bwd, topk_rows, window_attn, window_rows)

__all__ = ["attn_bwd_rows", "attn_rows", "build", "default_threads", "lowrank_project",
           "round_bf16", "score_topk", "scorer_bwd", "scorer_bwd_rows", "scorer_grouped_bwd",
           "scores", "scores_rows", "smooth_boundary", "sparse_attn", "sparse_attn_bwd",
           "sparse_attn_grouped_bwd", "topk_rows", "window_attn", "window_rows"]
