"""CPU oracle for dynamic top-k sparse attention (test infrastructure only)."""
from .oracle import (attn_rows, build, default_threads, lowrank_project, round_bf16, score_topk,
                     scores, scores_rows, smooth_boundary, sparse_attn, topk_rows, window_attn,
                     window_rows)

__all__ = ["attn_rows", "build", "default_threads", "lowrank_project", "round_bf16", "score_topk",
           "scores", "scores_rows", "smooth_boundary",
           "sparse_attn", "topk_rows", "window_attn", "window_rows"]
