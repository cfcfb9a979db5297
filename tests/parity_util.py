"""Helpers for the GPU parity tests: sampling rows, tolerances, invariants."""
from __future__ import annotations

import numpy as np
import torch

import oracle

TOL_BF16 = 2e-3     # max-abs, bf16 inputs with fp32 accumulation
TOL_F32 = 1e-5      # max-abs, fp32 inputs


def sample_rows(B, H, Tq, n, seed=0, tile=128):
    """Flat row ids (b*H + h)*Tq + i: ends of the sequence, tile edges, random."""
    g = np.random.default_rng(seed)
    rows = set()
    for bh in {0, B * H - 1, (B * H) // 2}:
        for i in [0, 1, Tq - 1, Tq - 2, min(tile - 1, Tq - 1), min(tile, Tq - 1),
                  min(tile + 1, Tq - 1), Tq // 2]:
            if 0 <= i < Tq:
                rows.add(bh * Tq + i)
    while len(rows) < n:
        rows.add(int(g.integers(0, B * H * Tq)))
    return np.array(sorted(rows), dtype=np.int64)


def bf16_round(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).float().numpy()


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    a = np.maximum(np.abs(np.asarray(x, np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def assert_out_close(gpu: np.ndarray, ref: np.ndarray, tol: float, bf16_out: bool):
    """max-abs tolerance; a bf16 output may instead sit within one bf16 ulp of
    the bf16-rounded exact value (the output rounding alone exceeds 2e-3 once
    |O| >= 0.5)."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref)
    if bf16_out:
        ok = (err <= tol) | (np.abs(gpu - bf16_round(ref)) <= bf16_ulp(ref))
    else:
        ok = err <= tol
    if not ok.all():
        bad = np.argwhere(~ok)[:5]
        raise AssertionError("max err %.3g at %s; gpu %s ref %s" % (
            err.max(), bad.tolist(), gpu[tuple(bad.T)], ref[tuple(bad.T)]))
    return float(err.max())


def valid_counts(Tq, Tk, causal, rows_i):
    i = np.asarray(rows_i, np.int64)
    if not causal:
        return np.full(i.shape, Tk, np.int64)
    return np.clip(i + (Tk - Tq) + 1, 0, Tk)


def check_topk_invariants(idx: torch.Tensor, score: torch.Tensor, Tq, Tk, k, causal):
    """Properties that hold at any size, checked on the device for every row:
    entries in range and admissible, padding only at the tail and exactly
    k - k_eff long, no repeated index, order (score desc, index asc)."""
    B, H = idx.shape[:2]
    dev = idx.device
    i = torch.arange(Tq, device=dev).view(1, 1, Tq, 1)
    if causal:
        nv = torch.clamp(i + (Tk - Tq) + 1, 0, Tk)
    else:
        nv = torch.full_like(i, Tk)
    keff = torch.clamp(nv, max=k)
    t = torch.arange(k, device=dev).view(1, 1, 1, k)
    real = t < keff
    assert torch.equal(idx >= 0, real.expand_as(idx)), "padding not exactly the tail k - k_eff"
    assert bool(((idx < nv) | ~real).all()), "index outside the admissible range"
    assert bool((idx[~real.expand_as(idx)] == -1).all())
    if score is not None:
        assert bool(torch.isneginf(score[~real.expand_as(score)]).all())
        s0, s1 = score[..., :-1], score[..., 1:]
        j0, j1 = idx[..., :-1], idx[..., 1:]
        both = real[..., 1:].expand_as(s1)
        ordered = (s0 > s1) | ((s0 == s1) & (j0 < j1))
        assert bool(ordered[both].all()), "selection not ordered by (score desc, index asc)"
    srt, _ = torch.sort(idx, dim=-1)
    dup = (srt[..., 1:] == srt[..., :-1]) & (srt[..., 1:] >= 0)
    assert not bool(dup.any()), "repeated index in a row"


def oracle_topk_for_rows(q_low_cpu, k_low_cpu, k, causal, rows):
    return oracle.score_topk(q_low_cpu, k_low_cpu, k, causal, rows=rows)
