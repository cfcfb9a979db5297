"""Python face of the CPU oracle — TEST INFRASTRUCTURE ONLY.

The arithmetic lives in ``oracle.c`` (plain fp64 loops, see its header for the
passages it follows). This module compiles it with gcc, loads it with ctypes
and converts tensors to float64 numpy arrays (exact for bf16 and fp32 inputs).
Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
it; the CUDA library never does, and shares no code with it.

Parity status: score_topk, sparse_attn, window_attn, lowrank_project and the
backward (sparse_attn_bwd, scorer_bwd) are pinned by the
``-m "not gpu"`` tests (brute force, closed forms, special cases and an
independent dense masked attention); none is pinned to printed values, because
the pages print none for this path.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, i32, f32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_double
        lib.oracle_topk_rows.argtypes = [P, P, i64, P, i64, i64, i32, i32, i32, f32, P, P, i32]
        lib.oracle_topk_rows.restype = i32
        lib.oracle_attn_rows.argtypes = [P, i64, P, P, i64, i32, P, i32, f64, P, i32]
        lib.oracle_attn_rows.restype = i64
        lib.oracle_window_rows.argtypes = [P, P, i64, P, P, i64, i32, i32, i32, f64, P, i32]
        lib.oracle_window_rows.restype = i32
        lib.oracle_scores_rows.argtypes = [P, P, i64, P, i64, i64, i32, i32, f32, P, i32]
        lib.oracle_project_rows.argtypes = [P, P, i64, i64, i32, P, i32]
        lib.oracle_scores_rows.restype = i32
        lib.oracle_attn_bwd_rows.argtypes = [P, i64, P, P, i64, i32, P, i32, f64, P, P, P, P, P,
                                             i32]
        lib.oracle_attn_bwd_rows.restype = i64
        lib.oracle_scorer_bwd_rows.argtypes = [P, i64, P, i64, i32, P, i32, f64, P, P, P]
        lib.oracle_scorer_bwd_rows.restype = i32
        _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def _f64(x) -> np.ndarray:
    """float64 C-contiguous copy of a torch tensor or array-like."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu", torch.float64).numpy()
    except ImportError:
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# ------------------------------------------------------------- per-head calls

def topk_rows(q_rows, qpos, k_low, k: int, Tq: int, causal: bool, scale: float = 0.0,
              nthreads: int | None = None):
    """Top-k of one head for the given query rows.

    q_rows [n, P] (query positions ``qpos`` [n]), k_low [Tk, P].
    Returns (idx int32 [n, k], score float32 [n, k]).
    """
    q = _f64(q_rows)
    kl = _f64(k_low)
    pos = np.ascontiguousarray(np.asarray(qpos, dtype=np.int64))
    n, P = q.shape
    Tk = kl.shape[0]
    assert kl.shape[1] == P and pos.shape == (n,)
    idx = np.empty((n, k), dtype=np.int32)
    sc = np.empty((n, k), dtype=np.float32)
    rc = _load().oracle_topk_rows(_ptr(q), _ptr(pos), n, _ptr(kl), Tq, Tk, P, k, int(causal),
                                  float(scale), _ptr(idx), _ptr(sc), nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_topk_rows: bad arguments")
    return idx, sc


def scores_rows(q_rows, qpos, k_low, Tq: int, causal: bool, scale: float = 0.0,
                nthreads: int | None = None):
    """Scaled low-rank scores of one head's query rows against all Tk keys,
    float32 [n, Tk]; masked keys hold -inf."""
    q = _f64(q_rows)
    kl = _f64(k_low)
    pos = np.ascontiguousarray(np.asarray(qpos, dtype=np.int64))
    n, P = q.shape
    Tk = kl.shape[0]
    out = np.empty((n, Tk), dtype=np.float32)
    rc = _load().oracle_scores_rows(_ptr(q), _ptr(pos), n, _ptr(kl), Tq, Tk, P, int(causal),
                                    float(scale), _ptr(out), nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_scores_rows: bad arguments")
    return out


def scores(q_low, k_low, causal: bool, scale: float = 0.0, nthreads: int | None = None):
    """Scaled low-rank scores [B,H,Tq,Tk] (float32, -inf where masked)."""
    B, H, Tq, P = q_low.shape
    Tk = k_low.shape[2]
    out = np.empty((B, H, Tq, Tk), np.float32)
    for b in range(B):
        for h in range(H):
            out[b, h] = scores_rows(q_low[b, h], np.arange(Tq), k_low[b, h], Tq, causal, scale,
                                    nthreads)
    return out


def attn_rows(q_rows, K, V, idx, scale: float = 0.0, nthreads: int | None = None):
    """Attention of one head's query rows over their index lists; float64 [n, D]."""
    q = _f64(q_rows)
    Kd = _f64(K)
    Vd = _f64(V)
    ix = np.ascontiguousarray(np.asarray(idx, dtype=np.int32))
    n, D = q.shape
    k = ix.shape[1]
    O = np.empty((n, D), dtype=np.float64)
    bad = _load().oracle_attn_rows(_ptr(q), n, _ptr(Kd), _ptr(Vd), Kd.shape[0], D, _ptr(ix), k,
                                   float(scale), _ptr(O), nthreads or default_threads())
    if bad < 0:
        raise ValueError("oracle_attn_rows: bad arguments")
    return O, int(bad)


def window_rows(q_rows, qpos, K, V, w_left: int, w_right: int, scale: float = 0.0,
                nthreads: int | None = None):
    """Sliding-window attention of one head's query rows; float64 [n, D]."""
    q = _f64(q_rows)
    Kd = _f64(K)
    Vd = _f64(V)
    pos = np.ascontiguousarray(np.asarray(qpos, dtype=np.int64))
    n, D = q.shape
    O = np.empty((n, D), dtype=np.float64)
    rc = _load().oracle_window_rows(_ptr(q), _ptr(pos), n, _ptr(Kd), _ptr(Vd), Kd.shape[0], D,
                                    w_left, w_right, float(scale), _ptr(O),
                                    nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_window_rows: bad arguments")
    return O


def lowrank_project(x, W, nthreads: int | None = None):
    """The scorer's projection x W^T in fp64: x [..., d_model], W [P, d_model];
    returns float64 [..., P] (unrounded)."""
    Wd = _f64(W)
    P, dm = Wd.shape
    xd = _f64(x)
    lead = xd.shape[:-1]
    xr = np.ascontiguousarray(xd.reshape(-1, dm))
    out = np.empty((xr.shape[0], P), dtype=np.float64)
    rc = _load().oracle_project_rows(_ptr(xr), _ptr(Wd), xr.shape[0], dm, P, _ptr(out),
                                     nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_project_rows: bad arguments")
    return out.reshape(lead + (P,))


def attn_bwd_rows(q_rows, K, V, idx, dO, scale: float = 0.0, nthreads: int | None = None):
    """Backward of one head's sparse attention under the straight-through
    estimator (mhpq.cn/news/1098205, section 2.3; the formulas are in
    oracle.c). q_rows and dO [n, D], K and V [Tk, D], idx [n, k].

    Returns (dQ [n, D], dK [Tk, D], dV [Tk, D], dS [n, k], bad): float64, dS the
    gradient each selected pair's score receives, bad the count of skipped
    out-of-range entries."""
    q = _f64(q_rows)
    Kd = _f64(K)
    Vd = _f64(V)
    g = _f64(dO)
    ix = np.ascontiguousarray(np.asarray(idx, dtype=np.int32))
    n, D = q.shape
    k = ix.shape[1]
    Tk = Kd.shape[0]
    assert g.shape == (n, D) and ix.shape[0] == n and Vd.shape == Kd.shape
    dQ = np.empty((n, D), np.float64)
    dK = np.empty((Tk, D), np.float64)
    dV = np.empty((Tk, D), np.float64)
    dS = np.empty((n, k), np.float64)
    bad = _load().oracle_attn_bwd_rows(_ptr(q), n, _ptr(Kd), _ptr(Vd), Tk, D, _ptr(ix), k,
                                       float(scale), _ptr(g), _ptr(dQ), _ptr(dK), _ptr(dV),
                                       _ptr(dS), nthreads or default_threads())
    if bad < 0:
        raise ValueError("oracle_attn_bwd_rows: bad arguments")
    return dQ, dK, dV, dS, int(bad)


def scorer_bwd_rows(q_low_rows, k_low, idx, dS, scale: float = 0.0):
    """The scorer's gradients of one head under the straight-through estimator:
    the selected pairs' scores receive dS [n, k]. q_low_rows [n, P], k_low
    [Tk, P]; scale <= 0 selects d_proj^-0.5 (as an fp32 factor, like the
    forward). Returns float64 (dq_low [n, P], dk_low [Tk, P])."""
    q = _f64(q_low_rows)
    kl = _f64(k_low)
    g = _f64(dS)
    ix = np.ascontiguousarray(np.asarray(idx, dtype=np.int32))
    n, P = q.shape
    Tk = kl.shape[0]
    k = ix.shape[1]
    assert kl.shape[1] == P and ix.shape[0] == n and g.shape == (n, k)
    dq = np.empty((n, P), np.float64)
    dk = np.empty((Tk, P), np.float64)
    rc = _load().oracle_scorer_bwd_rows(_ptr(q), n, _ptr(kl), Tk, P, _ptr(ix), k, float(scale),
                                        _ptr(g), _ptr(dq), _ptr(dk))
    if rc != 0:
        raise ValueError("oracle_scorer_bwd_rows: bad arguments")
    return dq, dk


def round_bf16(v) -> np.ndarray:
    """float64 -> the nearest bf16 value (ties to even), returned as float64.
    bf16 keeps 8 significant bits: a value m * 2^e with m in [0.5, 1) becomes
    rint(m * 256) / 256 * 2^e (numpy's rint rounds half to even). Normal range
    only (the values of these tests)."""
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


# ------------------------------------------------------- whole-tensor calls

def _rows_by_head(B, H, Tq, rows):
    """Group flat row ids (b*H + h)*Tq + i by head: {(b, h): [i...]}."""
    if rows is None:
        return {(b, h): np.arange(Tq) for b in range(B) for h in range(H)}, None
    rows = np.asarray(rows, dtype=np.int64)
    out = {}
    for r in rows:
        bh, i = divmod(int(r), Tq)
        b, h = divmod(bh, H)
        out.setdefault((b, h), []).append(i)
    return {key: np.asarray(v, dtype=np.int64) for key, v in out.items()}, rows


def score_topk(q_low, k_low, k: int, causal: bool, scale: float = 0.0, rows=None,
               nthreads: int | None = None):
    """Top-k of [B,H,Tq,P] x [B,H,Tk,P] for all rows, or for flat row ids ``rows``.

    Returns (idx, score): [B,H,Tq,k] for all rows, else [len(rows), k] in the
    order of ``rows``.
    """
    B, H, Tq, P = q_low.shape
    groups, flat = _rows_by_head(B, H, Tq, rows)
    if flat is None:
        idx = np.empty((B, H, Tq, k), np.int32)
        sc = np.empty((B, H, Tq, k), np.float32)
    else:
        idx = np.empty((len(flat), k), np.int32)
        sc = np.empty((len(flat), k), np.float32)
        where = {int(r): n for n, r in enumerate(flat)}
    for (b, h), qi in groups.items():
        i_, s_ = topk_rows(q_low[b, h][qi], qi, k_low[b, h], k, Tq, causal, scale, nthreads)
        if flat is None:
            idx[b, h], sc[b, h] = i_, s_
        else:
            for t, i in enumerate(qi):
                n = where[(b * H + h) * Tq + int(i)]
                idx[n], sc[n] = i_[t], s_[t]
    return idx, sc


def smooth_boundary(idx, score, k: int, delta: float):
    """Boundary smoothing of a top-(k+1) selection (mhpq.cn/news/1098205,
    section 4.2: when the k-th and the (k+1)-th scores differ by less than a
    threshold, both are selected, so k varies a little). ``idx``/``score`` are
    the sorted top-(k+1) lists [..., k+1]; slot k (the (k+1)-th key) is kept
    iff it holds a key and fp32(score[k-1] - score[k]) < delta, otherwise it
    becomes index -1 / score -inf. The gap is an fp32 subtraction of the two
    fp32 scores (the selection's own precision)."""
    idx = np.array(idx, dtype=np.int32, copy=True)
    score = np.array(score, dtype=np.float32, copy=True)
    with np.errstate(invalid="ignore"):   # -inf - -inf (padded rows) is NaN: not kept
        gap = (score[..., k - 1] - score[..., k]).astype(np.float32)
    keep = (idx[..., k] >= 0) & (gap < np.float32(delta))
    idx[..., k] = np.where(keep, idx[..., k], -1)
    score[..., k] = np.where(keep, score[..., k], np.float32(-np.inf))
    return idx, score


def sparse_attn(Q, K, V, idx, scale: float = 0.0, rows=None, nthreads: int | None = None):
    """Sparse attention; ``idx`` is [B,H,Tq,k] (all rows) or [len(rows), k].

    Returns float64 O: [B,H,Tq,D] or [len(rows), D].
    """
    B, H, Tq, D = Q.shape
    groups, flat = _rows_by_head(B, H, Tq, rows)
    idx = np.asarray(idx)
    if flat is None:
        O = np.empty((B, H, Tq, D), np.float64)
    else:
        O = np.empty((len(flat), D), np.float64)
        where = {int(r): n for n, r in enumerate(flat)}
    for (b, h), qi in groups.items():
        if flat is None:
            ix = idx[b, h][qi]
        else:
            ix = np.stack([idx[where[(b * H + h) * Tq + int(i)]] for i in qi])
        o_, _ = attn_rows(Q[b, h][qi], K[b, h], V[b, h], ix, scale, nthreads)
        if flat is None:
            O[b, h] = o_
        else:
            for t, i in enumerate(qi):
                O[where[(b * H + h) * Tq + int(i)]] = o_[t]
    return O


def window_attn(Q, K, V, w_left: int, w_right: int, scale: float = 0.0, rows=None,
                nthreads: int | None = None):
    """Sliding-window attention over [B,H,T,D]; float64 [B,H,T,D] or [len(rows), D]."""
    B, H, T, D = Q.shape
    groups, flat = _rows_by_head(B, H, T, rows)
    if flat is None:
        O = np.empty((B, H, T, D), np.float64)
    else:
        O = np.empty((len(flat), D), np.float64)
        where = {int(r): n for n, r in enumerate(flat)}
    for (b, h), qi in groups.items():
        o_ = window_rows(Q[b, h][qi], qi, K[b, h], V[b, h], w_left, w_right, scale, nthreads)
        if flat is None:
            O[b, h] = o_
        else:
            for t, i in enumerate(qi):
                O[where[(b * H + h) * T + int(i)]] = o_[t]
    return O


def sparse_attn_bwd(Q, K, V, idx, dO, scale: float = 0.0, nthreads: int | None = None):
    """Backward of sparse attention over [B,H,T,D] with idx [B,H,Tq,k] under the
    straight-through estimator. Returns float64 (dQ, dK, dV, dS)."""
    B, H, Tq, D = Q.shape
    Tk = K.shape[2]
    k = np.asarray(idx).shape[-1]
    dQ = np.empty((B, H, Tq, D), np.float64)
    dK = np.empty((B, H, Tk, D), np.float64)
    dV = np.empty((B, H, Tk, D), np.float64)
    dS = np.empty((B, H, Tq, k), np.float64)
    idx = np.asarray(idx)
    for b in range(B):
        for h in range(H):
            dQ[b, h], dK[b, h], dV[b, h], dS[b, h], _ = attn_bwd_rows(
                Q[b, h], K[b, h], V[b, h], idx[b, h], dO[b, h], scale, nthreads)
    return dQ, dK, dV, dS


def scorer_bwd(q_low, k_low, idx, dS, scale: float = 0.0):
    """The scorer's gradients over [B,H,T,P] with idx and dS [B,H,Tq,k]; float64
    (dq_low, dk_low)."""
    B, H, Tq, P = q_low.shape
    Tk = k_low.shape[2]
    dq = np.empty((B, H, Tq, P), np.float64)
    dk = np.empty((B, H, Tk, P), np.float64)
    idx = np.asarray(idx)
    dS = np.asarray(dS)
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h] = scorer_bwd_rows(q_low[b, h], k_low[b, h], idx[b, h], dS[b, h],
                                                 scale)
    return dq, dk


def sparse_attn_grouped_bwd(Q, K, V, idx, dO, scale: float = 0.0, nthreads: int | None = None):
    """Backward of attention with shared key/value heads and shared index
    lists (the grouped layouts of mhpq.cn/news/1098205, section 3.2, and of
    grouped-query attention), under the straight-through estimator.

    Q, dO [B,H,Tq,D]; K, V [B,H_kv,Tk,D]; idx [B,H_idx,Tq,k]. Query head h
    reads key/value head h // (H // H_kv) and index head h // (H // H_idx).
    Each query head's gradients are those of the plain routine on its own
    operands; a shared key/value head's dK, dV sum over the query heads that
    read it. Returns float64 (dQ [B,H,Tq,D], dK, dV [B,H_kv,Tk,D],
    dS [B,H,Tq,k])."""
    B, H, Tq, D = Q.shape
    H_kv, Tk = K.shape[1], K.shape[2]
    idx = np.asarray(idx)
    H_idx, k = idx.shape[1], idx.shape[3]
    gk, gi = H // H_kv, H // H_idx
    assert gk * H_kv == H and gi * H_idx == H
    dQ = np.empty((B, H, Tq, D), np.float64)
    dK = np.zeros((B, H_kv, Tk, D), np.float64)
    dV = np.zeros((B, H_kv, Tk, D), np.float64)
    dS = np.empty((B, H, Tq, k), np.float64)
    for b in range(B):
        for h in range(H):
            dQ[b, h], dKh, dVh, dS[b, h], _ = attn_bwd_rows(
                Q[b, h], K[b, h // gk], V[b, h // gk], idx[b, h // gi], dO[b, h], scale, nthreads)
            dK[b, h // gk] += dKh
            dV[b, h // gk] += dVh
    return dQ, dK, dV, dS


def scorer_grouped_bwd(q_low, k_low, idx, dS, scale: float = 0.0):
    """The scorer's gradients when H query heads share H_idx scorer heads
    (q_low, k_low, idx with H_idx heads; dS [B,H,Tq,k] from the attention
    backward): the score of a pair in index head hi feeds the logits of every
    query head that reads hi, so its gradient is the sum of their dS. Returns
    float64 (dq_low [B,H_idx,Tq,P], dk_low [B,H_idx,Tk,P])."""
    dS = np.asarray(dS, np.float64)
    B, H, Tq, k = dS.shape
    H_idx = q_low.shape[1]
    gi = H // H_idx
    assert gi * H_idx == H
    summed = dS.reshape(B, H_idx, gi, Tq, k).sum(axis=2)
    return scorer_bwd(q_low, k_low, idx, summed, scale)
