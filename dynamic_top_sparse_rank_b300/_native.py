"""ctypes binding of libssa.so: argument marshalling only.

Every step of the path runs in the CUDA kernels behind the C ABI declared in
include/ssa.h. The functions here check tensor placement, dtype and
contiguity, allocate outputs with torch (device memory is torch's job), pass raw
pointers and the current CUDA stream, and turn a non-zero status into an
exception. There is no CPU fallback: without the built library every call
raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libssa.so")

SSA_OK, SSA_ERR_INVALID, SSA_ERR_UNSUPPORTED, SSA_ERR_CUDA = 0, 1, 2, 3
SSA_ERR_TIMEOUT, SSA_ERR_WORKSPACE = 4, 5
SSA_F32, SSA_BF16 = 0, 1
SSA_DEV_BAD_INDEX, SSA_DEV_WAIT_LIMIT, SSA_DEV_OVERFLOW = 0x1, 0x2, 0x4

EXPORTS = ("ssa_version", "ssa_status_string", "ssa_score_topk_workspace_size", "ssa_score_topk",
           "ssa_sparse_attn", "ssa_window_attn", "ssa_score_topk_noalloc", "ssa_lowrank_scores",
           "ssa_lowrank_project", "ssa_sparse_attn_grouped", "ssa_score_topk_smooth",
           "ssa_score_topk_smooth_workspace_size", "ssa_trace_begin", "ssa_trace_end",
           "ssa_sparse_attn_bwd_workspace_size", "ssa_sparse_attn_bwd",
           "ssa_scorer_bwd_workspace_size", "ssa_scorer_bwd",
           "ssa_sparse_attn_grouped_bwd_workspace_size", "ssa_sparse_attn_grouped_bwd",
           "ssa_scorer_grouped_bwd_workspace_size", "ssa_scorer_grouped_bwd",
           "ssa_selftest_wait_limit", "ssa_device_status", "ssa_sparse_attn_scorer_bwd",
           "ssa_sparse_attn_scorer_bwd_workspace_size")

# Fixed scratch of ssa_score_topk_noalloc and the largest Tk it accepts.
NOALLOC_SCRATCH_BYTES = 32 << 20
NOALLOC_MAX_TK = NOALLOC_SCRATCH_BYTES // 4


class SSAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, status_string(status), status))


_lib = None


def load(path: str | None = None):
    """Load libssa.so (raises OSError when it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise OSError("libssa.so not built at %s: run __graft_entry__.build() or "
                      "python -m dynamic_top_sparse_rank_b300.build" % p)
    lib = ctypes.CDLL(p)
    V, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.ssa_version.restype = I
    lib.ssa_version.argtypes = []
    lib.ssa_status_string.restype = ctypes.c_char_p
    lib.ssa_status_string.argtypes = [I]
    lib.ssa_score_topk_workspace_size.restype = Z
    lib.ssa_score_topk_workspace_size.argtypes = [I, I, I, I, I, I, I]
    lib.ssa_score_topk.restype = I
    lib.ssa_score_topk.argtypes = [V, V, I, I, I, I, I, I, I, I, F, V, V, V, Z, V, V]
    lib.ssa_sparse_attn.restype = I
    lib.ssa_sparse_attn.argtypes = [V, V, V, I, I, I, I, I, I, V, I, F, V, I, V, V]
    lib.ssa_window_attn.restype = I
    lib.ssa_window_attn.argtypes = [V, V, V, I, I, I, I, I, I, I, F, V, I, V, V]
    lib.ssa_score_topk_noalloc.restype = I
    lib.ssa_score_topk_noalloc.argtypes = [V, V, I, I, I, I, I, I, I, I, F, V, V, V, V]
    lib.ssa_trace_begin.restype = I
    lib.ssa_trace_begin.argtypes = []
    lib.ssa_trace_end.restype = I
    lib.ssa_trace_end.argtypes = [V, I]
    lib.ssa_lowrank_scores.restype = I
    lib.ssa_lowrank_scores.argtypes = [V, V, I, I, I, I, I, I, I, F, V, V, V]
    lib.ssa_sparse_attn_grouped.restype = I
    lib.ssa_sparse_attn_grouped.argtypes = [V, V, V, I, I, I, I, I, I, I, V, I, I, F, V, I, V, V]
    lib.ssa_score_topk_smooth_workspace_size.restype = Z
    lib.ssa_score_topk_smooth_workspace_size.argtypes = [I, I, I, I, I, I, I]
    lib.ssa_score_topk_smooth.restype = I
    lib.ssa_score_topk_smooth.argtypes = [V, V, I, I, I, I, I, I, I, I, F, F, V, V, V, Z, V, V]
    lib.ssa_lowrank_project.restype = I
    lib.ssa_lowrank_project.argtypes = [V, V, I, ctypes.c_int64, I, I, V, V, V]
    lib.ssa_sparse_attn_bwd_workspace_size.restype = Z
    lib.ssa_sparse_attn_bwd_workspace_size.argtypes = [I, I, I, I, I]
    lib.ssa_sparse_attn_bwd.restype = I
    lib.ssa_sparse_attn_bwd.argtypes = [V, V, V, V, I, I, I, I, I, I, V, I, F, V, V, V, V, V, V, Z,
                                        V, V]
    lib.ssa_scorer_bwd_workspace_size.restype = Z
    lib.ssa_scorer_bwd_workspace_size.argtypes = [I, I, I, I, I]
    lib.ssa_scorer_bwd.restype = I
    lib.ssa_scorer_bwd.argtypes = [V, V, I, I, I, I, I, I, V, I, V, F, V, V, V, Z, V, V]
    lib.ssa_sparse_attn_grouped_bwd_workspace_size.restype = Z
    lib.ssa_sparse_attn_grouped_bwd_workspace_size.argtypes = [I, I, I, I, I, I]
    lib.ssa_sparse_attn_grouped_bwd.restype = I
    lib.ssa_sparse_attn_grouped_bwd.argtypes = [V, V, V, V, I, I, I, I, I, I, I, V, I, I, F, V, V,
                                                V, V, V, V, Z, V, V]
    lib.ssa_scorer_grouped_bwd_workspace_size.restype = Z
    lib.ssa_scorer_grouped_bwd_workspace_size.argtypes = [I, I, I, I, I, I]
    lib.ssa_scorer_grouped_bwd.restype = I
    lib.ssa_scorer_grouped_bwd.argtypes = [V, V, I, I, I, I, I, I, I, V, I, V, F, V, V, V, Z, V, V]
    lib.ssa_sparse_attn_scorer_bwd_workspace_size.restype = Z
    lib.ssa_sparse_attn_scorer_bwd_workspace_size.argtypes = [I, I, I, I, I]
    lib.ssa_sparse_attn_scorer_bwd.restype = I
    lib.ssa_sparse_attn_scorer_bwd.argtypes = [V, V, V, V, V, V, I, I, I, I, I, I, I, V, I, F, F,
                                               V, V, V, V, V, V, V, V, Z, V, V]
    lib.ssa_device_status.restype = I
    lib.ssa_device_status.argtypes = [V, V, V]
    lib.ssa_selftest_wait_limit.restype = I
    lib.ssa_selftest_wait_limit.argtypes = [V, ctypes.c_uint64, V]
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load().ssa_status_string(status).decode()
    except OSError:
        return "status %d" % status


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SSA_F32
    if t.dtype == torch.bfloat16:
        return SSA_BF16
    raise TypeError("unsupported dtype %s (float32 or bfloat16)" % t.dtype)


def _dev(*ts):
    dev = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("tensors must live on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError("tensors on different devices")
    return dev


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr() if t is not None else 0)


def _stream(dev) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _check(rc: int, where: str):
    if rc != SSA_OK:
        raise SSAError(rc, where)


def score_topk_workspace_size(B, H, Tq, Tk, P, k, causal) -> int:
    return int(load().ssa_score_topk_workspace_size(B, H, Tq, Tk, P, k, int(bool(causal))))


def ssa_score_topk(q_low: torch.Tensor, k_low: torch.Tensor, k: int, causal: bool,
                   scale: float = 0.0, with_score: bool = False, workspace: torch.Tensor = None,
                   idx: torch.Tensor = None, score: torch.Tensor = None,
                   dev_status: torch.Tensor = None):
    """Exact top-k of the low-rank scores; returns idx (and score if asked).

    q_low [B,H,Tq,P], k_low [B,H,Tk,P] (float32 or bfloat16, same dtype).
    idx int32 [B,H,Tq,k]; score float32 [B,H,Tq,k].
    """
    lib = load()
    dev = _dev(q_low, k_low, workspace, idx, score, dev_status)
    if q_low.dtype != k_low.dtype:
        raise TypeError("q_low and k_low must share a dtype")
    B, H, Tq, P = q_low.shape
    Bk, Hk, Tk, Pk = k_low.shape
    if (Bk, Hk, Pk) != (B, H, P):
        raise ValueError("k_low shape %s does not match q_low %s" % (tuple(k_low.shape), tuple(q_low.shape)))
    if idx is None:
        idx = torch.empty((B, H, Tq, k), dtype=torch.int32, device=dev)
    if with_score and score is None:
        score = torch.empty((B, H, Tq, k), dtype=torch.float32, device=dev)
    need = score_topk_workspace_size(B, H, Tq, Tk, P, k, causal)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    wbytes = workspace.numel() * workspace.element_size()
    rc = lib.ssa_score_topk(_ptr(q_low), _ptr(k_low), _dt(q_low), B, H, Tq, Tk, P, k,
                            int(bool(causal)), float(scale), _ptr(idx), _ptr(score),
                            _ptr(workspace), wbytes, _ptr(dev_status), _stream(dev))
    _check(rc, "ssa_score_topk")
    return (idx, score) if with_score else idx


def score_topk_smooth_workspace_size(B, H, Tq, Tk, P, k, causal) -> int:
    return int(load().ssa_score_topk_smooth_workspace_size(B, H, Tq, Tk, P, k, int(bool(causal))))


def ssa_score_topk_smooth(q_low: torch.Tensor, k_low: torch.Tensor, k: int, causal: bool,
                          delta: float, scale: float = 0.0, with_score: bool = False,
                          workspace: torch.Tensor = None, idx: torch.Tensor = None,
                          score: torch.Tensor = None, dev_status: torch.Tensor = None):
    """Top-k with boundary smoothing: k + 1 slots per row, the last one kept
    only when its score is within delta of the k-th (else -1 / -inf)."""
    lib = load()
    dev = _dev(q_low, k_low, workspace, idx, score, dev_status)
    if q_low.dtype != k_low.dtype:
        raise TypeError("q_low and k_low must share a dtype")
    B, H, Tq, P = q_low.shape
    Tk = k_low.shape[2]
    if tuple(k_low.shape) != (B, H, Tk, P):
        raise ValueError("k_low shape %s does not match q_low %s" % (tuple(k_low.shape), tuple(q_low.shape)))
    if idx is None:
        idx = torch.empty((B, H, Tq, k + 1), dtype=torch.int32, device=dev)
    if with_score and score is None:
        score = torch.empty((B, H, Tq, k + 1), dtype=torch.float32, device=dev)
    need = score_topk_smooth_workspace_size(B, H, Tq, Tk, P, k, causal)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    wbytes = workspace.numel() * workspace.element_size()
    rc = lib.ssa_score_topk_smooth(_ptr(q_low), _ptr(k_low), _dt(q_low), B, H, Tq, Tk, P, k,
                                   int(bool(causal)), float(scale), float(delta), _ptr(idx),
                                   _ptr(score), _ptr(workspace), wbytes, _ptr(dev_status),
                                   _stream(dev))
    _check(rc, "ssa_score_topk_smooth")
    return (idx, score) if with_score else idx


def ssa_score_topk_noalloc(q_low: torch.Tensor, k_low: torch.Tensor, k: int, causal: bool,
                           scale: float = 0.0, with_score: bool = False, idx: torch.Tensor = None,
                           score: torch.Tensor = None, dev_status: torch.Tensor = None):
    """ssa_score_topk without a workspace, for callers that cannot allocate
    device memory where they run the op: the library's fixed 32 MiB scratch
    array is used instead (Tk <= 8,388,608). Outputs are allocated here only
    when the caller does not pass them. Calls that overlap on the GPU race on
    the shared scratch."""
    lib = load()
    dev = _dev(q_low, k_low, idx, score, dev_status)
    if q_low.dtype != k_low.dtype:
        raise TypeError("q_low and k_low must share a dtype")
    B, H, Tq, P = q_low.shape
    Tk = k_low.shape[2]
    if tuple(k_low.shape) != (B, H, Tk, P):
        raise ValueError("k_low shape %s does not match q_low %s" % (tuple(k_low.shape), tuple(q_low.shape)))
    if Tk > NOALLOC_MAX_TK:
        raise ValueError("ssa_score_topk_noalloc: Tk=%d exceeds the fixed scratch limit %d"
                         % (Tk, NOALLOC_MAX_TK))
    if idx is None:
        idx = torch.empty((B, H, Tq, k), dtype=torch.int32, device=dev)
    if with_score and score is None:
        score = torch.empty((B, H, Tq, k), dtype=torch.float32, device=dev)
    rc = lib.ssa_score_topk_noalloc(_ptr(q_low), _ptr(k_low), _dt(q_low), B, H, Tq, Tk, P, k,
                                    int(bool(causal)), float(scale), _ptr(idx), _ptr(score),
                                    _ptr(dev_status), _stream(dev))
    _check(rc, "ssa_score_topk_noalloc")
    return (idx, score) if with_score else idx


def ssa_lowrank_scores(q_low: torch.Tensor, k_low: torch.Tensor, causal: bool,
                       scale: float = 0.0, out: torch.Tensor = None,
                       dev_status: torch.Tensor = None) -> torch.Tensor:
    """The scaled low-rank scores S [B,H,Tq,Tk] (float32, -inf where masked).

    Materialises the whole score matrix: meant for inspection and small
    problems; the selection path never stores it.
    """
    lib = load()
    dev = _dev(q_low, k_low, out, dev_status)
    if q_low.dtype != k_low.dtype:
        raise TypeError("q_low and k_low must share a dtype")
    B, H, Tq, P = q_low.shape
    Tk = k_low.shape[2]
    if tuple(k_low.shape) != (B, H, Tk, P):
        raise ValueError("k_low shape %s does not match q_low %s" % (tuple(k_low.shape), tuple(q_low.shape)))
    if out is None:
        out = torch.empty((B, H, Tq, Tk), dtype=torch.float32, device=dev)
    rc = lib.ssa_lowrank_scores(_ptr(q_low), _ptr(k_low), _dt(q_low), B, H, Tq, Tk, P,
                                int(bool(causal)), float(scale), _ptr(out), _ptr(dev_status),
                                _stream(dev))
    _check(rc, "ssa_lowrank_scores")
    return out


def ssa_lowrank_project(x: torch.Tensor, W: torch.Tensor, out: torch.Tensor = None,
                        dev_status: torch.Tensor = None) -> torch.Tensor:
    """The scorer's low-rank projection out = x W^T (bf16 in, fp32 sums, bf16
    out): x [..., d_model] (e.g. [B, H, T, d_model]), W [P, d_model] (a linear
    layer's weight); returns [..., P]."""
    lib = load()
    dev = _dev(x, W, out, dev_status)
    if x.dtype != W.dtype:
        raise TypeError("x and W must share a dtype")
    P, d_model = W.shape
    if x.shape[-1] != d_model:
        raise ValueError("x has %d columns, W %d" % (x.shape[-1], d_model))
    rows = x.numel() // d_model if d_model else 0
    if out is None:
        out = torch.empty(tuple(x.shape[:-1]) + (P,), dtype=x.dtype, device=dev)
    rc = lib.ssa_lowrank_project(_ptr(x), _ptr(W), _dt(x), rows, d_model, P, _ptr(out),
                                 _ptr(dev_status), _stream(dev))
    _check(rc, "ssa_lowrank_project")
    return out


def ssa_sparse_attn(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, idx: torch.Tensor,
                    scale: float = 0.0, out_dtype=None, out: torch.Tensor = None,
                    dev_status: torch.Tensor = None) -> torch.Tensor:
    """Attention of each query row over the keys its idx row lists; returns O."""
    lib = load()
    dev = _dev(Q, K, V, idx, out, dev_status)
    if not (Q.dtype == K.dtype == V.dtype):
        raise TypeError("Q, K, V must share a dtype")
    if idx.dtype != torch.int32:
        raise TypeError("idx must be int32")
    B, H, Tq, D = Q.shape
    Tk = K.shape[2]
    if tuple(K.shape) != (B, H, Tk, D) or tuple(V.shape) != (B, H, Tk, D):
        raise ValueError("K/V shapes do not match Q")
    if idx.shape[:3] != (B, H, Tq):
        raise ValueError("idx shape %s does not match Q" % (tuple(idx.shape),))
    k = idx.shape[3]
    odt = out_dtype or Q.dtype
    if out is None:
        out = torch.empty((B, H, Tq, D), dtype=odt, device=dev)
    rc = lib.ssa_sparse_attn(_ptr(Q), _ptr(K), _ptr(V), _dt(Q), B, H, Tq, Tk, D, _ptr(idx), k,
                             float(scale), _ptr(out), _dt(out), _ptr(dev_status), _stream(dev))
    _check(rc, "ssa_sparse_attn")
    return out


def ssa_sparse_attn_grouped(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, idx: torch.Tensor,
                            scale: float = 0.0, out_dtype=None, out: torch.Tensor = None,
                            dev_status: torch.Tensor = None) -> torch.Tensor:
    """Attention with shared key/value heads and/or shared index lists:
    Q [B,H,Tq,D], K/V [B,H_kv,Tk,D], idx [B,H_idx,Tq,k] (H_kv, H_idx divide H);
    head h reads K/V head h // (H // H_kv) and index list h // (H // H_idx)."""
    lib = load()
    dev = _dev(Q, K, V, idx, out, dev_status)
    if not (Q.dtype == K.dtype == V.dtype):
        raise TypeError("Q, K, V must share a dtype")
    if idx.dtype != torch.int32:
        raise TypeError("idx must be int32")
    B, H, Tq, D = Q.shape
    H_kv, Tk = K.shape[1], K.shape[2]
    if tuple(K.shape) != (B, H_kv, Tk, D) or tuple(V.shape) != (B, H_kv, Tk, D):
        raise ValueError("K/V shapes do not match Q")
    H_idx, k = idx.shape[1], idx.shape[3]
    if tuple(idx.shape) != (B, H_idx, Tq, k):
        raise ValueError("idx shape %s does not match Q" % (tuple(idx.shape),))
    odt = out_dtype or Q.dtype
    if out is None:
        out = torch.empty((B, H, Tq, D), dtype=odt, device=dev)
    rc = lib.ssa_sparse_attn_grouped(_ptr(Q), _ptr(K), _ptr(V), _dt(Q), B, H, H_kv, Tq, Tk, D,
                                     _ptr(idx), H_idx, k, float(scale), _ptr(out), _dt(out),
                                     _ptr(dev_status), _stream(dev))
    _check(rc, "ssa_sparse_attn_grouped")
    return out


def ssa_window_attn(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, w_left: int,
                    w_right: int = None, scale: float = 0.0, out_dtype=None,
                    out: torch.Tensor = None, dev_status: torch.Tensor = None) -> torch.Tensor:
    """Sliding-window attention, keys i - w_left .. i + w_right clipped to [0, T)."""
    lib = load()
    dev = _dev(Q, K, V, out, dev_status)
    if not (Q.dtype == K.dtype == V.dtype):
        raise TypeError("Q, K, V must share a dtype")
    B, H, T, D = Q.shape
    if tuple(K.shape) != (B, H, T, D) or tuple(V.shape) != (B, H, T, D):
        raise ValueError("K/V shapes do not match Q")
    if w_right is None:
        w_right = w_left
    odt = out_dtype or Q.dtype
    if out is None:
        out = torch.empty((B, H, T, D), dtype=odt, device=dev)
    rc = lib.ssa_window_attn(_ptr(Q), _ptr(K), _ptr(V), _dt(Q), B, H, T, D, int(w_left),
                             int(w_right), float(scale), _ptr(out), _dt(out), _ptr(dev_status),
                             _stream(dev))
    _check(rc, "ssa_window_attn")
    return out


class _TraceRecord(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 56), ("ms", ctypes.c_float)]


def sparse_attn_bwd_workspace_size(B, H, Tq, Tk, k) -> int:
    return int(load().ssa_sparse_attn_bwd_workspace_size(B, H, Tq, Tk, k))


def scorer_bwd_workspace_size(B, H, Tq, Tk, k) -> int:
    return int(load().ssa_scorer_bwd_workspace_size(B, H, Tq, Tk, k))


def ssa_sparse_attn_bwd(Q, K, V, idx, dO, scale: float = 0.0, workspace=None,
                        dev_status=None, with_prob: bool = False):
    """Gradients of ssa_sparse_attn under the straight-through estimator.

    Returns fp32 (dQ [B,H,Tq,D], dK, dV [B,H,Tk,D], dS [B,H,Tq,k]) (+ prob)."""
    lib = load()
    dev = _dev(Q, K, V, idx, dO, workspace, dev_status)
    if not (Q.dtype == K.dtype == V.dtype == dO.dtype):
        raise TypeError("Q, K, V, dO must share a dtype")
    if idx.dtype != torch.int32:
        raise TypeError("idx must be int32")
    B, H, Tq, D = Q.shape
    Tk = K.shape[2]
    if tuple(K.shape) != (B, H, Tk, D) or tuple(V.shape) != (B, H, Tk, D) or \
            tuple(dO.shape) != (B, H, Tq, D):
        raise ValueError("K/V/dO shapes do not match Q")
    if idx.shape[:3] != (B, H, Tq):
        raise ValueError("idx shape %s does not match Q" % (tuple(idx.shape),))
    k = idx.shape[3]
    f32 = dict(dtype=torch.float32, device=dev)
    dQ = torch.empty((B, H, Tq, D), **f32)
    dK = torch.empty((B, H, Tk, D), **f32)
    dV = torch.empty((B, H, Tk, D), **f32)
    dS = torch.empty((B, H, Tq, k), **f32)
    prob = torch.empty((B, H, Tq, k), **f32) if with_prob else None
    need = sparse_attn_bwd_workspace_size(B, H, Tq, Tk, k)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    wbytes = workspace.numel() * workspace.element_size()
    rc = lib.ssa_sparse_attn_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _dt(Q), B, H, Tq, Tk, D,
                                 _ptr(idx), k, float(scale), _ptr(dQ), _ptr(dK), _ptr(dV),
                                 _ptr(dS), _ptr(prob), _ptr(workspace), wbytes,
                                 _ptr(dev_status), _stream(dev))
    _check(rc, "ssa_sparse_attn_bwd")
    return (dQ, dK, dV, dS, prob) if with_prob else (dQ, dK, dV, dS)


def ssa_scorer_bwd(q_low, k_low, idx, dS, scale: float = 0.0, workspace=None, dev_status=None):
    """The scorer's gradients under the straight-through estimator; fp32
    (dq_low [B,H,Tq,P], dk_low [B,H,Tk,P])."""
    lib = load()
    dev = _dev(q_low, k_low, idx, dS, workspace, dev_status)
    if q_low.dtype != k_low.dtype:
        raise TypeError("q_low and k_low must share a dtype")
    if idx.dtype != torch.int32 or dS.dtype != torch.float32:
        raise TypeError("idx must be int32 and dS float32")
    B, H, Tq, P = q_low.shape
    Tk = k_low.shape[2]
    k = idx.shape[3]
    if tuple(dS.shape) != tuple(idx.shape) or idx.shape[:3] != (B, H, Tq):
        raise ValueError("idx/dS shapes do not match q_low")
    f32 = dict(dtype=torch.float32, device=dev)
    dq = torch.empty((B, H, Tq, P), **f32)
    dk = torch.empty((B, H, Tk, P), **f32)
    need = scorer_bwd_workspace_size(B, H, Tq, Tk, k)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    wbytes = workspace.numel() * workspace.element_size()
    rc = lib.ssa_scorer_bwd(_ptr(q_low), _ptr(k_low), _dt(q_low), B, H, Tq, Tk, P, _ptr(idx), k,
                            _ptr(dS), float(scale), _ptr(dq), _ptr(dk), _ptr(workspace), wbytes,
                            _ptr(dev_status), _stream(dev))
    _check(rc, "ssa_scorer_bwd")
    return dq, dk


def sparse_attn_scorer_bwd_workspace_size(B, H, Tq, Tk, k) -> int:
    return int(load().ssa_sparse_attn_scorer_bwd_workspace_size(B, H, Tq, Tk, k))


def ssa_sparse_attn_scorer_bwd(Q, K, V, dO, q_low, k_low, idx, scale: float = 0.0,
                               scorer_scale: float = 0.0, workspace=None, dev_status=None,
                               with_prob: bool = False):
    """ssa_sparse_attn_bwd then ssa_scorer_bwd in one call (the key-major lists
    built once). Returns fp32 (dQ, dK, dV, dS, dq_low, dk_low) (+ prob)."""
    lib = load()
    dev = _dev(Q, K, V, dO, q_low, k_low, idx, workspace, dev_status)
    if not (Q.dtype == K.dtype == V.dtype == dO.dtype == q_low.dtype == k_low.dtype):
        raise TypeError("Q, K, V, dO, q_low, k_low must share a dtype")
    if idx.dtype != torch.int32:
        raise TypeError("idx must be int32")
    B, H, Tq, D = Q.shape
    Tk, P, k = K.shape[2], q_low.shape[3], idx.shape[3]
    if (tuple(K.shape) != (B, H, Tk, D) or tuple(V.shape) != (B, H, Tk, D) or
            tuple(dO.shape) != (B, H, Tq, D) or tuple(q_low.shape) != (B, H, Tq, P) or
            tuple(k_low.shape) != (B, H, Tk, P) or tuple(idx.shape[:3]) != (B, H, Tq)):
        raise ValueError("shapes do not match")
    f32 = dict(dtype=torch.float32, device=dev)
    dQ = torch.empty((B, H, Tq, D), **f32)
    dK = torch.empty((B, H, Tk, D), **f32)
    dV = torch.empty((B, H, Tk, D), **f32)
    dS = torch.empty((B, H, Tq, k), **f32)
    dq = torch.empty((B, H, Tq, P), **f32)
    dk = torch.empty((B, H, Tk, P), **f32)
    prob = torch.empty((B, H, Tq, k), **f32) if with_prob else None
    need = sparse_attn_scorer_bwd_workspace_size(B, H, Tq, Tk, k)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    wbytes = workspace.numel() * workspace.element_size()
    rc = lib.ssa_sparse_attn_scorer_bwd(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(q_low), _ptr(k_low), _dt(Q), B, H, Tq, Tk, D, P,
        _ptr(idx), k, float(scale), float(scorer_scale), _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(dS),
        _ptr(prob), _ptr(dq), _ptr(dk), _ptr(workspace), wbytes, _ptr(dev_status), _stream(dev))
    _check(rc, "ssa_sparse_attn_scorer_bwd")
    out = (dQ, dK, dV, dS, dq, dk)
    return out + (prob,) if with_prob else out


def ssa_sparse_attn_grouped_bwd(Q, K, V, idx, dO, scale: float = 0.0, workspace=None,
                                dev_status=None, with_prob: bool = False):
    """ssa_sparse_attn_bwd for shared key/value heads and index lists: Q, dO
    [B,H,Tq,D]; K, V [B,H_kv,Tk,D]; idx [B,H_idx,Tq,k]. Returns fp32 (dQ
    [B,H,Tq,D], dK, dV [B,H_kv,Tk,D], dS [B,H,Tq,k]) (+ prob)."""
    lib = load()
    dev = _dev(Q, K, V, idx, dO, workspace, dev_status)
    if not (Q.dtype == K.dtype == V.dtype == dO.dtype):
        raise TypeError("Q, K, V, dO must share a dtype")
    if idx.dtype != torch.int32:
        raise TypeError("idx must be int32")
    B, H, Tq, D = Q.shape
    H_kv, Tk = K.shape[1], K.shape[2]
    H_idx, k = idx.shape[1], idx.shape[3]
    if tuple(K.shape) != (B, H_kv, Tk, D) or tuple(V.shape) != (B, H_kv, Tk, D) or \
            tuple(dO.shape) != (B, H, Tq, D) or tuple(idx.shape[:3]) != (B, H_idx, Tq):
        raise ValueError("shapes do not match: Q %s K %s V %s dO %s idx %s" % tuple(
            tuple(t.shape) for t in (Q, K, V, dO, idx)))
    f32 = dict(dtype=torch.float32, device=dev)
    dQ = torch.empty((B, H, Tq, D), **f32)
    dK = torch.empty((B, H_kv, Tk, D), **f32)
    dV = torch.empty((B, H_kv, Tk, D), **f32)
    dS = torch.empty((B, H, Tq, k), **f32)
    prob = torch.empty((B, H, Tq, k), **f32) if with_prob else None
    need = int(lib.ssa_sparse_attn_grouped_bwd_workspace_size(B, H, H_kv, Tq, Tk, k))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    wbytes = workspace.numel() * workspace.element_size()
    rc = lib.ssa_sparse_attn_grouped_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _dt(Q), B, H, H_kv,
                                         Tq, Tk, D, _ptr(idx), H_idx, k, float(scale), _ptr(dQ),
                                         _ptr(dK), _ptr(dV), _ptr(dS), _ptr(prob),
                                         _ptr(workspace), wbytes, _ptr(dev_status), _stream(dev))
    _check(rc, "ssa_sparse_attn_grouped_bwd")
    return (dQ, dK, dV, dS, prob) if with_prob else (dQ, dK, dV, dS)


def ssa_scorer_grouped_bwd(q_low, k_low, idx, dS, scale: float = 0.0, workspace=None,
                           dev_status=None):
    """The scorer's gradients for H_idx scorer heads shared by the H query
    heads of dS [B,H,Tq,k]; q_low [B,H_idx,Tq,P], k_low [B,H_idx,Tk,P], idx
    [B,H_idx,Tq,k]. Returns fp32 (dq_low, dk_low)."""
    lib = load()
    dev = _dev(q_low, k_low, idx, dS, workspace, dev_status)
    if q_low.dtype != k_low.dtype:
        raise TypeError("q_low and k_low must share a dtype")
    if idx.dtype != torch.int32 or dS.dtype != torch.float32:
        raise TypeError("idx must be int32 and dS float32")
    B, H_idx, Tq, P = q_low.shape
    Tk, k = k_low.shape[2], idx.shape[3]
    H = dS.shape[1]
    if tuple(idx.shape) != (B, H_idx, Tq, k) or tuple(dS.shape) != (B, H, Tq, k):
        raise ValueError("idx/dS shapes do not match q_low")
    f32 = dict(dtype=torch.float32, device=dev)
    dq = torch.empty((B, H_idx, Tq, P), **f32)
    dk = torch.empty((B, H_idx, Tk, P), **f32)
    need = int(lib.ssa_scorer_grouped_bwd_workspace_size(B, H, H_idx, Tq, Tk, k))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    wbytes = workspace.numel() * workspace.element_size()
    rc = lib.ssa_scorer_grouped_bwd(_ptr(q_low), _ptr(k_low), _dt(q_low), B, H, H_idx, Tq, Tk, P,
                                    _ptr(idx), k, _ptr(dS), float(scale), _ptr(dq), _ptr(dk),
                                    _ptr(workspace), wbytes, _ptr(dev_status), _stream(dev))
    _check(rc, "ssa_scorer_grouped_bwd")
    return dq, dk


def ssa_selftest_wait_limit(dev_status: torch.Tensor, limit_ns: int = 2_000_000):
    """Launch the bounded-wait self-test on the current stream: one block waits
    on an mbarrier nothing completes, gives up after limit_ns and ORs
    SSA_DEV_WAIT_LIMIT into dev_status (a device int32 tensor)."""
    lib = load()
    dev = _dev(dev_status)
    if dev_status.dtype != torch.int32:
        raise TypeError("dev_status must be int32")
    _check(lib.ssa_selftest_wait_limit(_ptr(dev_status), int(limit_ns), _stream(dev)),
           "ssa_selftest_wait_limit")


def device_status(dev_status: torch.Tensor):
    """Wait for the current stream, read the device-side error bits and return
    (status, bits): SSA_ERR_TIMEOUT when a bounded device wait ran out,
    SSA_ERR_INVALID when an index entry was out of range, else SSA_OK."""
    if dev_status.dtype != torch.int32 or dev_status.numel() < 1:
        raise TypeError("dev_status must be an int32 tensor")
    dev = _dev(dev_status)
    bits = ctypes.c_int32(0)
    rc = load().ssa_device_status(_ptr(dev_status), ctypes.cast(ctypes.byref(bits), ctypes.c_void_p),
                                  _stream(dev))
    if rc == SSA_ERR_CUDA:
        raise SSAError(rc, "ssa_device_status")
    return rc, int(bits.value)


def trace_begin():
    """Start timing every kernel the library launches (CUDA events on the
    launching stream)."""
    load().ssa_trace_begin()


def trace_end(max_records: int = 4096):
    """Stop tracing; returns [(kernel name, ms), ...] in launch order."""
    buf = (_TraceRecord * max_records)()
    n = load().ssa_trace_end(ctypes.cast(buf, ctypes.c_void_p), max_records)
    if n < 0:
        raise SSAError(SSA_ERR_CUDA, "ssa_trace_end")
    return [(buf[i].name.decode(), float(buf[i].ms)) for i in range(min(n, max_records))]


def default_scale(n: int) -> float:
    return 1.0 / math.sqrt(n)
