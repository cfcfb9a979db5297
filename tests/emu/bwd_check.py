"""The backward kernels under host emulation against the oracle (CPU).

build() compiles dynamic_top_sparse_rank_b300/csrc/attn_bwd.cu with
SSA_HOST_EMULATION (emu_device.h stands in for CUDA) into a host shared
library. check_all() calls its C entry points, ssa_sparse_attn_bwd and
ssa_scorer_bwd, exactly as a caller of libssa.so would, but with host buffers.
Each workspace is an exactly sized 256-byte-aligned block filled with garbage.
The outputs are compared with oracle.attn_bwd_rows / scorer_bwd_rows. Run as a
script, it exits non-zero on any mismatch (the AddressSanitizer run uses
that).

Inputs are exact in fp32 and the kernels sum in fp32, so one relative bound
serves both dtypes: TOL x the largest magnitude of the tensor.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402

TOL = 2e-5


def build(out_dir: str, asan: bool = False) -> str:
    out = os.path.join(out_dir, "libbwd_emu%s.so" % ("_asan" if asan else ""))
    cmd = ["g++", "-O1", "-std=c++17", "-fPIC", "-shared",
           "-I", HERE, "-I", os.path.join(ROOT, "dynamic_top_sparse_rank_b300", "csrc"),
           "-I", os.path.join(ROOT, "include"), os.path.join(HERE, "bwd_emu.cpp"), "-o", out]
    if asan:
        cmd[1:1] = ["-g", "-fsanitize=address", "-fno-omit-frame-pointer"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


class Emu:
    def __init__(self, path: str):
        self.lib = lib = ctypes.CDLL(path)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        for n in ("ssa_sparse_attn_bwd_workspace_size", "ssa_scorer_bwd_workspace_size"):
            getattr(lib, n).argtypes = [I] * 5
            getattr(lib, n).restype = Z
        lib.ssa_sparse_attn_bwd.argtypes = [P, P, P, P, I, I, I, I, I, I, P, I, F, P, P, P, P, P, P,
                                            Z, P, P]
        lib.ssa_sparse_attn_bwd.restype = I
        lib.ssa_scorer_bwd.argtypes = [P, P, I, I, I, I, I, I, P, I, P, F, P, P, P, Z, P, P]
        lib.ssa_scorer_bwd.restype = I
        lib.ssa_sparse_attn_grouped_bwd_workspace_size.argtypes = [I] * 6
        lib.ssa_sparse_attn_grouped_bwd_workspace_size.restype = Z
        lib.ssa_sparse_attn_grouped_bwd.argtypes = [P, P, P, P, I, I, I, I, I, I, I, P, I, I, F, P,
                                                    P, P, P, P, P, Z, P, P]
        lib.ssa_sparse_attn_grouped_bwd.restype = I
        lib.ssa_scorer_grouped_bwd_workspace_size.argtypes = [I] * 6
        lib.ssa_scorer_grouped_bwd_workspace_size.restype = Z
        lib.ssa_scorer_grouped_bwd.argtypes = [P, P, I, I, I, I, I, I, I, P, I, P, F, P, P, P, Z,
                                               P, P]
        lib.ssa_scorer_grouped_bwd.restype = I
        lib.ssa_sparse_attn_scorer_bwd_workspace_size.argtypes = [I] * 5
        lib.ssa_sparse_attn_scorer_bwd_workspace_size.restype = Z
        lib.ssa_sparse_attn_scorer_bwd.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, P, I, F,
                                                   F, P, P, P, P, P, P, P, P, Z, P, P]
        lib.ssa_sparse_attn_scorer_bwd.restype = I
        self.libc = libc = ctypes.CDLL(None)
        libc.aligned_alloc.argtypes = [Z, Z]
        libc.aligned_alloc.restype = P
        libc.free.argtypes = [P]
        libc.memset.argtypes = [P, I, Z]

    def _ws(self, n):
        p = self.libc.aligned_alloc(256, n)
        self.libc.memset(p, 0xA5, n)
        return p

    def attn_bwd(self, Q, K, V, dO, idx):
        """Q, dO [B,H,Tq,D], K, V [B,H,Tk,D] torch (bf16 or fp32); idx int32 numpy."""
        B, H, Tq, D = Q.shape
        Tk, k = K.shape[2], idx.shape[-1]
        bufs = [_raw(t) for t in (Q, K, V, dO)]
        outs = dict(dQ=np.full((B, H, Tq, D), np.nan, np.float32),
                    dK=np.full((B, H, Tk, D), np.nan, np.float32),
                    dV=np.full((B, H, Tk, D), np.nan, np.float32),
                    dS=np.full((B, H, Tq, k), np.nan, np.float32),
                    prob=np.full((B, H, Tq, k), np.nan, np.float32))
        st = np.zeros(1, np.int32)
        ix = np.ascontiguousarray(idx, np.int32)
        n = self.lib.ssa_sparse_attn_bwd_workspace_size(B, H, Tq, Tk, k)
        ws = self._ws(n)
        rc = self.lib.ssa_sparse_attn_bwd(
            *[_p(b) for b in bufs], int(Q.dtype == torch.bfloat16), B, H, Tq, Tk, D, _p(ix), k,
            0.0, *[_p(outs[n_]) for n_ in ("dQ", "dK", "dV", "dS", "prob")], ws, n, _p(st), None)
        self.libc.free(ws)
        return rc, outs, int(st[0])

    def scorer_bwd(self, ql, kl, idx, dS):
        B, H, Tq, P = ql.shape
        Tk, k = kl.shape[2], idx.shape[-1]
        dq = np.full((B, H, Tq, P), np.nan, np.float32)
        dk = np.full((B, H, Tk, P), np.nan, np.float32)
        st = np.zeros(1, np.int32)
        ix = np.ascontiguousarray(idx, np.int32)
        g = np.ascontiguousarray(dS, np.float32)
        n = self.lib.ssa_scorer_bwd_workspace_size(B, H, Tq, Tk, k)
        ws = self._ws(n)
        rc = self.lib.ssa_scorer_bwd(_p(_raw(ql)), _p(_raw(kl)), int(ql.dtype == torch.bfloat16),
                                     B, H, Tq, Tk, P, _p(ix), k, _p(g), 0.0, _p(dq), _p(dk), ws, n,
                                     _p(st), None)
        self.libc.free(ws)
        return rc, dq, dk, int(st[0])

    def fused_bwd(self, Q, K, V, dO, ql, kl, idx):
        """ssa_sparse_attn_scorer_bwd: both backward calls with one list build."""
        B, H, Tq, D = Q.shape
        Tk, k, P = K.shape[2], idx.shape[-1], ql.shape[-1]
        bufs = [_raw(t) for t in (Q, K, V, dO, ql, kl)]
        outs = dict(dQ=np.full((B, H, Tq, D), np.nan, np.float32),
                    dK=np.full((B, H, Tk, D), np.nan, np.float32),
                    dV=np.full((B, H, Tk, D), np.nan, np.float32),
                    dS=np.full((B, H, Tq, k), np.nan, np.float32),
                    prob=np.full((B, H, Tq, k), np.nan, np.float32),
                    dq=np.full((B, H, Tq, P), np.nan, np.float32),
                    dk=np.full((B, H, Tk, P), np.nan, np.float32))
        st = np.zeros(1, np.int32)
        ix = np.ascontiguousarray(idx, np.int32)
        n = self.lib.ssa_sparse_attn_scorer_bwd_workspace_size(B, H, Tq, Tk, k)
        ws = self._ws(n)
        rc = self.lib.ssa_sparse_attn_scorer_bwd(
            *[_p(b) for b in bufs], int(Q.dtype == torch.bfloat16), B, H, Tq, Tk, D, P, _p(ix), k,
            0.0, 0.0, *[_p(outs[n_]) for n_ in ("dQ", "dK", "dV", "dS", "prob", "dq", "dk")], ws,
            n, _p(st), None)
        self.libc.free(ws)
        return rc, outs, int(st[0])

    def grouped_attn_bwd(self, Q, K, V, dO, idx):
        """Q, dO [B,H,Tq,D]; K, V [B,H_kv,Tk,D]; idx [B,H_idx,Tq,k]."""
        B, H, Tq, D = Q.shape
        H_kv, Tk = K.shape[1], K.shape[2]
        H_idx, k = idx.shape[1], idx.shape[3]
        bufs = [_raw(t) for t in (Q, K, V, dO)]
        outs = dict(dQ=np.full((B, H, Tq, D), np.nan, np.float32),
                    dK=np.full((B, H_kv, Tk, D), np.nan, np.float32),
                    dV=np.full((B, H_kv, Tk, D), np.nan, np.float32),
                    dS=np.full((B, H, Tq, k), np.nan, np.float32))
        st = np.zeros(1, np.int32)
        ix = np.ascontiguousarray(idx, np.int32)
        n = self.lib.ssa_sparse_attn_grouped_bwd_workspace_size(B, H, H_kv, Tq, Tk, k)
        ws = self._ws(n)
        rc = self.lib.ssa_sparse_attn_grouped_bwd(
            *[_p(b) for b in bufs], int(Q.dtype == torch.bfloat16), B, H, H_kv, Tq, Tk, D, _p(ix),
            H_idx, k, 0.0, *[_p(outs[n_]) for n_ in ("dQ", "dK", "dV", "dS")], None, ws, n, _p(st),
            None)
        self.libc.free(ws)
        return rc, outs, int(st[0])


    def grouped_scorer_bwd(self, ql, kl, idx, dS):
        """ql, kl, idx with H_idx heads; dS [B,H,Tq,k] of the H query heads."""
        B, H_idx, Tq, P = ql.shape
        Tk, k = kl.shape[2], idx.shape[-1]
        H = dS.shape[1]
        dq = np.full((B, H_idx, Tq, P), np.nan, np.float32)
        dk = np.full((B, H_idx, Tk, P), np.nan, np.float32)
        st = np.zeros(1, np.int32)
        ix = np.ascontiguousarray(idx, np.int32)
        g = np.ascontiguousarray(dS, np.float32)
        n = self.lib.ssa_scorer_grouped_bwd_workspace_size(B, H, H_idx, Tq, Tk, k)
        ws = self._ws(n)
        rc = self.lib.ssa_scorer_grouped_bwd(_p(_raw(ql)), _p(_raw(kl)), int(ql.dtype == torch.bfloat16),
                                             B, H, H_idx, Tq, Tk, P, _p(ix), k, _p(g), 0.0, _p(dq),
                                             _p(dk), ws, n, _p(st), None)
        self.libc.free(ws)
        return rc, dq, dk, int(st[0])




def _raw(t):
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).numpy().copy()
    return t.contiguous().numpy().copy()


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _close(got, ref, what, fails):
    ref = np.asarray(ref, np.float64)
    bound = TOL * max(1.0, float(np.abs(ref).max(initial=0.0)))
    err = float(np.abs(np.asarray(got, np.float64) - ref).max(initial=0.0))
    if not err <= bound:   # also catches NaN (an output never written)
        fails.append("%s: max err %.3g > %.3g" % (what, err, bound))


def attn_inputs(B, H, Tq, Tk, D, k, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    mk = lambda T: torch.randn(B, H, T, D, generator=g).to(dtype)  # noqa: E731
    rng = np.random.default_rng(seed)
    idx = rng.integers(0, max(Tk, 1), size=(B, H, Tq, k)).astype(np.int32)   # repeats allowed
    if k > 1:
        idx[..., -1] = -1                   # a padded slot
    if Tq > 0:
        idx[0, 0, 0, :] = -1                # an empty row
    if Tk == 0:
        idx[:] = -1
    return mk(Tq), mk(Tk), mk(Tk), mk(Tq), idx


ATTN_CASES = [
    # B, H, Tq, Tk, D, k, dtype, seed
    (1, 2, 20, 50, 64, 7, torch.bfloat16, 1),
    (2, 1, 33, 70, 128, 40, torch.bfloat16, 2),
    (1, 1, 17, 40, 64, 5, torch.float32, 3),
    (1, 1, 9, 1500, 128, 64, torch.float32, 4),     # Tk > 1024: several keys per scan thread
    (1, 1, 40, 12, 64, 1, torch.bfloat16, 5),      # k = 1
    (1, 1, 3, 40, 128, 70, torch.float32, 6),      # k > Tk: repeats in every row
]

SCORER_CASES = [
    # B, H, Tq, Tk, P, k, dtype
    (1, 2, 30, 80, 64, 9, torch.bfloat16),
    (1, 1, 25, 40, 16, 6, torch.float32),
    (2, 1, 10, 300, 128, 33, torch.bfloat16),
    (1, 1, 12, 20, 32, 4, torch.float32),
]


def check_attn(emu, case, fails):
    B, H, Tq, Tk, D, k, dtype, seed = case
    Q, K, V, dO, idx = attn_inputs(B, H, Tq, Tk, D, k, dtype, seed)
    rc, o, st = emu.attn_bwd(Q, K, V, dO, idx)
    tag = "attn %s" % (case[:7],)
    if rc != 0 or st != 0:
        fails.append("%s: status %d, device status %d" % (tag, rc, st))
        return
    rQ, rK, rV, rS = oracle.sparse_attn_bwd(Q, K, V, idx, dO)
    for n_, r in (("dQ", rQ), ("dK", rK), ("dV", rV), ("dS", rS)):
        _close(o[n_], r, "%s %s" % (tag, n_), fails)
    live = idx >= 0
    p = o["prob"]
    if not ((p[~live] == 0).all() and np.allclose(p.sum(-1)[live.any(-1)], 1.0, atol=1e-6)):
        fails.append("%s: weights not zero in padding or not summing to 1" % tag)


def check_scorer(emu, case, fails):
    B, H, Tq, Tk, P, k, dtype = case
    g = torch.Generator().manual_seed(P + k)
    ql = torch.randn(B, H, Tq, P, generator=g).to(dtype)
    kl = torch.randn(B, H, Tk, P, generator=g).to(dtype)
    rng = np.random.default_rng(P)
    idx = rng.integers(0, Tk, size=(B, H, Tq, k)).astype(np.int32)
    idx[..., -1] = -1
    idx[0, 0, 0, :] = -1
    dS = rng.standard_normal((B, H, Tq, k)).astype(np.float32)
    rc, dq, dk, st = emu.scorer_bwd(ql, kl, idx, dS)
    tag = "scorer %s" % (case,)
    if rc != 0 or st != 0:
        fails.append("%s: status %d, device status %d" % (tag, rc, st))
        return
    rq, rk = oracle.scorer_bwd(ql, kl, idx, dS)
    _close(dq, rq, tag + " dq_low", fails)
    _close(dk, rk, tag + " dk_low", fails)


FUSED_CASES = [
    # B, H, Tq, Tk, D, P, k, dtype, seed
    (1, 2, 30, 80, 64, 64, 9, torch.bfloat16, 11),
    (2, 1, 12, 40, 128, 16, 6, torch.float32, 12),
]


def check_fused(emu, case, fails):
    """ssa_sparse_attn_scorer_bwd against the oracle: the attention's and the
    scorer's gradients of one backward step, the lists built once."""
    B, H, Tq, Tk, D, P, k, dtype, seed = case
    Q, K, V, dO, idx = attn_inputs(B, H, Tq, Tk, D, k, dtype, seed)
    g = torch.Generator().manual_seed(seed)
    ql = torch.randn(B, H, Tq, P, generator=g).to(dtype)
    kl = torch.randn(B, H, Tk, P, generator=g).to(dtype)
    rc, o, st = emu.fused_bwd(Q, K, V, dO, ql, kl, idx)
    tag = "fused %s" % (case[:8],)
    if rc != 0 or st != 0:
        fails.append("%s: status %d, device status %d" % (tag, rc, st))
        return
    rQ, rK, rV, rS = oracle.sparse_attn_bwd(Q, K, V, idx, dO)
    for n_, r in (("dQ", rQ), ("dK", rK), ("dV", rV), ("dS", rS)):
        _close(o[n_], r, "%s %s" % (tag, n_), fails)
    # the scorer's gradients from the dS the call produced
    rq, rk = oracle.scorer_bwd(ql, kl, idx, o["dS"])
    _close(o["dq"], rq, tag + " dq_low", fails)
    _close(o["dk"], rk, tag + " dk_low", fails)


GROUPED_CASES = [
    # B, H, H_kv, H_idx, Tq, Tk, D, k, dtype
    (2, 4, 2, 1, 15, 40, 64, 6, torch.bfloat16),     # grouped-query heads, one shared scorer
    (1, 4, 1, 2, 11, 30, 128, 5, torch.float32),     # one key/value head, two index heads
    (1, 6, 3, 3, 9, 50, 64, 7, torch.bfloat16),
    (1, 3, 3, 1, 13, 20, 64, 4, torch.bfloat16),     # the pages' layout: shared scorer only
]


def check_grouped(emu, case, fails):
    B, H, H_kv, H_idx, Tq, Tk, D, k, dtype = case
    g = torch.Generator().manual_seed(H * 10 + H_kv)
    Q = torch.randn(B, H, Tq, D, generator=g).to(dtype)
    dO = torch.randn(B, H, Tq, D, generator=g).to(dtype)
    K = torch.randn(B, H_kv, Tk, D, generator=g).to(dtype)
    V = torch.randn(B, H_kv, Tk, D, generator=g).to(dtype)
    rng = np.random.default_rng(H_idx + 7 * k)
    idx = rng.integers(0, Tk, size=(B, H_idx, Tq, k)).astype(np.int32)
    idx[..., -1] = -1
    idx[0, 0, 0, :] = -1
    tag = "grouped %s" % (case,)
    rc, o, st = emu.grouped_attn_bwd(Q, K, V, dO, idx)
    if rc != 0 or st != 0:
        fails.append("%s: status %d, device status %d" % (tag, rc, st))
        return
    ref = oracle.sparse_attn_grouped_bwd(Q, K, V, idx, dO)
    for n_, r in zip(("dQ", "dK", "dV", "dS"), ref):
        _close(o[n_], r, "%s %s" % (tag, n_), fails)
    P = 16
    ql = torch.randn(B, H_idx, Tq, P, generator=g).to(dtype)
    kl = torch.randn(B, H_idx, Tk, P, generator=g).to(dtype)
    rc, dq, dk, st = emu.grouped_scorer_bwd(ql, kl, idx, o["dS"])
    if rc != 0 or st != 0:
        fails.append("%s scorer: status %d, device status %d" % (tag, rc, st))
        return
    rq, rk = oracle.scorer_grouped_bwd(ql, kl, idx, o["dS"])
    _close(dq, rq, tag + " dq_low", fails)
    _close(dk, rk, tag + " dk_low", fails)


def check_near_equal_values(emu, fails):
    """Value rows that differ by 1% of their size make the dp of a row nearly
    equal, and dQ = sum_t p_t (dp_t - delta) K_t small next to its terms.
    dQ must keep the accuracy that dS (the same differences) has: 5e-4 of its
    largest entry. Accumulating dp K unshifted loses about 1e-3 here."""
    B, H, Tq, Tk, D, k = 1, 1, 16, 600, 128, 512
    g = torch.Generator().manual_seed(3)
    Q = torch.randn(B, H, Tq, D, generator=g)
    K = torch.randn(B, H, Tk, D, generator=g)
    V = 3 * torch.randn(1, 1, 1, D, generator=g) + 1e-2 * torch.randn(B, H, Tk, D, generator=g)
    dO = torch.randn(B, H, Tq, D, generator=g)
    rng = np.random.default_rng(4)
    idx = np.stack([rng.choice(Tk, k, replace=False) for _ in range(Tq)])[None, None]
    rc, o, st = emu.attn_bwd(Q, K, V, dO, idx.astype(np.int32))
    rQ, _, _, rS = oracle.sparse_attn_bwd(Q, K, V, idx, dO)
    for n_, got, ref in (("dQ", o["dQ"], rQ), ("dS", o["dS"], rS)):
        err = float(np.abs(got - ref).max())
        if rc != 0 or not err <= 5e-4 * float(np.abs(ref).max()):
            fails.append("near-equal value rows: %s error %.3g of max %.3g" % (
                n_, err, float(np.abs(ref).max())))


def check_edges(emu, fails):
    # an index outside [-1, Tk): reported, skipped
    Q, K, V, dO, idx = attn_inputs(1, 1, 8, 16, 64, 4, torch.bfloat16, 10)
    idx[0, 0, 3, 1] = 16 + 2
    rc, o, st = emu.attn_bwd(Q, K, V, dO, idx)
    ref = oracle.sparse_attn_bwd(Q, K, V, np.where(idx < 16, idx, -1).astype(np.int32), dO)
    if rc != 0 or not st & 1 or o["dS"][0, 0, 3, 1] != 0:
        fails.append("bad index: status %d, device status %d" % (rc, st))
    for n_, r in zip(("dQ", "dK", "dV", "dS"), ref):
        _close(o[n_], r, "bad index " + n_, fails)
    # no keys: every query-side gradient is zero
    Q, K, V, dO, idx = attn_inputs(1, 2, 6, 0, 64, 3, torch.bfloat16, 11)
    rc, o, st = emu.attn_bwd(Q, K, V, dO, idx)
    if rc != 0 or not all((o[n_] == 0).all() for n_ in ("dQ", "dS", "prob")):
        fails.append("Tk = 0: status %d or non-zero gradients" % rc)
    # no query rows: the key gradients are zero
    Q, K, V, dO, idx = attn_inputs(1, 2, 0, 30, 64, 3, torch.bfloat16, 12)
    rc, o, st = emu.attn_bwd(Q, K, V, dO, idx)
    if rc != 0 or not ((o["dK"] == 0).all() and (o["dV"] == 0).all()):
        fails.append("Tq = 0: status %d or non-zero key gradients" % rc)


def check_binding(emu, fails):
    """The Python binding (ssa_sparse_attn_bwd, ssa_scorer_bwd) over the
    emulated library: the same marshalling code, with host tensors standing
    in for device ones (placement checks and the stream lookup are bypassed)
    and a 256-byte-aligned host workspace."""
    from dynamic_top_sparse_rank_b300 import _native
    saved = (_native._lib, _native._dev, _native._stream)
    try:
        _native._lib = emu.lib
        _native._dev = lambda *ts: torch.device("cpu")
        _native._stream = lambda dev: None

        def ws(n):
            buf = torch.empty(n + 256, dtype=torch.uint8)
            off = (-buf.data_ptr()) % 256
            return buf[off:off + n]

        B, H, Tq, Tk, D, k, P = 1, 2, 12, 40, 64, 6, 16
        Q, K, V, dO, idx = attn_inputs(B, H, Tq, Tk, D, k, torch.bfloat16, 21)
        it = torch.from_numpy(idx)
        n = emu.lib.ssa_sparse_attn_bwd_workspace_size(B, H, Tq, Tk, k)
        dQ, dK, dV, dS, p = _native.ssa_sparse_attn_bwd(Q, K, V, it, dO, workspace=ws(n),
                                                        with_prob=True)
        ref = oracle.sparse_attn_bwd(Q, K, V, idx, dO)
        for n_, a, r in zip(("dQ", "dK", "dV", "dS"), (dQ, dK, dV, dS), ref):
            _close(a.numpy(), r, "binding " + n_, fails)
        g = torch.Generator().manual_seed(5)
        ql = torch.randn(B, H, Tq, P, generator=g)
        kl = torch.randn(B, H, Tk, P, generator=g)
        n = emu.lib.ssa_scorer_bwd_workspace_size(B, H, Tq, Tk, k)
        dq, dk = _native.ssa_scorer_bwd(ql, kl, it, dS, workspace=ws(n))
        rq, rk = oracle.scorer_bwd(ql, kl, idx, dS.numpy())
        _close(dq.numpy(), rq, "binding dq_low", fails)
        _close(dk.numpy(), rk, "binding dk_low", fails)
        # the grouped calls: 4 query heads on 2 key/value heads and 1 scorer head
        Qg = torch.cat([Q, Q.flip(1)], dim=1)
        dOg = torch.cat([dO, dO.flip(1)], dim=1)
        Kg, Vg = K, V
        ig = it[:, :1].contiguous()
        n = emu.lib.ssa_sparse_attn_grouped_bwd_workspace_size(B, 2 * H, H, Tq, Tk, k)
        gQ, gK, gV, gS = _native.ssa_sparse_attn_grouped_bwd(Qg, Kg, Vg, ig, dOg, workspace=ws(n))
        ref = oracle.sparse_attn_grouped_bwd(Qg, Kg, Vg, ig.numpy(), dOg)
        for n_, a, r in zip(("dQ", "dK", "dV", "dS"), (gQ, gK, gV, gS), ref):
            _close(a.numpy(), r, "grouped binding " + n_, fails)
        n = emu.lib.ssa_scorer_grouped_bwd_workspace_size(B, 2 * H, 1, Tq, Tk, k)
        gq, gk = _native.ssa_scorer_grouped_bwd(ql[:, :1].contiguous(), kl[:, :1].contiguous(), ig,
                                                gS, workspace=ws(n))
        rq, rk = oracle.scorer_grouped_bwd(ql[:, :1], kl[:, :1], ig.numpy(), gS.numpy())
        _close(gq.numpy(), rq, "grouped binding dq_low", fails)
        _close(gk.numpy(), rk, "grouped binding dk_low", fails)
    finally:
        _native._lib, _native._dev, _native._stream = saved


def check_random_shapes(emu, n, seed, fails):
    """n seeded random grouped shapes (plain when H_kv = H_idx = H): heads and
    their sharing, ragged lengths, k from 1 past Tk, head size, dtype."""
    g = np.random.default_rng(seed)
    for _ in range(n):
        H = int(g.choice([1, 2, 4]))
        H_kv = int(g.choice([d for d in (1, 2, 4) if H % d == 0]))
        H_idx = int(g.choice([d for d in (1, 2, 4) if H % d == 0]))
        case = (int(g.integers(1, 3)), H, H_kv, H_idx, int(g.integers(1, 40)),
                int(g.integers(1, 200)), int(g.choice([64, 128])), int(g.integers(1, 70)),
                torch.bfloat16 if g.integers(0, 2) else torch.float32)
        check_grouped(emu, case, fails)


def check_all(path: str, attn_cases=ATTN_CASES, scorer_cases=SCORER_CASES, edges=True,
              grouped_cases=GROUPED_CASES):
    emu = Emu(path)
    fails = []
    check_binding(emu, fails)
    for c in grouped_cases:
        check_grouped(emu, c, fails)
    for c in attn_cases:
        check_attn(emu, c, fails)
    for c in scorer_cases:
        check_scorer(emu, c, fails)
    for c in (FUSED_CASES if edges else FUSED_CASES[:1]):
        check_fused(emu, c, fails)
    if edges:
        check_edges(emu, fails)
        check_near_equal_values(emu, fails)
        if len(grouped_cases) == len(GROUPED_CASES):   # the full run, not the small one
            check_random_shapes(emu, 8, 7, fails)
    return fails


if __name__ == "__main__":
    # python bwd_check.py LIB [small]: check (a small set of cases) and exit 1 on a mismatch
    small = len(sys.argv) > 2 and sys.argv[2] == "small"
    f = check_all(sys.argv[1], ATTN_CASES[:2] if small else ATTN_CASES,
                  SCORER_CASES[:1] if small else SCORER_CASES,
                  grouped_cases=GROUPED_CASES[:1] if small else GROUPED_CASES)
    print("\n".join(f) if f else "OK")
    sys.exit(1 if f else 0)
