"""The forward's CUDA-core kernels under host emulation against the oracle
(CPU): the row-wise exact top-k (topk_rows_kernel), the gather and window
attention (attn_rows_kernel, plain and grouped heads) and the boundary
smoothing (smooth_boundary_kernel). build() compiles fwd_emu.cpp, which
includes the library's kernel files with SSA_HOST_EMULATION. check_all()
launches the kernels as the library does, on host buffers. Run as a script,
it exits non-zero on any mismatch (the AddressSanitizer run uses that).

Top-k: integer scorer data, so every score is exact and the indices and
scores must match the oracle bit for bit. Attention: the tolerances of the
GPU parity tests, 2e-3 for bf16 inputs and 1e-5 for fp32 inputs, on an fp32
output. A bf16 output may also sit within one bf16 ulp of the exact value
rounded to bf16.
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

TOPK_SLOTS = 64   # row slots of the workspace (the library uses up to 1024)


def build(out_dir: str, asan: bool = False) -> str:
    out = os.path.join(out_dir, "libfwd_emu%s.so" % ("_asan" if asan else ""))
    cmd = ["g++", "-O1", "-std=c++17", "-fPIC", "-shared",
           "-I", HERE, "-I", os.path.join(ROOT, "dynamic_top_sparse_rank_b300", "csrc"),
           "-I", os.path.join(ROOT, "include"), os.path.join(HERE, "fwd_emu.cpp"), "-o", out]
    if asan:
        cmd[1:1] = ["-g", "-fsanitize=address", "-fno-omit-frame-pointer"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def _raw(t):
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).numpy().copy()
    return t.contiguous().numpy().copy()


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Emu:
    def __init__(self, path):
        self.lib = lib = ctypes.CDLL(path)
        P, I, F, L = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_int64
        lib.emu_topk_rows.argtypes = [P, P, I, I, P, L, I, I, I, I, F, P, P, P, L, L]
        lib.emu_attn_rows.argtypes = [P, P, P, I, I, P, P, I, L, I, I, I, I, I, F, P, I, I, I, I,
                                      I, I]
        lib.emu_smooth.argtypes = [P, P, L, I, F]
        lib.emu_topk_chunks.argtypes = [P, P, I, I, L, I, I, I, I, F, P, P, P, P]
        lib.emu_topk_chunk_count.argtypes = [I, I]

    def topk(self, q, kl, k, causal, scale, row_list=None):
        """q [n_head_rows..] as [BH, Tq, P], kl [BH, Tk, P] torch; returns idx, score."""
        BH, Tq, P = q.shape
        Tk = kl.shape[1]
        rows = BH * Tq if row_list is None else len(row_list)
        idx = np.full((BH * Tq, k), -7, np.int32)
        sc = np.full((BH * Tq, k), np.nan, np.float32)
        stride = (Tk + 63) // 64 * 64
        ws = np.full(max(1, min(rows, TOPK_SLOTS) * stride), 0xA5A5A5A5, np.uint32)
        rl = None if row_list is None else np.ascontiguousarray(row_list, np.int64)
        rc = self.lib.emu_topk_rows(_p(_raw(q)), _p(_raw(kl)), int(q.dtype == torch.bfloat16), P,
                                    _p(rl), rows, Tq, Tk, k, int(causal), scale, _p(idx), _p(sc),
                                    _p(ws), TOPK_SLOTS, stride)
        assert rc == 0
        return idx.reshape(BH, Tq, k), sc.reshape(BH, Tq, k)

    def topk_chunks(self, q, kl, k, causal, scale):
        """The long-row path (chunk selections, then the merge); garbage-filled
        scratch of exactly the size the library's workspace gives it."""
        BH, Tq, P = q.shape
        Tk = kl.shape[1]
        rows = BH * Tq
        nchunks = self.lib.emu_topk_chunk_count(Tk, k)
        assert nchunks > 0
        kcap = min(k, 8192)
        cand = np.full(rows * nchunks * kcap, 0xA5A5A5A5A5A5A5A5, np.uint64)
        cnt = np.full(rows * nchunks, -9, np.int32)
        idx = np.full((rows, k), -7, np.int32)
        sc = np.full((rows, k), np.nan, np.float32)
        rc = self.lib.emu_topk_chunks(_p(_raw(q)), _p(_raw(kl)), int(q.dtype == torch.bfloat16), P,
                                      rows, Tq, Tk, k, int(causal), scale, _p(idx), _p(sc),
                                      _p(cand), _p(cnt))
        assert rc == 0
        return idx.reshape(BH, Tq, k), sc.reshape(BH, Tq, k)

    def attn(self, Q, K, V, idx, out_bf16, scale, H=1, H_kv=1, H_idx=1, grouped=0, head_inner=0,
             band=None):
        """Q [B*H, Tq, D] etc. flattened per head; idx [rows_of_idx, k] or None (band)."""
        rows = Q.shape[0] * Q.shape[1]
        Tq, D = Q.shape[1], Q.shape[2]
        Tk = K.shape[1]
        O = np.full((rows, D), np.nan, np.float32) if not out_bf16 else \
            np.full((rows, D), 0x7FC0, np.uint16)
        st = np.zeros(1, np.int32)
        k = 1 if idx is None else idx.shape[-1]
        ix = None if idx is None else np.ascontiguousarray(idx, np.int32)
        wl, wr = band if band is not None else (0, 0)
        rc = self.lib.emu_attn_rows(_p(_raw(Q)), _p(_raw(K)), _p(_raw(V)),
                                    int(Q.dtype == torch.bfloat16), D, _p(ix), _p(O), int(out_bf16),
                                    rows, Tq, Tk, k, wl, wr, scale, _p(st), H, H_kv, H_idx, grouped,
                                    head_inner, int(band is not None))
        assert rc == 0
        if out_bf16:
            O = (O.astype(np.uint32) << 16).view(np.float32)
        return O, int(st[0])


def _bf16_round(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).float().numpy()


def _bf16_ulp(x):
    a = np.maximum(np.abs(np.asarray(x, np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def _out_close(got, ref, tol, bf16_out, what, fails):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    ok = err <= tol
    if bf16_out:
        ok |= np.abs(got - _bf16_round(ref)) <= _bf16_ulp(ref)
    if not ok.all():
        fails.append("%s: max err %.3g" % (what, float(np.nanmax(err))))


def _ints(shape, seed, dtype):
    g = np.random.default_rng(seed)
    return torch.from_numpy(g.integers(-4, 5, size=shape).astype(np.float32)).to(dtype)


TOPK_CASES = [
    # BH, Tq, Tk, P, k, causal, dtype
    (2, 40, 40, 64, 8, True, torch.bfloat16),
    (1, 30, 300, 16, 33, False, torch.float32),
    (1, 50, 20, 32, 30, True, torch.bfloat16),      # Tq > Tk: early rows have no key; k > valid
    (1, 9, 1000, 128, 100, True, torch.bfloat16),   # Tq < Tk, several digits of the radix select
    (2, 12, 77, 64, 77, False, torch.float32),      # k = Tk: every key
    (1, 6, 150, 64, 5, False, torch.bfloat16),
    (1, 2, 6000, 64, 512, False, torch.bfloat16),   # the decode shape's k
    (1, 1, 5000, 128, 2048, False, torch.float32),  # the largest k
]


def check_topk(emu, case, fails):
    BH, Tq, Tk, P, k, causal, dtype = case
    q = _ints((BH, Tq, P), 100 + Tq, dtype)
    kl = _ints((BH, Tk, P), 200 + Tk, dtype)
    scale = float(np.float32(P ** -0.5))
    idx, sc = emu.topk(q, kl, k, causal, scale)
    for h in range(BH):
        ri, rs = oracle.topk_rows(q[h], np.arange(Tq), kl[h], k, Tq, causal)
        if not (np.array_equal(idx[h], ri) and np.array_equal(sc[h], rs)):
            bad = np.argwhere((idx[h] != ri).any(-1))[:3].ravel().tolist()
            fails.append("topk %s head %d: rows %s differ" % (case, h, bad))


def check_topk_ties_and_list(emu, fails):
    # every score equal: the lowest indices, in order
    q = torch.zeros(1, 20, 64, dtype=torch.bfloat16)
    kl = _ints((1, 90, 64), 5, torch.bfloat16)
    idx, sc = emu.topk(q, kl, 17, False, 0.125)
    if not (idx[0] == np.arange(17)).all():
        fails.append("topk all ties: not the 17 lowest indices")
    # a row list (the rows the tensor-core path hands back): only those rows
    q = _ints((2, 30, 64), 6, torch.bfloat16)
    kl = _ints((2, 60, 64), 7, torch.bfloat16)
    rows = np.array([3, 31, 59, 0], np.int64)
    idx, sc = emu.topk(q, kl, 9, True, 0.125, row_list=rows)
    flat = idx.reshape(-1, 9)
    for r in rows:
        h, i = divmod(int(r), 30)
        ri, _ = oracle.topk_rows(q[h][i:i + 1], np.array([i]), kl[h], 9, 30, True)
        if not np.array_equal(flat[r], ri[0]):
            fails.append("topk row list: row %d differs" % r)
    untouched = np.setdiff1d(np.arange(60), rows)
    if not (flat[untouched] == -7).all():
        fails.append("topk row list: a row outside the list was written")


CHUNK_CASES = [
    # BH, Tq, Tk, P, k, causal, dtype: rows of 2 or 3 key chunks of 8192
    (2, 1, 20000, 64, 64, False, torch.bfloat16),     # a ragged last chunk
    (1, 3, 17000, 32, 512, True, torch.float32),      # causal, Tq < Tk: rows end in chunk 2
    (1, 1, 16384, 64, 512, False, torch.bfloat16),    # two whole chunks, the decode k
]


def check_topk_chunks(emu, case, fails):
    BH, Tq, Tk, P, k, causal, dtype = case
    q = _ints((BH, Tq, P), 300 + Tq, dtype)
    kl = _ints((BH, Tk, P), 400 + Tk, dtype)
    scale = float(np.float32(P ** -0.5))
    idx, sc = emu.topk_chunks(q, kl, k, causal, scale)
    for h in range(BH):
        ri, rs = oracle.topk_rows(q[h], np.arange(Tq), kl[h], k, Tq, causal)
        if not (np.array_equal(idx[h], ri) and np.array_equal(sc[h], rs)):
            bad = np.argwhere((idx[h] != ri).any(-1))[:3].ravel().tolist()
            fails.append("topk chunks %s head %d: rows %s differ" % (case, h, bad))
    # all scores equal: the lowest indices of the row, across chunks
    q0 = torch.zeros(1, 1, 64, dtype=torch.bfloat16)
    kl0 = _ints((1, 16500, 64), 9, torch.bfloat16)
    idx0, _ = emu.topk_chunks(q0, kl0, 100, False, 0.125)
    if not (idx0[0, 0] == np.arange(100)).all():
        fails.append("topk chunks all ties: not the 100 lowest indices")


ATTN_CASES = [
    # B*H, Tq, Tk, D, k, dtype, out_bf16
    (2, 30, 100, 128, 7, torch.bfloat16, False),
    (1, 33, 400, 64, 40, torch.bfloat16, True),
    (2, 20, 90, 64, 5, torch.float32, False),
    (1, 17, 300, 128, 96, torch.float32, True),
    (1, 25, 50, 64, 1, torch.bfloat16, False),
]


def _normal(shape, seed, dtype):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(dtype)


def check_attn(emu, case, fails):
    BH, Tq, Tk, D, k, dtype, out_bf16 = case
    Q, K, V = (_normal((BH, T, D), 300 + n, dtype) for n, T in enumerate((Tq, Tk, Tk)))
    g = np.random.default_rng(k)
    idx = g.integers(0, Tk, size=(BH, Tq, k)).astype(np.int32)   # repeats allowed
    if k > 1:
        idx[..., -1] = -1
    idx[0, 0, :] = -1                                             # an empty row
    O, st = emu.attn(Q, K, V, idx.reshape(-1, k), out_bf16, D ** -0.5)
    tol = 1e-5 if dtype == torch.float32 else 2e-3
    if st != 0:
        fails.append("attn %s: device status %d" % (case, st))
    for h in range(BH):
        ref, _ = oracle.attn_rows(Q[h], K[h], V[h], idx[h])
        _out_close(O.reshape(BH, Tq, D)[h], ref, tol, out_bf16, "attn %s head %d" % (case, h),
                   fails)
    # a bad entry is reported and skipped
    bad = idx.copy()
    bad[0, 1, 0] = Tk + 3
    O2, st = emu.attn(Q, K, V, bad.reshape(-1, k), out_bf16, D ** -0.5)
    if not st & 1:
        fails.append("attn %s: bad index not reported" % (case,))


def check_window(emu, fails):
    for (BH, T, D, wl, wr, dtype) in [(2, 70, 64, 5, 5, torch.bfloat16),
                                      (1, 40, 128, 0, 7, torch.float32),
                                      (1, 33, 64, 40, 0, torch.bfloat16)]:
        Q, K, V = (_normal((BH, T, D), 400 + n, dtype) for n in range(3))
        O, st = emu.attn(Q, K, V, None, False, D ** -0.5, band=(wl, wr))
        tol = 1e-5 if dtype == torch.float32 else 2e-3
        for h in range(BH):
            ref = oracle.window_rows(Q[h], np.arange(T), K[h], V[h], wl, wr)
            _out_close(O.reshape(BH, T, D)[h], ref, tol, False,
                       "window T%d w(%d,%d) head %d" % (T, wl, wr, h), fails)


def check_grouped(emu, fails):
    for (B, H, H_kv, H_idx, head_inner) in [(2, 4, 2, 1, 1), (1, 4, 1, 2, 1), (1, 4, 4, 1, 0)]:
        Tq, Tk, D, k = 21, 60, 64, 9
        Q = _normal((B, H, Tq, D), 500, torch.bfloat16)
        K = _normal((B, H_kv, Tk, D), 501, torch.bfloat16)
        V = _normal((B, H_kv, Tk, D), 502, torch.bfloat16)
        g = np.random.default_rng(H_idx)
        idx = g.integers(0, Tk, size=(B, H_idx, Tq, k)).astype(np.int32)
        O, st = emu.attn(Q.reshape(B * H, Tq, D), K.reshape(B * H_kv, Tk, D),
                         V.reshape(B * H_kv, Tk, D), idx.reshape(-1, k), False, D ** -0.5, H=H,
                         H_kv=H_kv, H_idx=H_idx, grouped=1, head_inner=head_inner)
        O = O.reshape(B, H, Tq, D)
        for b in range(B):
            for h in range(H):
                ref, _ = oracle.attn_rows(Q[b, h], K[b, h // (H // H_kv)], V[b, h // (H // H_kv)],
                                          idx[b, h // (H // H_idx)])
                _out_close(O[b, h], ref, 2e-3, False,
                           "grouped H%d H_kv%d H_idx%d (b %d, h %d)" % (H, H_kv, H_idx, b, h), fails)


def check_smooth(emu, fails):
    g = np.random.default_rng(3)
    rows, k = 50, 6
    score = np.sort(g.integers(-5, 5, size=(rows, k + 1)).astype(np.float32) / 4, axis=1)[:, ::-1]
    score = np.ascontiguousarray(score)
    idx = np.tile(np.arange(k + 1, dtype=np.int32), (rows, 1))
    idx[3, k] = -1
    score[3, k] = -np.inf
    for delta in (0.0, 0.3, 1.0):
        i2, s2 = idx.copy(), score.copy()
        emu.lib.emu_smooth(_p(i2), _p(s2), rows, k, delta)
        ri, rs = oracle.smooth_boundary(idx, score, k, delta)
        if not (np.array_equal(i2, ri) and np.array_equal(s2, rs)):
            fails.append("smoothing delta %g differs" % delta)


def check_random_shapes(emu, n, seed, fails):
    """n seeded random shapes: heads, sequence lengths (ragged, Tq above and
    below Tk), k (1 up to past the valid count), d_proj, head size, dtypes,
    causal or not."""
    g = np.random.default_rng(seed)
    for c in range(n):
        BH = int(g.integers(1, 3))
        Tq, Tk = int(g.integers(1, 90)), int(g.integers(1, 400))
        P = int(g.choice([16, 32, 64, 128]))
        k = int(g.integers(1, min(Tk + 20, 300)))
        causal = bool(g.integers(0, 2))
        dtype = torch.bfloat16 if g.integers(0, 2) else torch.float32
        check_topk(emu, (BH, Tq, Tk, P, k, causal, dtype), fails)
        D = int(g.choice([64, 128]))
        check_attn(emu, (BH, Tq, max(Tk, 2), D, k, dtype, bool(g.integers(0, 2))), fails)


def check_all(path, small=False):
    emu = Emu(path)
    fails = []
    for c in (TOPK_CASES[:2] if small else TOPK_CASES):
        check_topk(emu, c, fails)
    check_topk_ties_and_list(emu, fails)
    for c in (CHUNK_CASES[:1] if small else CHUNK_CASES):
        check_topk_chunks(emu, c, fails)
    for c in (ATTN_CASES[:2] if small else ATTN_CASES):
        check_attn(emu, c, fails)
    check_window(emu, fails)
    check_grouped(emu, fails)
    check_smooth(emu, fails)
    if not small:
        check_random_shapes(emu, 12, 2024, fails)
    return fails


if __name__ == "__main__":
    f = check_all(sys.argv[1], small=len(sys.argv) > 2 and sys.argv[2] == "small")
    print("\n".join(f) if f else "OK")
    sys.exit(1 if f else 0)
