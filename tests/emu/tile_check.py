"""The selection stages of the tensor-core top-k under host emulation (CPU).

The score passes themselves run on tcgen05 and have no host stand-in. Their
outputs are built here from exact scores instead, and the two selection
kernels run on them:

- group_select_kernel gets the 16-bit group maxima of every row, laid out
  as the group-maximum pass writes them ([unit][group][256 rows], units of a
  head in reverse query-block order). The key -> group map is re-derived from
  the score kernel's tile order, independently of tile.h, as
  tests/tile_layout_check.cpp does. Its bound must equal the k-th largest
  truncated group maximum of the row, bit for bit (0 for a row with at most
  k keys).
- cand_sort_kernel gets candidate lists as the candidate pass writes them:
  (raw score bits, key) pairs in two lists per row, in any order, with their
  counts. Its output must equal the oracle's top-k bit for bit. A row whose
  list holds more than its capacity, or with more than 256 candidates tied at
  its k-th score, must go to the overflow list.

Scores come from integer q_low, k_low, so every score is exact.
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

UNIT = 256


def build(out_dir: str, asan: bool = False) -> str:
    out = os.path.join(out_dir, "libtile_emu%s.so" % ("_asan" if asan else ""))
    cmd = ["g++", "-O1", "-std=c++17", "-fPIC", "-shared",
           "-I", HERE, "-I", os.path.join(ROOT, "dynamic_top_sparse_rank_b300", "csrc"),
           "-I", os.path.join(ROOT, "include"), os.path.join(HERE, "tile_emu.cpp"), "-o", out]
    if asan:
        cmd[1:1] = ["-g", "-fsanitize=address", "-fno-omit-frame-pointer"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def valid_count(i, Tq, Tk, causal):
    if not causal:
        return Tk
    last = i + (Tk - Tq)
    return 0 if last < 0 else min(last + 1, Tk)


def group_size(n_lo, n_hi, k):
    """Groups of at least min(n, 2k) per row: the power of two <= n_ref / 2k."""
    if n_hi <= k:
        return 0
    q = max(n_lo, k + 1) // (2 * k)
    g = 1
    while g * 2 <= q:
        g *= 2
    return g


def group_of_key(j, g):
    """Key j's group: consecutive keys for g < 32; otherwise the 32-key chunk
    of its 128-key tile, tiles alternating between two accumulators, g/32
    consecutive tiles of one accumulator per group."""
    if g < 32:
        return j // g
    m = g // 32
    t = j // 128
    return (((t // 2) // m) * 2 + t % 2) * 4 + (j % 128) // 32


def order_keys(s):
    u = np.asarray(s, np.float32).copy()
    u[u == 0] = 0.0                                  # fold -0 onto +0
    b = u.view(np.uint32)
    return np.where(b >> 31, ~b, b | np.uint32(0x80000000)).astype(np.uint32)


def exact_scores(BH, Tq, Tk, P, causal, seed, ties=False):
    """Integer q_low/k_low and their fp32 scores (raw dot products and scaled)."""
    g = np.random.default_rng(seed)
    q = g.integers(-4, 5, size=(BH, Tq, P)).astype(np.float64)
    kl = g.integers(-4, 5, size=(BH, Tk, P)).astype(np.float64)
    if ties:
        q[:] = 0.0
    raw = np.einsum("hip,hjp->hij", q, kl).astype(np.float32)   # exact integers
    return q, kl, raw


class Emu:
    def __init__(self, path):
        self.lib = lib = ctypes.CDLL(path)
        P, I, F, L = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_int64
        lib.emu_group_select.argtypes = [P, P, I, I, I, I, I]
        lib.emu_cand_sort.argtypes = [P, P, L, I, I, I, I, F, P, P, P, P]
        lib.emu_tile_cand_cap.argtypes = [I]
        lib.emu_tile_group_stride.argtypes = [I]


def check_bound(emu, BH, Tq, Tk, k, causal, seed, fails):
    P = 64
    scale = np.float32(0.125)
    _, _, raw = exact_scores(BH, Tq, Tk, P, causal, seed)
    s = raw * scale
    uph = (Tq + UNIT - 1) // UNIT
    stride = emu.lib.emu_tile_group_stride(k)
    gm = np.full((BH * uph, stride, UNIT), 0xA5A5, np.uint16)   # garbage where no group is
    want = np.zeros((BH, Tq), np.uint32)
    for bh in range(BH):
        for qb in range(uph):
            u = bh * uph + (uph - 1 - qb)
            i0 = qb * UNIT
            rows = min(UNIT, Tq - i0)
            g = group_size(valid_count(i0, Tq, Tk, causal),
                           valid_count(i0 + rows - 1, Tq, Tk, causal), k)
            for r in range(rows):
                i = i0 + r
                n = valid_count(i, Tq, Tk, causal)
                if n <= k:
                    continue
                grp = np.array([group_of_key(j, g) for j in range(n)])
                key16 = (order_keys(s[bh, i, :n]) >> 16).astype(np.uint32)
                gmax = {}
                for gg, kk in zip(grp, key16):
                    gmax[gg] = max(gmax.get(gg, 0), int(kk))
                assert max(gmax) < stride
                for gg, kk in gmax.items():
                    gm[u, gg, r] = kk
                want[bh, i] = sorted(gmax.values(), reverse=True)[k - 1] << 16
    tau = np.full((BH, Tq), 0xDEADBEEF, np.uint32)
    emu.lib.emu_group_select(_p(gm), _p(tau), BH, Tq, Tk, k, int(causal))
    if not np.array_equal(tau, want):
        bad = np.argwhere(tau != want)[:3].tolist()
        fails.append("bound BH%d Tq%d Tk%d k%d causal %d: rows %s differ" % (BH, Tq, Tk, k,
                                                                              causal, bad))


def check_sort(emu, BH, Tq, Tk, k, causal, seed, fails, margin=20, ties=False, overfill=()):
    """Candidates: each row's valid keys scoring at least its (k + margin)-th
    score, split at random between the two lists and shuffled."""
    P = 64
    scale = np.float32(0.125)
    q, kl, raw = exact_scores(BH, Tq, Tk, P, causal, seed, ties)
    s = raw * scale
    cap = emu.lib.emu_tile_cand_cap(k)
    capc = cap // 2
    rows = BH * Tq
    cand = np.zeros((rows, 2, capc), np.uint64)
    cnt = np.zeros((rows, 2), np.int32)
    g = np.random.default_rng(seed + 1)
    expect_ovf = set()
    for bh in range(BH):
        for i in range(Tq):
            row = bh * Tq + i
            n = valid_count(i, Tq, Tk, causal)
            if n == 0:
                continue
            order = np.sort(s[bh, i, :n])[::-1]
            thr = order[min(n, k + margin) - 1]
            js = np.nonzero(s[bh, i, :n] >= thr)[0]
            g.shuffle(js)
            side = g.integers(0, 2, size=len(js))
            for lst in (0, 1):
                sel = js[side == lst]
                c = len(sel)
                if c > capc:
                    expect_ovf.add(row)
                w = sel[:capc]
                bits = raw[bh, i, w].view(np.uint32).astype(np.uint64)
                cand[row, lst, :len(w)] = (bits << np.uint64(32)) | w.astype(np.uint64)
                cnt[row, lst] = c
            if row in overfill:
                cnt[row, 0] = capc + 1
                expect_ovf.add(row)
            # more than 256 candidates tied at the k_eff-th score, only some of
            # them selected: the tie list overflows
            keff = min(k, n)
            cs = np.sort(s[bh, i, js])[::-1]
            if keff < len(cs):
                T = cs[keff - 1]
                above, inbin = int((cs > T).sum()), int((cs == T).sum())
                if keff - above < inbin and inbin > 256:
                    expect_ovf.add(row)
    idx = np.full((rows, k), -7, np.int32)
    sc = np.full((rows, k), np.nan, np.float32)
    ovf = np.full(rows + 1, -1, np.int64)
    ocount = np.zeros(1, np.int32)
    emu.lib.emu_cand_sort(_p(cand), _p(cnt), rows, Tq, Tk, k, int(causal), float(scale), _p(idx),
                          _p(sc), _p(ovf), _p(ocount))
    got_ovf = set(ovf[:ocount[0]].tolist())
    tag = "sort BH%d Tq%d Tk%d k%d causal %d%s" % (BH, Tq, Tk, k, causal, " ties" if ties else "")
    if got_ovf != expect_ovf:
        fails.append("%s: overflow rows %s, want %s" % (tag, sorted(got_ovf)[:5],
                                                         sorted(expect_ovf)[:5]))
    qt = torch.from_numpy(q)
    kt = torch.from_numpy(kl)
    for bh in range(BH):
        ri, rs = oracle.topk_rows(qt[bh], np.arange(Tq), kt[bh], k, Tq, causal, float(scale))
        for i in range(Tq):
            row = bh * Tq + i
            if row in expect_ovf:
                if not (idx[row] == -7).all():
                    fails.append("%s: overflow row %d was written" % (tag, row))
                continue
            if not (np.array_equal(idx[row], ri[i]) and np.array_equal(sc[row], rs[i])):
                fails.append("%s: row %d differs" % (tag, row))
                return


BOUND_CASES = [
    # BH, Tq, Tk, k, causal
    (1, 20, 131072, 512, True),   # the headline shape's last rows: g = 64 (two tiles a group)
    (1, 300, 300, 16, True),      # g from 1 up; the first rows select everything
    (2, 260, 2000, 8, True),      # Tq < Tk: g >= 32 chunks across tiles
    (1, 100, 700, 40, False),
    (1, 513, 513, 64, True),      # a ragged last unit
]

SORT_CASES = [
    # BH, Tq, Tk, k, causal
    (1, 70, 70, 16, True),
    (2, 40, 500, 33, False),
    (1, 30, 900, 100, True),
    (1, 20, 64, 64, False),       # k = Tk
    (1, 8, 4000, 512, False),     # the headline k: 1024-entry capacity, 16 winners per lane
]


def check_all(path, small=False):
    emu = Emu(path)
    fails = []
    for c in (BOUND_CASES[:2] if small else BOUND_CASES):
        check_bound(emu, *c, seed=sum(c), fails=fails)
    for c in (SORT_CASES[:2] if small else SORT_CASES):
        check_sort(emu, *c, seed=sum(c), fails=fails)
    # a row over its list's capacity; heavy ties at the k-th score
    check_sort(emu, 1, 40, 300, 16, False, seed=5, fails=fails, overfill=(3, 17))
    # all scores equal: 300 candidates (two lists of at most 256) for k = 200
    check_sort(emu, 1, 6, 300, 200, False, seed=6, fails=fails, ties=True, margin=400)
    # 200 tied candidates for k = 150: a partial tie list that fits
    check_sort(emu, 1, 6, 200, 150, False, seed=7, fails=fails, ties=True, margin=400)
    return fails


if __name__ == "__main__":
    f = check_all(sys.argv[1], small=len(sys.argv) > 2 and sys.argv[2] == "small")
    print("\n".join(f) if f else "OK")
    sys.exit(1 if f else 0)
