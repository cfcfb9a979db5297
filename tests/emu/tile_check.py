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
  counts. Its output must equal the oracle's top-k bit for bit, however many
  candidates tie at the k-th score. A row whose list count is over its
  capacity must go to the overflow list.
- The full-list rule of the candidate pass, end to end: lists are built the
  way that pass fills them (keys of alternate 128-key tiles, in key order,
  the first cap/2 kept; once a list is full a key scoring exactly at the
  row's bound is dropped and a key above it marks the row as overflowing),
  with the bound from the group maxima; the sort of those lists must give
  the oracle's answer on every unmarked row. This checks the argument that
  makes the drop exact (each dropped key is beaten by the cap/2 >= k earlier
  keys of its list), including equal scores everywhere and ties above the
  16-bit bound.

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
    """Integer q_low/k_low and their fp32 scores (raw dot products and scaled).

    ties: False; True (q_low = 0: every score equal); "few" (one-hot q_low,
    k_low in {0, 1, 2}: three distinct scores, the top one held by about a
    third of the keys); "wide" (a third of the keys score 1001, twelve score
    1002, the rest below 1000: the two top scores share their 16-bit
    truncated order key, so the bound sits below both, and the late 1002 keys
    find the lists full)."""
    g = np.random.default_rng(seed)
    q = g.integers(-4, 5, size=(BH, Tq, P)).astype(np.float64)
    kl = g.integers(-4, 5, size=(BH, Tk, P)).astype(np.float64)
    if ties is True:
        q[:] = 0.0
    elif ties == "few":
        q[:] = 0.0
        q[np.arange(BH)[:, None], np.arange(Tq)[None, :], g.integers(0, P, size=(BH, Tq))] = 1.0
        kl = g.integers(0, 3, size=(BH, Tk, P)).astype(np.float64)
    elif ties == "wide":
        q[:] = 0.0
        q[:, :, 0] = 1.0
        kl[:] = 0.0
        kl[:, :, 0] = np.where(g.random((BH, Tk)) < 0.3, 1001, g.integers(0, 1000, size=(BH, Tk)))
        for bh in range(BH):   # a few keys scoring 1002, most of them late in the row
            kl[bh, g.choice(np.arange(Tk // 4, Tk), size=12, replace=False), 0] = 1002
    raw = np.einsum("hip,hjp->hij", q, kl).astype(np.float32)   # exact integers
    return q, kl, raw


class Emu:
    def __init__(self, path):
        self.lib = lib = ctypes.CDLL(path)
        P, I, F, L = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_int64
        lib.emu_group_select.argtypes = [P, P, I, I, I, I, I]
        lib.emu_cand_sort.argtypes = [P, P, L, I, I, I, I, F, P, P, P, P, P]
        lib.emu_tile_cand_cap.argtypes = [I]
        lib.emu_tile_group_stride.argtypes = [I]


def row_bounds(emu, s, BH, Tq, Tk, k, causal):
    """The group maxima as the group-maximum pass writes them, and each row's
    bound: the k-th largest truncated group maximum (0 for <= k keys)."""
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
    return gm, want


def check_bound(emu, BH, Tq, Tk, k, causal, seed, fails):
    P = 64
    scale = np.float32(0.125)
    _, _, raw = exact_scores(BH, Tq, Tk, P, causal, seed)
    s = raw * scale
    gm, want = row_bounds(emu, s, BH, Tq, Tk, k, causal)
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
    tag = "sort BH%d Tq%d Tk%d k%d causal %d%s" % (BH, Tq, Tk, k, causal, " ties" if ties else "")
    sort_and_compare(emu, q, kl, cand, cnt, expect_ovf, BH, Tq, Tk, k, causal, scale, tag, fails)


def sort_and_compare(emu, q, kl, cand, cnt, expect_ovf, BH, Tq, Tk, k, causal, scale, tag, fails):
    rows = BH * Tq
    idx = np.full((rows, k), -7, np.int32)
    sc = np.full((rows, k), np.nan, np.float32)
    ovf = np.full(rows + 1, -1, np.int64)
    ocount = np.zeros(1, np.int32)
    status = np.zeros(1, np.int32)
    emu.lib.emu_cand_sort(_p(cand), _p(cnt), rows, Tq, Tk, k, int(causal), float(scale), _p(idx),
                          _p(sc), _p(ovf), _p(ocount), _p(status))
    got_ovf = set(ovf[:ocount[0]].tolist())
    if bool(status[0] & 0x4) != bool(got_ovf) or status[0] & ~0x4:
        fails.append("%s: status %#x with %d overflow rows (SSA_DEV_OVERFLOW iff some)" % (
            tag, status[0], len(got_ovf)))
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


def check_full_lists(emu, BH, Tq, Tk, k, causal, seed, fails, ties, want_ovf=None):
    """Lists built by the candidate pass's full-list rule (see the module
    notes); want_ovf: whether some row must be marked (None: either)."""
    P = 64
    scale = np.float32(0.125)
    q, kl, raw = exact_scores(BH, Tq, Tk, P, causal, seed, ties)
    s = raw * scale
    _, tau = row_bounds(emu, s, BH, Tq, Tk, k, causal)
    capc = emu.lib.emu_tile_cand_cap(k) // 2
    rows = BH * Tq
    cand = np.zeros((rows, 2, capc), np.uint64)
    cnt = np.zeros((rows, 2), np.int32)
    marked = set()
    dropped = 0
    for bh in range(BH):
        for i in range(Tq):
            row = bh * Tq + i
            n = valid_count(i, Tq, Tk, causal)
            if n == 0:
                continue
            ok = order_keys(s[bh, i, :n]).astype(np.int64)
            t = int(tau[bh, i])
            js = np.arange(n) if t == 0 else np.nonzero(ok >= t)[0]   # ascending keys
            for lst in (0, 1):
                sel = js[(js // 128) % 2 == lst]
                w = sel[:capc]
                late = sel[capc:]
                bits = raw[bh, i, w].view(np.uint32).astype(np.uint64)
                cand[row, lst, :len(w)] = (bits << np.uint64(32)) | w.astype(np.uint64)
                cnt[row, lst] = len(w)
                if len(late):
                    if (ok[late] > t).any():
                        cnt[row, lst] = capc + 1
                        marked.add(row)
                    dropped += int((ok[late] == t).sum())
    tag = "full lists BH%d Tq%d Tk%d k%d causal %d ties %s" % (BH, Tq, Tk, k, causal, ties)
    if not want_ovf and dropped == 0:
        fails.append("%s: no key was dropped, the case does not exercise the rule" % tag)
    if want_ovf is not None and bool(marked) != want_ovf:
        fails.append("%s: %d marked rows, want %s" % (tag, len(marked), "some" if want_ovf else "none"))
    sort_and_compare(emu, q, kl, cand, cnt, marked, BH, Tq, Tk, k, causal, scale, tag, fails)


FULL_CASES = [
    # BH, Tq, Tk, k, causal, ties, some row marked
    (1, 24, 3000, 150, False, True, False),    # every score equal: the first k keys
    (1, 40, 1400, 50, True, True, False),      # causal, equal scores, rows of every length
    (2, 16, 2500, 200, False, "few", False),   # three distinct scores
    (1, 16, 2000, 40, False, "wide", True),    # ties above the truncated bound: marked rows
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
    # 900 tied candidates for k = 512: the index radix select
    check_sort(emu, 1, 3, 900, 512, False, seed=8, fails=fails, ties=True, margin=2000)
    for c in (FULL_CASES[:1] if small else FULL_CASES):
        check_full_lists(emu, *c[:5], seed=sum(c[:5]), fails=fails, ties=c[5], want_ovf=c[6])
    return fails


if __name__ == "__main__":
    f = check_all(sys.argv[1], small=len(sys.argv) > 2 and sys.argv[2] == "small")
    print("\n".join(f) if f else "OK")
    sys.exit(1 if f else 0)
