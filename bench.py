#!/usr/bin/env python
"""Throughput of the dynamic top-k sparse attention forward on one B300.

A step is one pass of the whole path over one batch of synthetic input:
ssa_score_topk (low-rank scorer + exact top-k) followed by ssa_sparse_attn
(gather attention over the selected keys), on the causal 128K-token workload
(B1 H8 T131072, head_dim 128, d_proj 64, k 512, bf16, planted keys).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0). ``value`` is queries/s (query rows B*H*Tq per
second over the whole job) with inputs resident in HBM; ``e2e`` is the same
metric through the public calls with pinned host buffers, the host<->device
copies inside the timed region (the copies of Q, K and V, which only the
attention call reads, run on a second stream while the scorer computes; with
B = 1 the step runs in groups of heads (four, or two) so that copies of one
group overlap the other groups' kernels; the scorer's inputs are copied a step
ahead into a second buffer set, and a step's other input copies overlap the
previous step's last output copy). Under torchrun (N > 1) every rank runs its own
independent batch (weak scaling, no collective on the data path); the timed
region is bracketed by barriers and the slowest rank's time is used.

``--impl reference`` times the CPU oracle (plain fp64 C) on a bounded sample
of the same workload on this host's cores; it is a deliberately slow program,
not a target.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from workloads import (WORKLOADS, fill, make_attn_inputs, make_grad_output,  # noqa: E402
                       make_scorer_inputs)

DEFAULT_WORKLOAD = "topk_causal_bf16_t128k_k512_planted"
METRIC = "queries/s and effective TFLOP/s at T=128K, k=512; % of phase roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
L2_FLUSH_BYTES = 512 << 20
# A device-side wait queued after the L2 flush and before the first event of a
# timed step: the GPU stays busy while Python enqueues the step, so the events
# measure the step's device time and not the host's call overhead (which
# matters only for sub-millisecond steps such as the window workload).
HOST_COVER_CYCLES = 2_000_000


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ counts

def valid_pairs(w):
    """Sum over query rows of |valid(i)| (scorer work) and of k_eff(i)."""
    i = np.arange(w.Tq, dtype=np.int64)
    nv = np.clip(i + (w.Tk - w.Tq) + 1, 0, w.Tk) if w.causal else np.full(w.Tq, w.Tk, np.int64)
    keff = np.minimum(nv, w.k)
    bh = w.B * w.H
    return int(nv.sum()) * bh, int(keff.sum()) * bh


def band_pairs(w):
    """(query, key) pairs of the sliding window |i - j| <= w, clipped at both ends."""
    i = np.arange(w.Tq, dtype=np.int64)
    lo = np.maximum(0, i - w.window)
    hi = np.minimum(w.Tk - 1, i + w.window)
    return int((hi - lo + 1).sum()) * w.B * w.H


def algorithmic(w):
    esize = 4 if w.dtype == "f32" else 2
    if w.P == 0:   # the sliding-window workload: no scorer
        sel = band_pairs(w)
        return {"score_flops": 0.0, "attn_flops": 4.0 * w.D * sel,
                "gather_bytes": 2.0 * sel * w.D * esize, "selected_pairs": sel,
                "scored_pairs": 0,
                "window_bytes": float(esize * w.D * w.B * w.H * (w.Tq * 2 + w.Tk * 2))}
    pairs, sel = valid_pairs(w)
    rows = w.B * w.H * w.Tq
    return {
        "score_flops": 2.0 * w.P * pairs,
        "attn_flops": 4.0 * w.D * sel,
        "gather_bytes": 2.0 * sel * w.D * esize,    # selected K and V rows
        # the attention's other traffic: the index lists (int32), Q read and O
        # written once (in the input dtype)
        "gather_aux_bytes": float(rows * w.k * 4 + 2 * rows * w.D * esize),
        "selected_pairs": sel,
        "scored_pairs": pairs,
    }


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the
# score passes, from one-launch ncu captures on the 32K workload; to be
# re-measured, or dropped, when the kernels change. Their traffic is the group
# maxima and candidate lists they write, which grow with rows x k, so the
# 128K figures are the 32K ones scaled by that ratio (4), not captured at 128K.
MEASURED_TRAFFIC = {
    ("topk_causal_bf16_t32k_k256", "tile_scores.groupmax"): 0.897e9,
    ("topk_causal_bf16_t32k_k256", "tile_scores.collect"): 1.860e9,
    ("topk_causal_bf16_t128k_k512_planted", "tile_scores.groupmax"): 4 * 0.897e9,
    ("topk_causal_bf16_t128k_k512_planted", "tile_scores.collect"): 4 * 1.860e9,
    ("window_bf16_t4096_w128", "window_tc"): 25.22e6,   # Q, K, V read once; O stays in L2
}

# Read throughput of the L2 slices (GB/s) that serve the gather: the kernel's
# lts__t_sectors_srcunit_tex_op_read bytes divided by its duration and by the
# fraction of peak ncu reports for that counter, on the 32K workload (66.2 GB
# in 3.774 ms at 75.5% of peak). The gather's K/V rows come from L2 (97% hits),
# so this, not the HBM copy rate, is the ceiling it runs against.
L2_SLICE_READ_GBS = 23.2e3


def roofline_for(name, ms, w, alg, pk, pk_kind):
    """Roofline of one kernel launch: algorithmic work per launch / its time.

    Scorer passes (tensor cores): 2 * d_proj FLOP per valid (query, key) pair.
    Gather attention: the selected K and V rows (k_eff * D * esize * 2 bytes per
    query row); they stream from L2 when a head's K/V fits there, so the
    fraction of the HBM copy peak can exceed 1. Selection and sort kernels: the
    bytes they must read and write.
    """
    rows = w.B * w.H * w.Tq
    sec = ms * 1e-3
    if name.startswith("tile_scores"):
        achieved = alg["score_flops"] / sec / 1e12
        return {"kernel": name, "bound": "tensor", "achieved": achieved,
                "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"],
                "traffic": MEASURED_TRAFFIC.get((w.name, name)),
                "peak_kind": pk_kind + " bf16 burst (clocks at max during the run)",
                "algorithmic": "2 * d_proj FLOP per valid (query, key) pair, %.4g per launch"
                % alg["score_flops"]}
    if name in ("attn_rows.window", "window_tc"):
        by = alg["window_bytes"]
        what = "unique Q, K, V and O bytes of the window workload"
    elif name.startswith("attn_rows"):
        by = alg["gather_bytes"]
        what = "selected K+V rows: k_eff * D * esize * 2 per query row"
    elif name == "cand_sort":
        by = alg["selected_pairs"] * 8 * 1.25 + rows * w.k * 4
        what = "candidate keys read (about 1.25 k_eff x 8 B) + index list written (k x 4 B) per row"
    elif name == "group_select":
        by = rows * 3 * w.k * 2 * 2
        what = "group maxima read twice (about 3k x 2 B per row)"
    elif name == "topk_merge":
        kcap = min(w.k, 8192)
        nch = (w.Tk + 8191) // 8192
        by = rows * nch * kcap * 8 + rows * w.k * 4
        what = "the key chunks' selections read (8 B each) + index list written (k x 4 B) per row"
    else:   # the row-wise top-k: every valid key's k_low row, once per query row
        by = alg["scored_pairs"] * w.P * (4 if w.dtype == "f32" else 2)
        what = "k_low rows scored: d_proj * esize per valid (query, key) pair"
    achieved = by / sec / 1e9
    line = {"kernel": name, "bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"],
            "unit": "GB/s", "frac": achieved / pk["hbm_gbs"], "traffic": MEASURED_TRAFFIC.get((w.name, name)),
            "peak_kind": pk_kind + " HBM copy", "algorithmic": "%s, %.4g B per launch" % (what, by)}
    if name == "attn_rows.sparse":
        line["l2"] = {"achieved": achieved, "peak": L2_SLICE_READ_GBS, "unit": "GB/s",
                      "frac": achieved / L2_SLICE_READ_GBS,
                      "peak_kind": "L2 slice read throughput derived from ncu (the gather is L2-served)"}
    return line


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        with open(self.path) as f:
            lines = f.readlines()
        os.unlink(self.path)
        return parse_clock_samples(lines)


THROTTLE_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


def parse_clock_samples(lines):
    """Summary of `nvidia-smi --query-gpu=<ClockSampler.Q> --format=csv,noheader,nounits`
    lines: median SM clock, the largest max clock, and every throttle reason
    seen "Active" in any sample (None without a parsable sample)."""
    sm, mx, reasons = [], 0.0, set()
    for line in lines:
        f = [x.strip() for x in line.split(",")]
        if len(f) < 9:
            continue
        try:
            sm.append(float(f[1]))
            mx = max(mx, float(f[2]))
        except ValueError:
            continue
        for n, v in zip(THROTTLE_REASONS, f[5:9]):
            if v.lower().startswith("active"):
                reasons.add(n)
    if not sm:
        return None
    return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
            "samples": len(sm)}


# ------------------------------------------------------------------ ranks

def rank_workload(w, rank: int):
    """The batch rank `rank` processes: the same workload with its own seed
    (weak scaling: independent batches, no data exchanged between ranks)."""
    return w.with_(seed_base=w.seed_base + 1000 * rank)


def max_over_ranks(vals, world: int, device):
    """Element-wise maximum of `vals` over all ranks (the slowest rank's times)."""
    t = torch.tensor(list(vals), dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


# ------------------------------------------------------------------ ours

# The 128K workload in the pages' shared-scorer layout (mhpq.cn/news/1098205,
# section 3.2): one q_low/k_low per position, scored once, its index list
# broadcast to the 8 query heads, which read 2 key/value heads (grouped-query
# attention). Its inputs are those of the 128K workload's first head (scorer)
# and first two heads (K, V).
SHARED_WORKLOAD = "topk_causal_bf16_t128k_k512_shared_scorer_kv2"
SHARED_BASE, SHARED_KV = "topk_causal_bf16_t128k_k512_planted", 2
# The 128K workload with the boundary smoothing of mhpq.cn/news/1098205,
# section 4.2: k = 511 (the k + 1 selection stays on the tensor-core path),
# threshold 0.5 on the scaled scores (q_low . k_low / 8: integer dot products
# within 4 of each other); the index lists have k + 1 = 512 slots.
SMOOTH_WORKLOAD = "topk_causal_bf16_t128k_k511_smooth_delta0.5"
SMOOTH_K, SMOOTH_DELTA = 511, 0.5


def run_ours(args, rank, world, local_rank):
    import dynamic_top_sparse_rank_b300 as ssa

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    shared = args.workload == SHARED_WORKLOAD
    smooth = args.workload == SMOOTH_WORKLOAD
    w = WORKLOADS[SHARED_BASE if (shared or smooth) else args.workload]
    if smooth:
        w = w.with_(k=SMOOTH_K)
    w = rank_workload(w, rank)   # each rank: its own batch of the workload
    window = w.P == 0
    if shared:
        Q = make_attn_inputs(w, dev)[0]
        _, K, V = make_attn_inputs(w.with_(H=SHARED_KV), dev)
        torch.cuda.empty_cache()
        ws_sc = w.with_(H=1)   # the scorer runs once per position
    else:
        Q, K, V = make_attn_inputs(w, dev)
        ws_sc = w
    if window:
        q_low = k_low = ws = idx = None
    else:
        q_low, k_low = make_scorer_inputs(ws_sc, dev)
        wsize = (ssa.score_topk_smooth_workspace_size if smooth else ssa.score_topk_workspace_size)
        ws = torch.empty(wsize(ws_sc.B, ws_sc.H, w.Tq, w.Tk, w.P, w.k, w.causal),
                         dtype=torch.uint8, device=dev)
        idx = torch.empty((w.B, ws_sc.H, w.Tq, w.k + (1 if smooth else 0)), dtype=torch.int32,
                          device=dev)
    if smooth:
        topk = lambda ql, kl, ix=idx: ssa.ssa_score_topk_smooth(   # noqa: E731
            ql, kl, w.k, w.causal, SMOOTH_DELTA, workspace=ws, idx=ix)
    else:
        topk = lambda ql, kl, ix=idx: ssa.ssa_score_topk(   # noqa: E731
            ql, kl, w.k, w.causal, workspace=ws, idx=ix)
    attn = ssa.ssa_sparse_attn_grouped if shared else ssa.ssa_sparse_attn
    torch.cuda.synchronize()
    O = torch.empty((w.B, w.H, w.Tq, w.D), dtype=w.torch_dtype, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    # the phases of one step: (name, call)
    if window:
        phase_list = [("window_attn", lambda: ssa.ssa_window_attn(Q, K, V, w.window, out=O))]
    else:
        phase_list = [("score_topk", lambda: topk(q_low, k_low)),
                      ("sparse_attn", lambda: attn(Q, K, V, idx, out=O))]

    def step():
        for _, fn in phase_list:
            fn()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # device-resident timing: per step one event before and after each phase,
    # on the launching stream
    nph = len(phase_list)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nph + 1)] for _ in range(args.steps)]
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                          else local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    for s in range(args.steps):
        flush.fill_(s & 0xFF)                       # L2 flush, outside the events
        torch.cuda._sleep(HOST_COVER_CYCLES)        # host call overhead stays outside the events
        ev[s][0].record(stream)
        for ph, (_, fn) in enumerate(phase_list):
            fn()
            ev[s][ph + 1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    t_phase = [[ev[s][ph].elapsed_time(ev[s][ph + 1]) for s in range(args.steps)]
               for ph in range(nph)]
    ms_step = float(np.mean([sum(t_phase[ph][s] for ph in range(nph)) for s in range(args.steps)]))

    # per-kernel times: the same steps again with the library's launch tracing
    # (CUDA events recorded on the launching stream around every kernel)
    ssa.trace_begin()
    for s in range(args.steps):
        flush.fill_(s & 0xFF)
        step()
    recs = ssa.trace_end()
    torch.cuda.synchronize()
    launches = len(recs) // args.steps
    per_kernel = {}
    for name, ms in recs:
        per_kernel.setdefault(name, []).append(ms)
    kernels = {n: {"launches_per_step": len(v) // args.steps, "ms": float(np.sum(v)) / args.steps}
               for n, v in per_kernel.items()}

    # end to end through the public calls: pinned host in, O back to host
    dev_src = [Q, K, V] if window else [q_low, k_low, Q, K, V]
    host_in = [t.cpu().pin_memory() for t in dev_src]
    host_out = torch.empty(O.shape, dtype=O.dtype, pin_memory=True)
    dev_in = [torch.empty_like(t) for t in dev_src]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_out.numel() * host_out.element_size()

    copy_stream = torch.cuda.Stream(dev)
    d2h_stream = torch.cuda.Stream(dev)
    # one batch of heads split in groups of contiguous heads (four when each
    # keeps at least four heads, else two: a scorer call over fewer heads
    # loses more to its tail than the finer overlap gains): a group's inputs
    # arrive while the groups before it compute and its output returns while
    # the groups after it run.
    # Consecutive steps overlap too: a step's input copies start once the
    # previous step's last attention is done (the buffers are free), while
    # that step's last output copy is still running; a group's attention waits
    # only for the previous step's read of the same output slice.
    split = not window and not shared and w.B == 1 and w.H >= 2
    ngroups = 4 if w.H % 4 == 0 and w.H // 4 >= 4 else 2
    groups = [(g * w.H // ngroups, (g + 1) * w.H // ngroups) for g in range(ngroups)]
    # q_low and k_low in two buffer sets: a step prefetches the next step's
    # into the other set while it computes (the last timed step does not, so
    # every copy in the timed region is a timed step's)
    qk_sets = [dev_in[:2], [torch.empty_like(t) for t in dev_in[:2]]] if split else None
    prev = {"done": None, "read": [None] * ngroups, "topk_done": None, "qk_ready": None, "n": 0}

    def copy_qk(n, after):
        """q_low, k_low of step n into buffer set n % 2, group by group."""
        evs = []
        with torch.cuda.stream(copy_stream):
            if after is not None:
                copy_stream.wait_event(after)
            for h0, h1 in groups:
                for d, h in zip(qk_sets[n % 2], host_in[:2]):
                    d[:, h0:h1].copy_(h[:, h0:h1], non_blocking=True)
                evs.append(torch.cuda.Event())
                evs[-1].record(copy_stream)
        return evs

    def e2e_step_split(prefetch_next):
        n = prev["n"]
        ev_qk = prev["qk_ready"] or copy_qk(n, prev["done"])
        ev_in = []
        with torch.cuda.stream(copy_stream):
            if prev["done"] is not None:
                copy_stream.wait_event(prev["done"])   # its compute is done with Q, K, V
            for h0, h1 in groups:
                for d, h in zip(dev_in[2:], host_in[2:]):
                    d[:, h0:h1].copy_(h[:, h0:h1], non_blocking=True)
                ev_in.append(torch.cuda.Event())
                ev_in[-1].record(copy_stream)
        qk = qk_sets[n % 2]
        for g, (h0, h1) in enumerate(groups):
            stream.wait_event(ev_qk[g])
            topk(qk[0][:, h0:h1], qk[1][:, h0:h1], idx[:, h0:h1])
        topk_done = torch.cuda.Event()
        topk_done.record(stream)
        # the next step's q_low, k_low into the set the previous step's scorer read
        prev["qk_ready"] = copy_qk(n + 1, prev["topk_done"]) if prefetch_next else None
        prev["topk_done"] = topk_done
        for g, (h0, h1) in enumerate(groups):
            stream.wait_event(ev_in[g])
            if prev["read"][g] is not None:
                stream.wait_event(prev["read"][g])   # the previous step has read this slice
            attn(dev_in[2][:, h0:h1], dev_in[3][:, h0:h1], dev_in[4][:, h0:h1], idx[:, h0:h1],
                 out=O[:, h0:h1])
            ev_o = torch.cuda.Event()
            ev_o.record(stream)
            d2h_stream.wait_event(ev_o)
            with torch.cuda.stream(d2h_stream):
                host_out[:, h0:h1].copy_(O[:, h0:h1], non_blocking=True)
                prev["read"][g] = torch.cuda.Event()
                prev["read"][g].record(d2h_stream)
        prev["done"] = torch.cuda.Event()
        prev["done"].record(stream)
        prev["n"] = n + 1

    def e2e_step(prefetch_next=False):
        if split:
            e2e_step_split(prefetch_next)
            return
        if window:
            for d, h in zip(dev_in, host_in):
                d.copy_(h, non_blocking=True)
            ssa.ssa_window_attn(dev_in[0], dev_in[1], dev_in[2], w.window, out=O)
        else:
            # q_low and k_low on the launching stream; Q, K and V, which only
            # the attention call reads, on a copy stream while the scorer runs
            dev_in[0].copy_(host_in[0], non_blocking=True)
            dev_in[1].copy_(host_in[1], non_blocking=True)
            copy_stream.wait_stream(stream)   # the previous step's attention is done with them
            with torch.cuda.stream(copy_stream):
                for d, h in zip(dev_in[2:], host_in[2:]):
                    d.copy_(h, non_blocking=True)
            topk(dev_in[0], dev_in[1])
            stream.wait_stream(copy_stream)
            attn(dev_in[2], dev_in[3], dev_in[4], idx, out=O)
        host_out.copy_(O, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    stream.wait_stream(d2h_stream)
    e0.record(stream)
    prev["done"] = e0   # the first timed step's copies start after the start event
    for st in range(args.steps):
        e2e_step(prefetch_next=st + 1 < args.steps)
    stream.wait_stream(d2h_stream)   # the last step's result is read back
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = e0.elapsed_time(e1) / args.steps

    # max over ranks
    vals = max_over_ranks([ms_step, ms_e2e] + [float(np.mean(tp)) for tp in t_phase], world, dev)
    ms_step, ms_e2e, ms_phase = vals[0], vals[1], vals[2:]

    if rank != 0:
        return None
    alg = algorithmic(w)
    if smooth:   # the gather runs over k + 1 slots per row
        alg_g = algorithmic(w.with_(k=w.k + 1))
        alg["gather_bytes"], alg["attn_flops"] = alg_g["gather_bytes"], alg_g["attn_flops"]
        alg["gather_aux_bytes"] = alg_g["gather_aux_bytes"]
    if shared:   # one scorer for all heads
        alg["score_flops"] /= w.H
        alg["scored_pairs"] //= w.H
    pk, pk_kind = peaks()
    nq = w.n_queries * world
    value = nq / (ms_step * 1e-3)
    eff_tflops = world * (alg["score_flops"] + alg["attn_flops"]) / (ms_step * 1e-3) / 1e12

    # roofline of the dominant kernel (largest time per step)
    dom = max(kernels, key=lambda n: kernels[n]["ms"])
    dom_ms = kernels[dom]["ms"] / max(1, kernels[dom]["launches_per_step"])   # per launch
    roof = roofline_for(dom, dom_ms, w, alg, pk, pk_kind)
    for n, kinfo in kernels.items():
        if kinfo["ms"] < 0.01 * ms_step:   # e.g. the overflow pass with nothing to redo
            continue
        r = roofline_for(n, kinfo["ms"] / max(1, kinfo["launches_per_step"]), w, alg, pk, pk_kind)
        kinfo.update({"bound": r["bound"], "achieved": r["achieved"], "unit": r["unit"],
                      "frac": r["frac"]})
    phases = {}
    for (name, _), ms in zip(phase_list, ms_phase):
        ph = {"ms": ms}
        if name == "score_topk":
            ph["tflops"] = alg["score_flops"] / (ms * 1e-3) / 1e12
            ph["frac_bf16_peak"] = ph["tflops"] / pk["bf16_tflops"]
        elif name == "sparse_attn":
            ph["gbs"] = alg["gather_bytes"] / (ms * 1e-3) / 1e9
            ph["frac_hbm"] = ph["gbs"] / pk["hbm_gbs"]
            ph["frac_l2"] = ph["gbs"] / L2_SLICE_READ_GBS   # the ceiling of an L2-served gather
            ph["aux_bytes"] = alg.get("gather_aux_bytes")   # idx, Q and O, beside the gather
        else:
            ph["gbs"] = alg["window_bytes"] / (ms * 1e-3) / 1e9
            ph["frac_hbm"] = ph["gbs"] / pk["hbm_gbs"]
        phases[name] = ph
    line = {
        "metric": METRIC, "value": value, "unit": "queries/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded SplitMix64; integer q_low/k_low in [-4,4] with planted keys, Q/K/V ~ N(0,1))",
        "config": {"workload": (SHARED_WORKLOAD if shared else SMOOTH_WORKLOAD if smooth
                                else w.name), "B": w.B, "H": w.H,
                   "scorer_heads": ws_sc.H, "kv_heads": SHARED_KV if shared else w.H,
                   "Tq": w.Tq, "Tk": w.Tk, "D": w.D,
                   "d_proj": w.P, "k": w.k, "causal": w.causal, "window": w.window,
                   "boundary_delta": SMOOTH_DELTA if smooth else None,
                   "l2": "flushed between timed steps (512 MB write) and inputs > L2",
                   "parallelism": "replicas" if world == 1 else "dp%d (independent batches)" % world},
        "effective_tflops": eff_tflops,
        "tokens_per_s": w.B * w.Tq * world / (ms_step * 1e-3),
        "phases": phases,
        "kernels": kernels,
        "roofline": roof,
        "e2e": {"value": nq / (ms_e2e * 1e-3), "unit": "queries/s", "ms_per_step": ms_e2e,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches * args.steps,
        "clocks": clk,
    }
    return line


# ------------------------------------------------------------ CPU oracle

def cpu_baseline(w, n_rows: int, seed: int = 0):
    """The oracle (plain fp64 C, all host cores) on a bounded sample of the
    workload's query rows, the whole path for each (score + top-k + attention,
    or window attention). Returns (queries/s, cores, sample description)."""
    import oracle
    g = np.random.default_rng(seed)
    cores = oracle.default_threads()
    if w.P == 0:   # sliding window: rows of head (0, 0)
        n = min(n_rows, w.Tq)
        qi = np.sort(g.choice(w.Tq, size=n, replace=False)).astype(np.int64)
        Q, K, V = make_attn_inputs(w.with_(B=1, H=1))
        t0 = time.perf_counter()
        oracle.window_rows(Q[0, 0][qi], qi, K[0, 0], V[0, 0], w.window, w.window, nthreads=cores)
        dt = time.perf_counter() - t0
        return n / dt, cores, "%d random query rows of head 0 of %s (window attention)" % (n, w.name), n
    if w.Tq >= n_rows:   # long sequences: random rows of head (0, 0)
        qi = np.sort(g.choice(w.Tq, size=n_rows, replace=False)).astype(np.int64)
        wl = w.with_(B=1, H=1)   # the same elements as head (0, 0) of the workload
        q_low, k_low = make_scorer_inputs(wl)
        Q, K, V = make_attn_inputs(wl)
        t0 = time.perf_counter()
        idx, _ = oracle.topk_rows(q_low[0, 0][qi], qi, k_low[0, 0], w.k, w.Tq, w.causal,
                                  nthreads=cores)
        oracle.attn_rows(Q[0, 0][qi], K[0, 0], V[0, 0], idx, nthreads=cores)
        dt = time.perf_counter() - t0
        return n_rows / dt, cores, ("%d random query rows of head 0 of %s (score + top-k + "
                                    "attention)" % (n_rows, w.name)), n_rows
    # few query rows per head (decode): every row of the first heads
    heads = max(1, min(16, n_rows // max(1, w.Tq)))
    wl = w.with_(B=1, H=heads)
    q_low, k_low = make_scorer_inputs(wl)
    Q, K, V = make_attn_inputs(wl)
    t0 = time.perf_counter()
    idx, _ = oracle.score_topk(q_low, k_low, w.k, w.causal, nthreads=cores)
    oracle.sparse_attn(Q, K, V, idx, nthreads=cores)
    dt = time.perf_counter() - t0
    n = heads * w.Tq
    return n / dt, cores, ("all %d query rows of the first %d heads of %s (score + top-k + "
                           "attention)" % (n, heads, w.name)), n


def run_reference(args):
    w = WORKLOADS[SHARED_BASE if args.workload in (SHARED_WORKLOAD, SMOOTH_WORKLOAD)
                  else args.workload]
    vals = []
    cores, sample, n = 1, "", 1
    for s in range(args.warmup + args.steps):
        v, cores, sample, n = cpu_baseline(w, args.cpu_rows, seed=s)
        if s >= args.warmup:
            vals.append(v)
    value = float(np.mean(vals))
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "queries/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * n / value, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "queries/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "queries/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_reference_backward(args):
    """The reference arm of the backward workload: the oracle's backward on a
    bounded sample per step (see cpu_baseline_backward)."""
    vals, cores, sample, n = [], 1, "", 256
    for s in range(args.warmup + args.steps):
        v, cores, sample = cpu_baseline_backward(n, seed=s)
        if s >= args.warmup:
            vals.append(v)
    value = float(np.mean(vals))
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "queries/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * n / value, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": BACKWARD_WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "queries/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "queries/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------ projection

# The scorer's projections q_low = q_proj(query), k_low = k_proj(key) at the
# 32K shape of the pages' scorer: 8 heads x 32768 rows, d_model 4096 -> d_proj
# 64 (x is 2.1 GB, above L2). One step = one call (the query side).
PROJECT_WORKLOAD = "project_bf16_h8_t32k_d4096_p64"
PROJ_SHAPE = (1, 8, 32768, 4096, 64)   # B, H, T, d_model, d_proj


def run_project(args, rank, world, local_rank):
    import dynamic_top_sparse_rank_b300 as ssa

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    B, H, T, DM, P = PROJ_SHAPE
    rows = B * H * T
    x = fill((B, H, T, DM), "normal", 1234 + 1000 * rank, 31, torch.bfloat16, dev)
    W = fill((P, DM), "normal", 1234, 32, torch.bfloat16, dev)
    out = torch.empty((B, H, T, P), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    step = lambda: ssa.ssa_lowrank_project(x, W, out=out)   # noqa: E731
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                          else local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    for s_ in range(args.steps):
        flush.fill_(s_ & 0xFF)
        torch.cuda._sleep(HOST_COVER_CYCLES)
        ev[s_][0].record(stream)
        step()
        ev[s_][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    ssa.trace_begin()
    for s_ in range(args.steps):
        flush.fill_(s_ & 0xFF)
        step()
    recs = ssa.trace_end()
    torch.cuda.synchronize()
    k_ms = float(np.mean([t for n, t in recs if n == "lowrank_project"]))
    # end to end: x from pinned host memory, out back to the host
    hx = x.cpu().pin_memory()
    hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    dx = torch.empty_like(x)

    def e2e_step():
        dx.copy_(hx, non_blocking=True)
        ssa.ssa_lowrank_project(dx, W, out=out)
        hout.copy_(out, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = e0.elapsed_time(e1) / args.steps
    ms, ms_e2e, k_ms = max_over_ranks([ms, ms_e2e, k_ms], world, dev)
    if rank != 0:
        return None
    pk, pk_kind = peaks()
    traffic = 2.0 * rows * DM + 2.0 * P * DM + 2.0 * rows * P   # x, W, out
    achieved = traffic / (k_ms * 1e-3) / 1e9
    flops = 2.0 * rows * DM * P
    return {
        "metric": METRIC, "value": rows * world / (ms * 1e-3), "unit": "queries/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded SplitMix64; x, W ~ N(0,1))",
        "config": {"workload": PROJECT_WORKLOAD, "B": B, "H": H, "T": T, "d_model": DM,
                   "d_proj": P, "l2": "flushed between timed steps (512 MB write) and inputs > L2",
                   "parallelism": "replicas"},
        "effective_tflops": flops / (ms * 1e-3) / 1e12,
        "kernels": {"lowrank_project": {"launches_per_step": 1, "ms": k_ms, "bound": "hbm",
                                        "achieved": achieved, "unit": "GB/s",
                                        "frac": achieved / pk["hbm_gbs"]}},
        "roofline": {"kernel": "lowrank_project", "bound": "hbm", "achieved": achieved,
                     "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
                     "traffic": None, "peak_kind": pk_kind + " HBM copy",
                     "algorithmic": "x, W and out bytes, %.4g per launch (%.4g FLOP)" % (traffic, flops)},
        "e2e": {"value": rows * world / (ms_e2e * 1e-3), "unit": "queries/s", "ms_per_step": ms_e2e,
                "h2d_bytes_per_step": hx.numel() * 2, "d2h_bytes_per_step": hout.numel() * 2},
        "gpu_launches": 1,
        "clocks": clk,
    }


def cpu_baseline_project(n_rows: int = 256):
    """The oracle's projection of a bounded sample of rows of the projection
    workload on this host's cores; rows per second."""
    import oracle
    B, H, T, DM, P = PROJ_SHAPE
    x = fill((n_rows, DM), "normal", 1234, 31, torch.bfloat16, "cpu")
    W = fill((P, DM), "normal", 1234, 32, torch.bfloat16, "cpu")
    cores = oracle.default_threads()
    t0 = time.perf_counter()
    oracle.lowrank_project(x, W, nthreads=cores)
    dt = time.perf_counter() - t0
    return n_rows / dt, cores, "%d rows of %s" % (n_rows, PROJECT_WORKLOAD)


# ------------------------------------------------------------ backward

# The backward of the 128K workload under the straight-through estimator
# (mhpq.cn/news/1098205, section 2.3). The forward's index lists (the exact
# top-k, computed once before timing) and an incoming gradient dO ~ N(0,1)
# are given. One step = ssa_sparse_attn_bwd (dQ, dK, dV and the pair
# gradients dS) + ssa_scorer_bwd (dq_low, dk_low).
BACKWARD_WORKLOAD = "backward_topk_causal_bf16_t128k_k512"
BACKWARD_BASE = "topk_causal_bf16_t128k_k512_planted"


def backward_bytes(w, name):
    """Algorithmic bytes of one launch of a backward kernel: its row gathers
    per selected pair (K and V, or Q and dO: 2 D elements; k_low or q_low: P
    elements), plus what it reads and writes per pair slot (dS, p, pair ids,
    index lists)."""
    esize = 4 if w.dtype == "f32" else 2
    _, sel = valid_pairs(w)
    slots = w.B * w.H * w.Tq * w.k
    return {
        "attn_bwd.query": sel * 2 * w.D * esize + slots * (4 + 8),   # idx in; dS, p out
        "attn_bwd.key": sel * (2 * w.D * esize + 12),                # Q, dO; dS, p, pair id
        "scorer_bwd.query": sel * w.P * esize + slots * 8,           # k_low; idx, dS
        "scorer_bwd.key": sel * (w.P * esize + 8),                   # q_low; dS, pair id
        "pair_lists.count": slots * 4,
        "pair_lists.fill": slots * 4 + sel * 4,
        "pair_lists.scan": w.B * w.H * w.Tk * 12,
    }.get(name)


def run_backward(args, rank, world, local_rank):
    import dynamic_top_sparse_rank_b300 as ssa

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = rank_workload(WORKLOADS[BACKWARD_BASE], rank)
    q_low, k_low = make_scorer_inputs(w, dev)
    Q, K, V = make_attn_inputs(w, dev)
    dO = make_grad_output(w, dev)
    idx = ssa.ssa_score_topk(q_low, k_low, w.k, w.causal)
    ws = torch.empty(ssa.sparse_attn_scorer_bwd_workspace_size(w.B, w.H, w.Tq, w.Tk, w.k),
                     dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(q_, k_, Q_, K_, V_, dO_, idx_):
        # the attention's and the scorer's gradients in one call: the
        # key-major lists both key sides walk are built once
        dQ, dK, dV, dS, dq, dk = ssa.ssa_sparse_attn_scorer_bwd(Q_, K_, V_, dO_, q_, k_, idx_,
                                                               workspace=ws)
        return dQ, dK, dV, dq, dk

    args_dev = (q_low, k_low, Q, K, V, dO, idx)
    for _ in range(args.warmup):
        step(*args_dev)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                          else local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    for s_ in range(args.steps):
        flush.fill_(s_ & 0xFF)
        torch.cuda._sleep(HOST_COVER_CYCLES)
        ev[s_][0].record(stream)
        step(*args_dev)
        ev[s_][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    ssa.trace_begin()
    for s_ in range(args.steps):
        flush.fill_(s_ & 0xFF)
        step(*args_dev)
    recs = ssa.trace_end()
    torch.cuda.synchronize()
    per_kernel = {}
    for name, t in recs:
        per_kernel.setdefault(name, []).append(t)
    kernels = {n: {"launches_per_step": len(v) // args.steps, "ms": float(np.sum(v)) / args.steps}
               for n, v in per_kernel.items()}
    launches = len(recs) // args.steps
    # end to end: every input from pinned host memory, every gradient back.
    # The heads run in two groups, each group's gradients read back while the
    # next computes; the inputs sit in two buffer sets, each step copying the
    # next step's into the other set while it computes (the last timed step
    # copies nothing ahead, so every copy in the timed region is a timed
    # step's).
    hin = [t.cpu().pin_memory() for t in args_dev]
    dsets = [[torch.empty_like(t) for t in args_dev] for _ in range(2)]
    outs = step(*args_dev)
    hout = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
    copy_stream, d2h_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    halves = [(0, w.H // 2), (w.H // 2, w.H)] if w.H >= 2 else [(0, w.H)]
    prev = {"n": 0, "ready": None, "done": [None, None], "read": [None] * len(halves)}

    def copy_in(n, after):
        evs = []
        with torch.cuda.stream(copy_stream):
            if after is not None:
                copy_stream.wait_event(after)
            for h0, h1 in halves:
                for d, h in zip(dsets[n % 2], hin):
                    d[:, h0:h1].copy_(h[:, h0:h1], non_blocking=True)
                evs.append(torch.cuda.Event())
                evs[-1].record(copy_stream)
        return evs

    def e2e_step(prefetch_next=False):
        n = prev["n"]
        ev_in = prev["ready"] or copy_in(n, prev["done"][(n + 1) % 2])
        din = dsets[n % 2]
        for g, (h0, h1) in enumerate(halves):
            stream.wait_event(ev_in[g])
            if prev["read"][g] is not None:
                stream.wait_event(prev["read"][g])
            res = step(*[t[:, h0:h1] for t in din])
            ev_o = torch.cuda.Event()
            ev_o.record(stream)
            d2h_stream.wait_event(ev_o)
            with torch.cuda.stream(d2h_stream):
                for h, o in zip(hout, res):
                    o.record_stream(d2h_stream)   # freed only after the copy has read it
                    h[:, h0:h1].copy_(o, non_blocking=True)
                prev["read"][g] = torch.cuda.Event()
                prev["read"][g].record(d2h_stream)
        done = torch.cuda.Event()
        done.record(stream)
        # the next step's inputs into the set the previous step read
        prev["ready"] = copy_in(n + 1, prev["done"][(n + 1) % 2]) if prefetch_next else None
        prev["done"][n % 2] = done
        prev["n"] = n + 1

    e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream.wait_stream(d2h_stream)
    e0.record(stream)
    prev["done"] = [e0, e0]   # the first timed step's copies start after the start event
    for st in range(args.steps):
        e2e_step(prefetch_next=st + 1 < args.steps)
    stream.wait_stream(d2h_stream)   # the last step's gradients are read back
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = e0.elapsed_time(e1) / args.steps
    ms, ms_e2e = max_over_ranks([ms, ms_e2e], world, dev)
    if rank != 0:
        return None
    pk, pk_kind = peaks()
    for n, kinfo in kernels.items():
        b = backward_bytes(w, n)
        if b is not None and kinfo["ms"] > 0:
            kinfo.update({"bound": "hbm", "unit": "GB/s",
                          "achieved": b / (kinfo["ms"] * 1e-3) / 1e9})
            kinfo["frac"] = kinfo["achieved"] / pk["hbm_gbs"]
    dom = max(kernels, key=lambda n: kernels[n]["ms"])
    dk_ = kernels[dom]
    nq = w.n_queries * world
    return {
        "metric": METRIC, "value": nq / (ms * 1e-3), "unit": "queries/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded SplitMix64; integer q_low/k_low with planted keys, "
                "Q/K/V/dO ~ N(0,1))",
        "config": {"workload": BACKWARD_WORKLOAD, "B": w.B, "H": w.H, "Tq": w.Tq, "Tk": w.Tk,
                   "D": w.D, "d_proj": w.P, "k": w.k, "causal": w.causal,
                   "l2": "flushed between timed steps (512 MB write) and inputs > L2",
                   "parallelism": "replicas" if world == 1 else "dp%d (independent batches)" % world},
        "kernels": kernels,
        "roofline": {"kernel": dom, "bound": "hbm", "achieved": dk_.get("achieved"),
                     "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": dk_.get("frac"),
                     "traffic": None, "peak_kind": pk_kind + " HBM copy",
                     "algorithmic": "row gathers and per-slot traffic of the kernel, %.4g bytes"
                                    % (backward_bytes(w, dom) or 0.0)},
        "e2e": {"value": nq / (ms_e2e * 1e-3), "unit": "queries/s", "ms_per_step": ms_e2e,
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in hin),
                "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in hout)},
        "gpu_launches": launches * args.steps,
        "clocks": clk,
    }


def cpu_baseline_backward(n_rows: int = 256, seed: int = 0):
    """The oracle's backward (attention + scorer) on a bounded sample of query
    rows of head 0 of the backward workload; rows per second. The sample's
    index lists come from the oracle's top-k, outside the timed part."""
    import oracle
    w = WORKLOADS[BACKWARD_BASE].with_(B=1, H=1)
    g = np.random.default_rng(seed)
    qi = np.sort(g.choice(w.Tq, size=n_rows, replace=False)).astype(np.int64)
    q_low, k_low = make_scorer_inputs(w)
    Q, K, V = make_attn_inputs(w)
    dO = make_grad_output(w)
    cores = oracle.default_threads()
    idx, _ = oracle.topk_rows(q_low[0, 0][qi], qi, k_low[0, 0], w.k, w.Tq, w.causal,
                              nthreads=cores)
    t0 = time.perf_counter()
    _, _, _, dS, _ = oracle.attn_bwd_rows(Q[0, 0][qi], K[0, 0], V[0, 0], idx, dO[0, 0][qi],
                                          nthreads=cores)
    oracle.scorer_bwd_rows(q_low[0, 0][qi], k_low[0, 0], idx, dS)
    dt = time.perf_counter() - t0
    return n_rows / dt, cores, ("%d random query rows of head 0 of %s (attention and scorer "
                                "backward)" % (n_rows, BACKWARD_WORKLOAD))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(WORKLOADS) + [PROJECT_WORKLOAD, SHARED_WORKLOAD,
                                                 SMOOTH_WORKLOAD, BACKWARD_WORKLOAD])
    ap.add_argument("--cpu-rows", type=int, default=2048,
                    help="query rows the CPU oracle times (bounded sample)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.workload == PROJECT_WORKLOAD:
        if args.impl == "reference":
            if rank == 0:
                v, cores, sample = cpu_baseline_project()
                print(json.dumps({"impl": "reference", "metric": METRIC, "value": v,
                                  "unit": "queries/s", "n_gpus": args.gpus, "steps": 1,
                                  "warmup": args.warmup, "ms_per_step": 1e3 * 256 / v,
                                  "higher_is_better": True, "scaling": "weak",
                                  "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                                  "config": {"workload": PROJECT_WORKLOAD, "sample": sample},
                                  "cpu_baseline": {"value": v, "unit": "queries/s", "cores": cores,
                                                   "kind": "oracle", "sample": sample},
                                  "e2e": {"value": v, "unit": "queries/s", "h2d_bytes_per_step": 0,
                                          "d2h_bytes_per_step": 0}}), flush=True)
            return
        if world > 1:
            torch.distributed.init_process_group("nccl")
        line = run_project(args, rank, world, local_rank)
        if rank == 0:
            if not args.no_cpu_baseline:
                v, cores, sample = cpu_baseline_project()
                line["cpu_baseline"] = {"value": v, "unit": "queries/s", "cores": cores,
                                        "kind": "oracle", "sample": sample}
            print(json.dumps(line), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    if args.workload == BACKWARD_WORKLOAD:
        if args.impl == "reference":
            if rank == 0:
                print(json.dumps(run_reference_backward(args)), flush=True)
            return
        if world > 1:
            torch.distributed.init_process_group("nccl")
        line = run_backward(args, rank, world, local_rank)
        if rank == 0:
            if not args.no_cpu_baseline:
                v, cores, sample = cpu_baseline_backward()
                line["cpu_baseline"] = {"value": v, "unit": "queries/s", "cores": cores,
                                        "kind": "oracle", "sample": sample}
            print(json.dumps(line), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        torch.distributed.init_process_group("nccl")
    line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline:
            base = (SHARED_BASE if args.workload in (SHARED_WORKLOAD, SMOOTH_WORKLOAD)
                    else args.workload)
            v, cores, sample, _ = cpu_baseline(WORKLOADS[base], args.cpu_rows)
            line["cpu_baseline"] = {"value": v, "unit": "queries/s", "cores": cores,
                                    "kind": "oracle", "sample": sample}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
