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
copies inside the timed region. Under torchrun (N > 1) every rank runs its own
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

from workloads import WORKLOADS, make_attn_inputs, make_scorer_inputs  # noqa: E402

DEFAULT_WORKLOAD = "topk_causal_bf16_t128k_k512_planted"
METRIC = "queries/s and effective TFLOP/s at T=128K, k=512; % of phase roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
L2_FLUSH_BYTES = 512 << 20


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


def algorithmic(w):
    esize = 4 if w.dtype == "f32" else 2
    pairs, sel = valid_pairs(w)
    return {
        "score_flops": 2.0 * w.P * pairs,
        "attn_flops": 4.0 * w.D * sel,
        "gather_bytes": 2.0 * sel * w.D * esize,    # selected K and V rows
        "selected_pairs": sel,
        "scored_pairs": pairs,
    }


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
                "traffic": None, "peak_kind": pk_kind + " bf16 burst (clocks at max during the run)",
                "algorithmic": "2 * d_proj FLOP per valid (query, key) pair, %.4g per launch"
                % alg["score_flops"]}
    if name.startswith("attn_rows"):
        by = alg["gather_bytes"]
        what = "selected K+V rows: k_eff * D * esize * 2 per query row"
    elif name == "cand_sort":
        by = alg["selected_pairs"] * 8 * 1.25 + rows * w.k * 4
        what = "candidate keys read (about 1.25 k_eff x 8 B) + index list written (k x 4 B) per row"
    elif name == "group_select":
        by = rows * 3 * w.k * 2 * 2
        what = "group maxima read twice (about 3k x 2 B per row)"
    else:
        by = alg["scored_pairs"] * 4
        what = "one 32-bit key per valid (query, key) pair"
    achieved = by / sec / 1e9
    return {"kernel": name, "bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"],
            "unit": "GB/s", "frac": achieved / pk["hbm_gbs"], "traffic": None,
            "peak_kind": pk_kind + " HBM copy", "algorithmic": "%s, %.4g B per launch" % (what, by)}


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
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ ours

def run_ours(args, rank, world, local_rank):
    import dynamic_top_sparse_rank_b300 as ssa

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.workload]
    # each rank: its own batch of the workload (independent seed per rank)
    w = w.with_(seed_base=w.seed_base + 1000 * rank)
    q_low, k_low = make_scorer_inputs(w, dev)
    Q, K, V = make_attn_inputs(w, dev)
    torch.cuda.synchronize()
    ws = torch.empty(ssa.score_topk_workspace_size(w.B, w.H, w.Tq, w.Tk, w.P, w.k, w.causal),
                     dtype=torch.uint8, device=dev)
    idx = torch.empty((w.B, w.H, w.Tq, w.k), dtype=torch.int32, device=dev)
    O = torch.empty((w.B, w.H, w.Tq, w.D), dtype=w.torch_dtype, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        ssa.ssa_score_topk(q_low, k_low, w.k, w.causal, workspace=ws, idx=idx)
        ssa.ssa_sparse_attn(Q, K, V, idx, out=O)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # device-resident timing: per step three events on the launching stream
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                          else local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    for s in range(args.steps):
        flush.fill_(s & 0xFF)                       # L2 flush, outside the events
        ev[s][0].record(stream)
        ssa.ssa_score_topk(q_low, k_low, w.k, w.causal, workspace=ws, idx=idx)
        ev[s][1].record(stream)
        ssa.ssa_sparse_attn(Q, K, V, idx, out=O)
        ev[s][2].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    t_score = [ev[s][0].elapsed_time(ev[s][1]) for s in range(args.steps)]
    t_attn = [ev[s][1].elapsed_time(ev[s][2]) for s in range(args.steps)]
    ms_step = float(np.mean([a + b for a, b in zip(t_score, t_attn)]))

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
    host_in = [t.cpu().pin_memory() for t in (q_low, k_low, Q, K, V)]
    host_out = torch.empty(O.shape, dtype=O.dtype, pin_memory=True)
    dev_in = [torch.empty_like(t) for t in (q_low, k_low, Q, K, V)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_out.numel() * host_out.element_size()

    def e2e_step():
        for d, h in zip(dev_in, host_in):
            d.copy_(h, non_blocking=True)
        ssa.ssa_score_topk(dev_in[0], dev_in[1], w.k, w.causal, workspace=ws, idx=idx)
        ssa.ssa_sparse_attn(dev_in[2], dev_in[3], dev_in[4], idx, out=O)
        host_out.copy_(O, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = e0.elapsed_time(e1) / args.steps

    # max over ranks
    t = torch.tensor([ms_step, ms_e2e, float(np.mean(t_score)), float(np.mean(t_attn))],
                     dtype=torch.float64, device=dev)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    ms_step, ms_e2e, ms_score, ms_attn = t.tolist()

    if rank != 0:
        return None
    alg = algorithmic(w)
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
    phases = {
        "score_topk": {"ms": ms_score, "tflops": alg["score_flops"] / (ms_score * 1e-3) / 1e12,
                       "frac_bf16_peak": alg["score_flops"] / (ms_score * 1e-3) / 1e12 / pk["bf16_tflops"]},
        "sparse_attn": {"ms": ms_attn, "gbs": alg["gather_bytes"] / (ms_attn * 1e-3) / 1e9,
                        "frac_hbm": alg["gather_bytes"] / (ms_attn * 1e-3) / 1e9 / pk["hbm_gbs"]},
    }
    line = {
        "metric": METRIC, "value": value, "unit": "queries/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded SplitMix64; integer q_low/k_low in [-4,4] with planted keys, Q/K/V ~ N(0,1))",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "Tq": w.Tq, "Tk": w.Tk, "D": w.D,
                   "d_proj": w.P, "k": w.k, "causal": w.causal,
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
    """The oracle (plain fp64 C, all host cores) on n_rows sampled query rows of
    the workload: score + top-k and attention. Returns (queries/s, cores, sample)."""
    import oracle
    g = np.random.default_rng(seed)
    qi = np.sort(g.choice(w.Tq, size=n_rows, replace=False)).astype(np.int64)
    # head (0, 0) of the workload: the same elements as the one-head workload
    wl = w.with_(B=1, H=1)
    q_low, k_low = make_scorer_inputs(wl)
    Q, K, V = make_attn_inputs(wl)
    cores = oracle.default_threads()
    qd = q_low[0, 0][qi]
    t0 = time.perf_counter()
    idx, _ = oracle.topk_rows(qd, qi, k_low[0, 0], w.k, w.Tq, w.causal, nthreads=cores)
    oracle.attn_rows(Q[0, 0][qi], K[0, 0], V[0, 0], idx, nthreads=cores)
    dt = time.perf_counter() - t0
    return n_rows / dt, cores, ("%d random query rows of head 0 of %s (score + top-k + attention)"
                                % (n_rows, w.name))


def run_reference(args):
    w = WORKLOADS[args.workload]
    vals = []
    cores = 1
    sample = ""
    for s in range(args.warmup + args.steps):
        v, cores, sample = cpu_baseline(w, args.cpu_rows, seed=s)
        if s >= args.warmup:
            vals.append(v)
    value = float(np.mean(vals))
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "queries/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * args.cpu_rows / value, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "queries/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "queries/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-rows", type=int, default=2048,
                    help="query rows the CPU oracle times (bounded sample)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        torch.distributed.init_process_group("nccl")
    line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline:
            v, cores, sample = cpu_baseline(WORKLOADS[args.workload], args.cpu_rows)
            line["cpu_baseline"] = {"value": v, "unit": "queries/s", "cores": cores,
                                    "kind": "oracle", "sample": sample}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
