"""The algorithmic work behind the bench's roofline fractions, against closed
forms (CPU): scored pairs, selected pairs, window band pairs, FLOP and bytes."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from workloads import WORKLOADS  # noqa: E402


def test_causal_pairs_closed_form():
    """Causal with Tq == Tk: row i has i + 1 valid keys, so a head scores
    T(T+1)/2 pairs and selects sum_i min(i + 1, k) = k(k+1)/2 + (T-k)k."""
    w = WORKLOADS["topk_causal_bf16_t128k_k512_planted"]
    T, k, BH = w.Tq, w.k, w.B * w.H
    pairs, sel = bench.valid_pairs(w)
    assert pairs == BH * T * (T + 1) // 2
    assert sel == BH * (k * (k + 1) // 2 + (T - k) * k)


def test_noncausal_and_decode_pairs():
    w = WORKLOADS["decode_bf16_b32_tk64k_k512"]   # one query per head, every key valid
    pairs, sel = bench.valid_pairs(w)
    assert pairs == w.B * w.H * w.Tk and sel == w.B * w.H * w.k
    w = WORKLOADS["topk_f32_t1024_k32"]
    pairs, sel = bench.valid_pairs(w)
    assert pairs == w.B * w.H * w.Tq * w.Tk and sel == w.B * w.H * w.Tq * w.k


def test_window_band_pairs_closed_form():
    """|i - j| <= w clipped to [0, T): interior rows have 2w + 1 keys, the
    first and last w rows lose sum_{d=1..w} d keys each end."""
    w = WORKLOADS["window_bf16_t4096_w128"]
    T, r, BH = w.Tq, w.window, w.B * w.H
    per_head = T * (2 * r + 1) - 2 * (r * (r + 1) // 2)
    assert bench.band_pairs(w) == BH * per_head


def test_algorithmic_flops_and_bytes():
    """Scorer: 2 d_proj FLOP per scored pair (8.796e12 at 128K); gather: one K
    and one V row per selected pair; attention 4 D FLOP per selected pair."""
    w = WORKLOADS["topk_causal_bf16_t128k_k512_planted"]
    alg = bench.algorithmic(w)
    pairs, sel = bench.valid_pairs(w)
    assert alg["score_flops"] == 2.0 * w.P * pairs
    assert abs(alg["score_flops"] - 8.796e12) / 8.796e12 < 1e-3
    assert alg["gather_bytes"] == 2.0 * sel * w.D * 2
    assert alg["attn_flops"] == 4.0 * w.D * sel
    ww = WORKLOADS["window_bf16_t4096_w128"]
    a2 = bench.algorithmic(ww)
    assert a2["window_bytes"] == 2.0 * ww.D * ww.B * ww.H * ww.Tq * 4   # Q, K, V and O once


def test_roofline_fraction_is_work_over_time_over_peak():
    w = WORKLOADS["topk_causal_bf16_t128k_k512_planted"]
    alg = bench.algorithmic(w)
    pk = {"bf16_tflops": 1000.0, "hbm_gbs": 5000.0}
    r = bench.roofline_for("tile_scores.collect", 10.0, w, alg, pk, "test")
    assert r["bound"] == "tensor" and np.isclose(r["achieved"], alg["score_flops"] / 1e-2 / 1e12)
    assert np.isclose(r["frac"], r["achieved"] / 1000.0)
    r = bench.roofline_for("attn_rows.sparse", 10.0, w, alg, pk, "test")
    assert r["bound"] == "hbm" and np.isclose(r["achieved"], alg["gather_bytes"] / 1e-2 / 1e9)


def test_projection_workload_bytes():
    """The projection reads x and W once and writes out: 2 bytes per element."""
    B, H, T, DM, P = bench.PROJ_SHAPE
    rows = B * H * T
    traffic = 2.0 * rows * DM + 2.0 * P * DM + 2.0 * rows * P
    assert abs(traffic - 2.181e9) / 2.181e9 < 1e-3
    assert DM % 64 == 0 and P in (64, 128)


def test_clock_samples_summary():
    """nvidia-smi CSV lines (noheader, nounits) -> median SM clock, max clock,
    the throttle reasons seen active; malformed lines are skipped."""
    lines = [
        "0, 2032, 2032, 812.40, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n",
        "0, 1980, 2032, 1099.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n",
        "0, 2010, 2032, 1050.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n",
        "garbage\n",
        "0, [N/A], 2032, 1.0, 0x0, Not Active, Active, Not Active, Not Active\n",
    ]
    c = bench.parse_clock_samples(lines)
    assert c["samples"] == 3 and c["sm_mhz"] == 2010.0 and c["sm_max_mhz"] == 2032.0
    assert c["reasons"] == ["sw_power_cap"]
    assert bench.parse_clock_samples(["x\n"]) is None
    hot = lines[0].replace("Not Active, Not Active, Not Active, Not Active",
                           "Active, Not Active, Active, Not Active")
    assert bench.parse_clock_samples([hot])["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_gather_aux_bytes():
    """Besides the selected K/V rows the attention reads the index lists
    (int32) and Q and writes O: at 128K 2.15 GB + 2 x 268 MB."""
    w = WORKLOADS["topk_causal_bf16_t128k_k512_planted"]
    alg = bench.algorithmic(w)
    rows = w.B * w.H * w.Tq
    assert alg["gather_aux_bytes"] == rows * w.k * 4 + 2 * rows * w.D * 2
    assert abs(alg["gather_aux_bytes"] - 2.684e9) / 2.684e9 < 1e-3


def test_backward_kernel_bytes():
    """Backward: each side gathers two rows of D elements per selected pair
    (K and V, or Q and dO) plus its per-slot traffic; the scorer sides gather
    one d_proj row per pair."""
    w = WORKLOADS[bench.BACKWARD_BASE]
    _, sel = bench.valid_pairs(w)
    slots = w.B * w.H * w.Tq * w.k
    assert bench.backward_bytes(w, "attn_bwd.query") == sel * 2 * w.D * 2 + slots * 12
    assert bench.backward_bytes(w, "attn_bwd.key") == sel * (2 * w.D * 2 + 12)
    assert bench.backward_bytes(w, "scorer_bwd.key") == sel * (w.P * 2 + 8)
    assert abs(bench.backward_bytes(w, "attn_bwd.query") - 2.808e11) / 2.808e11 < 1e-3
    assert bench.backward_bytes(w, "something else") is None
