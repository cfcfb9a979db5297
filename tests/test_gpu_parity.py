"""CUDA path vs the CPU oracle, through the C ABI (needs a B300).

Top-k indices and scores must match the oracle bit for bit (the scorer inputs
are integers in [-4, 4], so every score is exact in fp32). Attention outputs
must be within max-abs 2e-3 for bf16 inputs and 1e-5 for fp32 inputs. Small
cases compare every row; the full-size workloads compare sampled rows against
the oracle and check size-independent invariants on every row.
"""
import numpy as np
import pytest
import torch

import dynamic_top_sparse_rank_b300 as ssa
import oracle
from parity_util import (TOL_BF16, TOL_F32, assert_out_close, check_topk_invariants,
                         sample_rows)
from workloads import WORKLOADS, fill, make_attn_inputs, make_scorer_inputs

pytestmark = pytest.mark.gpu


def _int_inputs(B, H, Tq, Tk, P, dtype, seed):
    q = fill((B, H, Tq, P), "int", seed, 1, dtype, "cpu")
    k = fill((B, H, Tk, P), "int", seed, 2, dtype, "cpu")
    return q, k


def _normal_inputs(B, H, Tq, Tk, D, dtype, seed):
    Q = fill((B, H, Tq, D), "normal", seed, 3, dtype, "cpu")
    K = fill((B, H, Tk, D), "normal", seed, 4, dtype, "cpu")
    V = fill((B, H, Tk, D), "normal", seed, 5, dtype, "cpu")
    return Q, K, V


# ---------------------------------------------------------------- score_topk

TOPK_CASES = [
    # B, H, Tq, Tk, P, k, causal, dtype
    (1, 2, 1024, 1024, 16, 32, False, torch.float32),   # the fp32 T=1024 k=32 workload
    (1, 1, 1, 1, 64, 1, True, torch.bfloat16),
    (1, 1, 7, 7, 64, 4, True, torch.bfloat16),
    (1, 2, 127, 127, 64, 33, True, torch.bfloat16),
    (2, 1, 129, 129, 32, 31, False, torch.bfloat16),
    (1, 1, 1000, 1000, 128, 256, True, torch.bfloat16),
    (1, 1, 300, 1000, 64, 2, True, torch.bfloat16),     # Tq < Tk, bottom-right causal
    (1, 1, 40, 20, 16, 8, True, torch.float32),         # Tq > Tk: empty first rows
    (1, 1, 200, 200, 64, 200, True, torch.bfloat16),    # k = T
    (1, 1, 200, 200, 64, 199, False, torch.bfloat16),   # k = T - 1
    (1, 1, 100, 100, 64, 300, False, torch.bfloat16),   # k > T: padding
    (1, 1, 64, 3000, 64, 2048, False, torch.bfloat16),  # largest k
    (2, 3, 33, 4099, 32, 64, False, torch.float32),
    (1, 1, 16, 65536, 64, 512, False, torch.bfloat16),  # decode-like long rows
]


@pytest.mark.parametrize("B,H,Tq,Tk,P,k,causal,dtype", TOPK_CASES)
def test_score_topk_matches_oracle(cuda_dev, B, H, Tq, Tk, P, k, causal, dtype):
    q, kl = _int_inputs(B, H, Tq, Tk, P, dtype, seed=100 + Tq + k)
    idx, sc = ssa.ssa_score_topk(q.to(cuda_dev), kl.to(cuda_dev), k, causal, with_score=True)
    torch.cuda.synchronize()
    ref_idx, ref_sc = oracle.score_topk(q, kl, k, causal)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    np.testing.assert_array_equal(sc.cpu().numpy(), ref_sc)


def test_score_topk_all_ties(cuda_dev):
    B, H, T, P, k = 1, 2, 700, 64, 100
    q = torch.zeros(B, H, T, P, dtype=torch.bfloat16)
    _, kl = _int_inputs(B, H, T, T, P, torch.bfloat16, 5)
    for causal in (False, True):
        idx = ssa.ssa_score_topk(q.to(cuda_dev), kl.to(cuda_dev), k, causal).cpu().numpy()
        ref, _ = oracle.score_topk(q, kl, k, causal)
        np.testing.assert_array_equal(idx, ref)
        assert (idx[0, 0, T - 1] == np.arange(k)).all()


def test_score_topk_duplicate_boundary_scores(cuda_dev):
    """Many keys share the k-th score: only the lowest indices among them win."""
    B, H, Tq, Tk, P, k = 1, 1, 64, 4096, 16, 50
    q, kl = _int_inputs(B, H, Tq, Tk, P, torch.float32, 6)
    kl = torch.clamp(kl, -1, 1)           # few distinct scores, large tie groups
    idx = ssa.ssa_score_topk(q.to(cuda_dev), kl.to(cuda_dev), k, False).cpu().numpy()
    ref, _ = oracle.score_topk(q, kl, k, False)
    np.testing.assert_array_equal(idx, ref)


def test_score_topk_reuses_workspace_and_outputs(cuda_dev):
    """Two calls in a row on one workspace give the same answer (no stale state)."""
    q, kl = _int_inputs(1, 2, 300, 2000, 64, torch.bfloat16, 7)
    qd, kd = q.to(cuda_dev), kl.to(cuda_dev)
    ws = torch.full((ssa.score_topk_workspace_size(1, 2, 300, 2000, 64, 77, 1),), 0xAB,
                    dtype=torch.uint8, device=cuda_dev)
    a = ssa.ssa_score_topk(qd, kd, 77, True, workspace=ws).clone()
    b = ssa.ssa_score_topk(qd, kd, 77, True, workspace=ws)
    assert torch.equal(a, b)
    ref, _ = oracle.score_topk(q, kl, 77, True)
    np.testing.assert_array_equal(b.cpu().numpy(), ref)


# -------------------------------------------------------------- sparse_attn

def test_sparse_attn_fp32_workload(cuda_dev):
    """The fp32 T=1024 k=32 workload end to end: 1e-5 against the oracle."""
    w = WORKLOADS["topk_f32_t1024_k32"]
    q, kl = make_scorer_inputs(w)
    Q, K, V = make_attn_inputs(w)
    dev = [t.to(cuda_dev) for t in (q, kl, Q, K, V)]
    idx = ssa.ssa_score_topk(dev[0], dev[1], w.k, w.causal)
    O = ssa.ssa_sparse_attn(dev[2], dev[3], dev[4], idx)
    ref_idx, _ = oracle.score_topk(q, kl, w.k, w.causal)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    ref = oracle.sparse_attn(Q, K, V, ref_idx)
    assert O.dtype == torch.float32
    assert_out_close(O.cpu().numpy(), ref, TOL_F32, False)


ATTN_CASES = [
    # B, H, Tq, Tk, D, k, dtype
    (1, 2, 100, 300, 128, 1, torch.bfloat16),
    (1, 2, 100, 300, 128, 7, torch.bfloat16),
    (2, 1, 129, 1000, 128, 33, torch.bfloat16),
    (1, 3, 65, 5000, 64, 256, torch.bfloat16),
    (1, 1, 50, 2000, 128, 512, torch.bfloat16),
    (1, 2, 77, 400, 64, 40, torch.float32),
    (1, 1, 31, 700, 128, 96, torch.float32),
]


@pytest.mark.parametrize("B,H,Tq,Tk,D,k,dtype", ATTN_CASES)
def test_sparse_attn_matches_oracle(cuda_dev, B, H, Tq, Tk, D, k, dtype):
    Q, K, V = _normal_inputs(B, H, Tq, Tk, D, dtype, seed=200 + k)
    g = np.random.default_rng(k)
    idx = g.integers(0, Tk, size=(B, H, Tq, k)).astype(np.int32)   # repeats allowed
    idx[..., -1] = -1 if k > 1 else idx[..., -1]                   # a padding entry
    idx[0, 0, 0, :] = -1                                           # an empty row
    idx_t = torch.from_numpy(idx)
    ref = oracle.sparse_attn(Q, K, V, idx)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    dq, dk, dv, di = (t.to(cuda_dev) for t in (Q, K, V, idx_t))
    O32 = ssa.ssa_sparse_attn(dq, dk, dv, di, out_dtype=torch.float32)
    assert_out_close(O32.cpu().numpy(), ref, tol, False)
    assert (O32[0, 0, 0] == 0).all()
    if dtype == torch.bfloat16:
        Ob = ssa.ssa_sparse_attn(dq, dk, dv, di)
        assert Ob.dtype == torch.bfloat16
        assert_out_close(Ob.float().cpu().numpy(), ref, TOL_BF16, True)


@pytest.mark.parametrize("H,H_kv,H_idx,dtype", [
    (4, 1, 1, torch.bfloat16), (4, 2, 2, torch.bfloat16), (4, 4, 1, torch.bfloat16),
    (4, 2, 1, torch.bfloat16), (4, 1, 4, torch.bfloat16), (4, 4, 4, torch.bfloat16),
    (6, 3, 2, torch.float32),
])
def test_sparse_attn_grouped_heads(cuda_dev, H, H_kv, H_idx, dtype):
    """Shared key/value heads (grouped- and multi-query attention) and shared
    index lists: head h reads K/V head h // (H // H_kv) and index list
    h // (H // H_idx). The reference expands the shared heads and runs the
    plain per-head oracle."""
    B, Tq, Tk, D, k = 2, 150, 500, 128 if dtype == torch.bfloat16 else 64, 48
    Q = fill((B, H, Tq, D), "normal", 300 + H_kv, 3, dtype, "cpu")
    K = fill((B, H_kv, Tk, D), "normal", 300 + H_kv, 4, dtype, "cpu")
    V = fill((B, H_kv, Tk, D), "normal", 300 + H_kv, 5, dtype, "cpu")
    g = np.random.default_rng(H * 100 + H_kv * 10 + H_idx)
    idx = g.integers(0, Tk, size=(B, H_idx, Tq, k)).astype(np.int32)
    idx[..., -1] = -1
    idx_t = torch.from_numpy(idx)
    ref = oracle.sparse_attn(Q, K.repeat_interleave(H // H_kv, dim=1),
                             V.repeat_interleave(H // H_kv, dim=1),
                             idx_t.repeat_interleave(H // H_idx, dim=1).numpy())
    dq, dk, dv, di = (t.to(cuda_dev) for t in (Q, K, V, idx_t))
    O = ssa.ssa_sparse_attn_grouped(dq, dk, dv, di, out_dtype=torch.float32)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    assert_out_close(O.cpu().numpy(), ref, tol, False)
    if H_kv == H and H_idx == H:   # the plain layout: the same arithmetic as ssa_sparse_attn
        assert torch.equal(O, ssa.ssa_sparse_attn(dq, dk, dv, di, out_dtype=torch.float32))


def test_head_shared_scorer_feeds_grouped_attention(cuda_dev):
    """The page's shared-scorer layout: one q_low/k_low per position scored
    once ([B, 1, T, d_proj]), the index list broadcast to 8 query heads that
    read 2 key/value heads."""
    B, H, H_kv, T, P, D, k = 1, 8, 2, 600, 64, 128, 64
    q = fill((B, 1, T, P), "int", 41, 1, torch.bfloat16, "cpu")
    kl = fill((B, 1, T, P), "int", 41, 2, torch.bfloat16, "cpu")
    Q = fill((B, H, T, D), "normal", 41, 3, torch.bfloat16, "cpu")
    K = fill((B, H_kv, T, D), "normal", 41, 4, torch.bfloat16, "cpu")
    V = fill((B, H_kv, T, D), "normal", 41, 5, torch.bfloat16, "cpu")
    idx = ssa.ssa_score_topk(q.to(cuda_dev), kl.to(cuda_dev), k, True)
    ref_idx, _ = oracle.score_topk(q, kl, k, True)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    O = ssa.ssa_sparse_attn_grouped(Q.to(cuda_dev), K.to(cuda_dev), V.to(cuda_dev), idx,
                                    out_dtype=torch.float32)
    ref = oracle.sparse_attn(Q, K.repeat_interleave(H // H_kv, dim=1),
                             V.repeat_interleave(H // H_kv, dim=1),
                             np.repeat(ref_idx, H, axis=1))
    assert_out_close(O.cpu().numpy(), ref, TOL_BF16, False)


def test_sparse_attn_grouped_rejects_bad_groups(cuda_dev):
    Q = torch.zeros((1, 4, 8, 64), dtype=torch.bfloat16, device=cuda_dev)
    K = torch.zeros((1, 3, 8, 64), dtype=torch.bfloat16, device=cuda_dev)
    idx = torch.zeros((1, 1, 8, 4), dtype=torch.int32, device=cuda_dev)
    with pytest.raises(ssa.SSAError):
        ssa.ssa_sparse_attn_grouped(Q, K, K, idx)   # 3 does not divide 4


def test_sparse_attn_k1_is_exact_value_row(cuda_dev):
    Q, K, V = _normal_inputs(1, 2, 64, 500, 128, torch.bfloat16, 9)
    idx = torch.randint(0, 500, (1, 2, 64, 1), dtype=torch.int32, generator=torch.Generator().manual_seed(1))
    O = ssa.ssa_sparse_attn(Q.to(cuda_dev), K.to(cuda_dev), V.to(cuda_dev), idx.to(cuda_dev))
    want = torch.gather(V, 2, idx.long().expand(-1, -1, -1, 128))
    assert torch.equal(O.cpu(), want)


def test_sparse_attn_reports_bad_index(cuda_dev):
    Q, K, V = _normal_inputs(1, 1, 8, 100, 64, torch.bfloat16, 10)
    idx = torch.tensor([[[[3, 5, 100, -7] + [1] * 4] * 8]], dtype=torch.int32)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    O = ssa.ssa_sparse_attn(Q.to(cuda_dev), K.to(cuda_dev), V.to(cuda_dev), idx.to(cuda_dev),
                            out_dtype=torch.float32, dev_status=st)
    assert int(st.item()) & ssa.SSA_DEV_BAD_INDEX
    ref, bad = oracle.attn_rows(Q[0, 0], K[0, 0], V[0, 0], idx[0, 0].numpy())
    assert bad == 16
    assert_out_close(O[0, 0].cpu().numpy(), ref, TOL_BF16, False)


# -------------------------------------------------------------- window_attn

def test_window_workload_full(cuda_dev):
    """The sliding-window workload (B2 H8 T4096 D64, |i-j| <= 128), every row."""
    w = WORKLOADS["window_bf16_t4096_w128"]
    Q, K, V = make_attn_inputs(w)
    dq, dk, dv = (t.to(cuda_dev) for t in (Q, K, V))
    ref = oracle.window_attn(Q, K, V, w.window, w.window)
    O32 = ssa.ssa_window_attn(dq, dk, dv, w.window, out_dtype=torch.float32)
    assert_out_close(O32.cpu().numpy(), ref, TOL_BF16, False)
    Ob = ssa.ssa_window_attn(dq, dk, dv, w.window)
    assert_out_close(Ob.float().cpu().numpy(), ref, TOL_BF16, True)


@pytest.mark.parametrize("T,D,wl,wr,dtype", [
    (1, 64, 0, 0, torch.bfloat16), (130, 64, 0, 0, torch.bfloat16),
    (300, 128, 5, 5, torch.bfloat16), (257, 64, 300, 300, torch.bfloat16),
    (500, 64, 7, 130, torch.bfloat16), (200, 64, 128, 128, torch.float32),
])
def test_window_edges(cuda_dev, T, D, wl, wr, dtype):
    Q, K, V = _normal_inputs(2, 2, T, T, D, dtype, seed=T + wl)
    ref = oracle.window_attn(Q, K, V, wl, wr)
    O = ssa.ssa_window_attn(Q.to(cuda_dev), K.to(cuda_dev), V.to(cuda_dev), wl, wr,
                            out_dtype=torch.float32)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    assert_out_close(O.cpu().numpy(), ref, tol, False)
    if wl == 0 and wr == 0:
        assert torch.equal(O.cpu(), V.float())


@pytest.mark.parametrize("T,wl,wr", [
    (1, 0, 0), (2, 1, 1), (128, 128, 0), (129, 64, 64), (300, 100, 20), (385, 0, 128),
    (1000, 128, 128), (2048, 3, 117),
])
def test_window_tensor_core_tiles(cuda_dev, T, wl, wr):
    """bf16, head size 64 and a band of at most three 128-key tiles per
    128-query tile run as dense tensor-core tiles (the launch is window_tc);
    every row is compared with the oracle."""
    Q, K, V = _normal_inputs(2, 3, T, T, 64, torch.bfloat16, seed=7 * T + wl + 3 * wr)
    ref = oracle.window_attn(Q, K, V, wl, wr)
    dq, dk, dv = (t.to(cuda_dev) for t in (Q, K, V))
    ssa.trace_begin()
    O = ssa.ssa_window_attn(dq, dk, dv, wl, wr, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert [n for n, _ in ssa.trace_end()] == ["window_tc"]
    assert_out_close(O.cpu().numpy(), ref, TOL_BF16, False)
    Ob = ssa.ssa_window_attn(dq, dk, dv, wl, wr)
    assert_out_close(Ob.float().cpu().numpy(), ref, TOL_BF16, True)
    if wl == 0 and wr == 0:
        assert torch.equal(O.cpu(), V.float())


def test_window_wide_band_uses_gather(cuda_dev):
    """A band wider than three key tiles per query tile goes to the gather kernel."""
    T, wl, wr = 1000, 300, 300
    Q, K, V = _normal_inputs(1, 2, T, T, 64, torch.bfloat16, seed=99)
    ref = oracle.window_attn(Q, K, V, wl, wr)
    ssa.trace_begin()
    O = ssa.ssa_window_attn(Q.to(cuda_dev), K.to(cuda_dev), V.to(cuda_dev), wl, wr,
                            out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert [n for n, _ in ssa.trace_end()] == ["attn_rows.window"]
    assert_out_close(O.cpu().numpy(), ref, TOL_BF16, False)


# ------------------------------------------------- full-size sampled parity

FULL = ["topk_causal_bf16_t32k_k256", "topk_causal_bf16_t128k_k512_planted",
        "decode_bf16_b32_tk64k_k512"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload_sampled(cuda_dev, name):
    """Full-size inputs in the benchmark's launch configuration: every row is
    checked for the invariants, sampled rows against the oracle (its own index
    lists feed its attention)."""
    w = WORKLOADS[name]
    q, kl = make_scorer_inputs(w, cuda_dev)
    Q, K, V = make_attn_inputs(w, cuda_dev)
    ws = torch.empty(ssa.score_topk_workspace_size(w.B, w.H, w.Tq, w.Tk, w.P, w.k, w.causal),
                     dtype=torch.uint8, device=cuda_dev)
    idx, sc = ssa.ssa_score_topk(q, kl, w.k, w.causal, with_score=True, workspace=ws)
    O = ssa.ssa_sparse_attn(Q, K, V, idx, out_dtype=torch.float32)
    torch.cuda.synchronize()
    check_topk_invariants(idx, sc, w.Tq, w.Tk, w.k, w.causal)
    rows = sample_rows(w.B, w.H, w.Tq, 48, seed=w.cfg_id)
    flat_idx = idx.view(-1, w.k)[torch.from_numpy(rows).to(cuda_dev)].cpu().numpy()
    flat_sc = sc.view(-1, w.k)[torch.from_numpy(rows).to(cuda_dev)].cpu().numpy()
    gpu_O = O.view(-1, w.D)[torch.from_numpy(rows).to(cuda_dev)].cpu().numpy()
    # oracle, one head at a time (only the sampled heads are copied to the host)
    by_head = {}
    for n, r in enumerate(rows):
        bh, i = divmod(int(r), w.Tq)
        by_head.setdefault(bh, []).append((n, i))
    for bh, items in by_head.items():
        b, h = divmod(bh, w.H)
        ns = [n for n, _ in items]
        qi = np.array([i for _, i in items], dtype=np.int64)
        ref_idx, ref_sc = oracle.topk_rows(q[b, h].cpu()[qi], qi, kl[b, h].cpu(), w.k, w.Tq,
                                           w.causal)
        np.testing.assert_array_equal(flat_idx[ns], ref_idx)
        np.testing.assert_array_equal(flat_sc[ns], ref_sc)
        ref_O, bad = oracle.attn_rows(Q[b, h].cpu()[qi], K[b, h].cpu(), V[b, h].cpu(), ref_idx)
        assert bad == 0
        assert_out_close(gpu_O[ns], ref_O, TOL_BF16, False)
