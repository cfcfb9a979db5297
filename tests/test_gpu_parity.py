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


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("T,wl,wr", [
    (1, 0, 0), (2, 1, 1), (128, 128, 0), (129, 64, 64), (300, 100, 20), (385, 0, 128),
    (1000, 128, 128), (2048, 3, 117),
])
def test_window_tensor_core_tiles(cuda_dev, T, wl, wr, D):
    """bf16, head size 64 or 128 and a band of at most three 128-key tiles per
    128-query tile run as dense tensor-core tiles (the launch is window_tc);
    every row is compared with the oracle."""
    Q, K, V = _normal_inputs(2, 3, T, T, D, torch.bfloat16, seed=7 * T + wl + 3 * wr + D)
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


@pytest.mark.parametrize("D", [64, 128])
def test_window_tensor_core_many_items_per_cta(cuda_dev, D):
    """More 128-query items than SMs (80 heads x 8 tiles): each persistent CTA
    takes several items in turn, through both shared-memory stages (D 64) or
    its one stage (D 128) and the TMEM hand-offs between items; every row
    against the oracle, fp32 and bf16 output."""
    T, wl, wr = 1024, 128, 128
    Q, K, V = _normal_inputs(2, 40, T, T, D, torch.bfloat16, seed=500 + D)
    ref = oracle.window_attn(Q, K, V, wl, wr)
    dq, dk, dv = (t.to(cuda_dev) for t in (Q, K, V))
    st = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    ssa.trace_begin()
    O = ssa.ssa_window_attn(dq, dk, dv, wl, wr, out_dtype=torch.float32, dev_status=st)
    torch.cuda.synchronize()
    assert [n for n, _ in ssa.trace_end()] == ["window_tc"]
    assert int(st.item()) == 0
    assert_out_close(O.cpu().numpy(), ref, TOL_BF16, False)
    Ob = ssa.ssa_window_attn(dq, dk, dv, wl, wr)
    assert_out_close(Ob.float().cpu().numpy(), ref, TOL_BF16, True)


@pytest.mark.parametrize("D", [64, 128])
def test_window_tensor_core_rescales(cuda_dev, D):
    """Scores that grow along the key axis (q . k_j = c j, c such that the
    weights grow by about 2^10 per 64 keys), so a row's maximum moves by more
    than 2^8 in weight from one 64-key step of the band to the next: the running shift moves at almost every step and O, summed
    at the old shift, is scaled each time (after the previous step's P V has
    finished). A scale applied to a partial O, or not at all, would be off by
    about the step's weight ratio; every row against the oracle."""
    B, H, T, wl, wr = 1, 4, 600, 128, 128
    g = torch.Generator().manual_seed(900 + D)
    sign = torch.randint(0, 2, (D,), generator=g).float() * 2 - 1          # v0: entries +-1
    j = torch.arange(T, dtype=torch.float32)
    Q = sign.expand(B, H, T, D).clone()
    c = 10.0 * D ** 0.5 / (64 * 1.4427)                                     # log2 weight +10 per 64 keys
    K = (c * j / D)[None, None, :, None] * sign                              # q . k_j = c j
    K = K + 0.01 * torch.randn(B, H, T, D, generator=g)
    V = torch.randn(B, H, T, D, generator=g)
    Q, K, V = (t.to(torch.bfloat16) for t in (Q, K.expand(B, H, T, D), V))
    ref = oracle.window_attn(Q, K, V, wl, wr)
    dq, dk, dv = (t.to(cuda_dev) for t in (Q, K, V))
    ssa.trace_begin()
    O = ssa.ssa_window_attn(dq, dk, dv, wl, wr, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert [n for n, _ in ssa.trace_end()] == ["window_tc"]
    assert_out_close(O.cpu().numpy(), ref, TOL_BF16, False)
    Ob = ssa.ssa_window_attn(dq, dk, dv, wl, wr)
    assert_out_close(Ob.float().cpu().numpy(), ref, TOL_BF16, True)


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


# ------------------------------------------------- full-size parity

UNIT_ROWS = 256   # query rows per work unit of the tensor-core top-k


def unit_rows(B, H, Tq, seed):
    """Flat row ids: one row of every 256-row work unit of every head (its
    first, its last or a random row, in turn), every row of one pair of units
    that share a work item (unit qb of head 0 and unit units-1-qb), and the
    sequence ends and tile edges of sample_rows."""
    g = np.random.default_rng(seed)
    units = (Tq + UNIT_ROWS - 1) // UNIT_ROWS
    rows = set(int(r) for r in sample_rows(B, H, Tq, 0, seed=seed))
    for bh in range(B * H):
        for u in range(units):
            n = min(UNIT_ROWS, Tq - UNIT_ROWS * u)
            off = (0, n - 1, int(g.integers(0, n)))[(bh + u) % 3]
            rows.add(bh * Tq + UNIT_ROWS * u + off)
    qb = units // 3
    for u in {qb, units - 1 - qb}:
        for i in range(UNIT_ROWS * u, min(Tq, UNIT_ROWS * (u + 1))):
            rows.add(i)
    return np.array(sorted(rows), dtype=np.int64)


def _by_head(rows, Tq):
    out = {}
    for n, r in enumerate(rows):
        bh, i = divmod(int(r), Tq)
        out.setdefault(bh, []).append((n, i))
    return out


def _oracle_compare(w, q, kl, Q, K, V, rows, idx, sc, O32, O16, attn_heads=None):
    """The oracle on the given flat rows, one head at a time (only those heads
    are copied to the host): top-k bit for bit, attention (from the oracle's
    own index lists) within the tolerance in fp32 and in bf16 output."""
    dev = idx.device
    rt = torch.from_numpy(rows).to(dev)
    flat_idx = idx.view(-1, w.k)[rt].cpu().numpy()
    flat_sc = sc.view(-1, w.k)[rt].cpu().numpy()
    o32 = O32.view(-1, w.D)[rt].cpu().numpy()
    o16 = O16.view(-1, w.D)[rt].float().cpu().numpy()
    heads = _by_head(rows, w.Tq)
    import concurrent.futures as cf

    def one(bh):
        items = heads[bh]
        b, h = divmod(bh, w.H)
        ns = [n for n, _ in items]
        qi = np.array([i for _, i in items], dtype=np.int64)
        threads = 1 if len(qi) < 64 else None
        ref_idx, ref_sc = oracle.topk_rows(q[b, h].cpu()[qi], qi, kl[b, h].cpu(), w.k, w.Tq,
                                           w.causal, nthreads=threads)
        np.testing.assert_array_equal(flat_idx[ns], ref_idx)
        np.testing.assert_array_equal(flat_sc[ns], ref_sc)
        if attn_heads is not None and bh not in attn_heads:
            return len(ns)
        ref_O, bad = oracle.attn_rows(Q[b, h].cpu()[qi], K[b, h].cpu(), V[b, h].cpu(), ref_idx,
                                      nthreads=threads)
        assert bad == 0
        assert_out_close(o32[ns], ref_O, TOL_BF16, False)
        assert_out_close(o16[ns], ref_O, TOL_BF16, True)
        return len(ns)

    workers = 16 if len(heads) > 64 else 1
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        checked = sum(ex.map(one, sorted(heads)))
    assert checked == len(rows)


def _run_full(w, dev):
    q, kl = make_scorer_inputs(w, dev)
    Q, K, V = make_attn_inputs(w, dev)
    ws = torch.empty(ssa.score_topk_workspace_size(w.B, w.H, w.Tq, w.Tk, w.P, w.k, w.causal),
                     dtype=torch.uint8, device=dev)
    idx, sc = ssa.ssa_score_topk(q, kl, w.k, w.causal, with_score=True, workspace=ws)
    O16 = ssa.ssa_sparse_attn(Q, K, V, idx)                           # as the bench runs it
    O32 = ssa.ssa_sparse_attn(Q, K, V, idx, out_dtype=torch.float32)
    torch.cuda.synchronize()
    del ws
    return q, kl, Q, K, V, idx, sc, O32, O16


@pytest.mark.parametrize("name", ["topk_causal_bf16_t32k_k256",
                                  "topk_causal_bf16_t128k_k512_planted"])
def test_full_size_workload_every_unit(cuda_dev, name):
    """Full-size inputs in the benchmark's launch configuration: every row is
    checked for the invariants; one row of every 256-row work unit of every
    head, and every row of one paired work item, against the oracle (top-k
    bit for bit, attention in fp32 and bf16 output)."""
    w = WORKLOADS[name]
    q, kl, Q, K, V, idx, sc, O32, O16 = _run_full(w, cuda_dev)
    check_topk_invariants(idx, sc, w.Tq, w.Tk, w.k, w.causal)
    rows = unit_rows(w.B, w.H, w.Tq, seed=w.cfg_id)
    assert len(rows) >= w.B * w.H * ((w.Tq + UNIT_ROWS - 1) // UNIT_ROWS)
    _oracle_compare(w, q, kl, Q, K, V, rows, idx, sc, O32, O16)


def test_full_size_decode_every_row(cuda_dev):
    """The decode workload (B32 H32, one query against 65536 keys per head):
    all 1024 rows' top-k against the oracle bit for bit; attention against
    the oracle on 64 heads (their K and V are copied to the host)."""
    w = WORKLOADS["decode_bf16_b32_tk64k_k512"]
    q, kl, Q, K, V, idx, sc, O32, O16 = _run_full(w, cuda_dev)
    check_topk_invariants(idx, sc, w.Tq, w.Tk, w.k, w.causal)
    rows = np.arange(w.B * w.H * w.Tq, dtype=np.int64)
    g = np.random.default_rng(w.cfg_id)
    attn_heads = set(int(x) for x in g.choice(w.B * w.H, 64, replace=False)) | {0, w.B * w.H - 1}
    _oracle_compare(w, q, kl, Q, K, V, rows, idx, sc, O32, O16, attn_heads=attn_heads)


def test_full_size_equal_scores_every_row(cuda_dev):
    """The 128K workload with q_low = 0 (every score ties): every row of every
    head must select its first k_eff valid keys with score 0, -1 / -inf past
    them (the lower index wins ties)."""
    w = WORKLOADS["topk_causal_bf16_t128k_k512_equal_scores"]
    q, kl = make_scorer_inputs(w, cuda_dev)
    assert not q.any()
    idx, sc = ssa.ssa_score_topk(q, kl, w.k, w.causal, with_score=True)
    torch.cuda.synchronize()
    i = torch.arange(w.Tq, device=cuda_dev).view(-1, 1)
    j = torch.arange(w.k, device=cuda_dev).view(1, -1)
    valid = j <= i + (w.Tk - w.Tq)
    want_idx = torch.where(valid, j, torch.full_like(j, -1)).to(torch.int32)
    want_sc = torch.where(valid, torch.zeros((), device=cuda_dev),
                          torch.full((), -float("inf"), device=cuda_dev))
    assert torch.equal(idx, want_idx.expand_as(idx))
    assert torch.equal(sc, want_sc.expand_as(sc))


@pytest.mark.parametrize("name", ["topk_causal_bf16_t32k_k256",
                                  "topk_causal_bf16_t128k_k512_planted"])
def test_full_size_tile_path_matches_rowwise_every_row(cuda_dev, name):
    """Every row of the full-size workload: the tensor-core top-k (bf16
    inputs) against the row-wise kernel, which an fp32 input selects. The
    inputs are integers, so both compute the same exact scores; the two
    selections share no code beyond the output format, and the row-wise
    kernel is itself checked against the oracle above."""
    w = WORKLOADS[name]
    q, kl = make_scorer_inputs(w, cuda_dev)
    idx, sc = ssa.ssa_score_topk(q, kl, w.k, w.causal, with_score=True)
    torch.cuda.synchronize()
    q32, kl32 = q.float(), kl.float()
    del q, kl
    ssa.trace_begin()
    idx_r, sc_r = ssa.ssa_score_topk(q32, kl32, w.k, w.causal, with_score=True)
    torch.cuda.synchronize()
    assert {n for n, _ in ssa.trace_end()} == {"topk_rows"}
    assert torch.equal(idx, idx_r)
    assert torch.equal(sc, sc_r)
