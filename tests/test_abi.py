"""The C ABI library: it loads, exports what include/ssa.h declares, and
rejects bad arguments on the host without launching anything (CPU only)."""
import ctypes
import os
import re

import pytest

import dynamic_top_sparse_rank_b300 as ssa
from dynamic_top_sparse_rank_b300 import _native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"^\s*(?:const\s+)?[\w\*\s]+?\b(ssa_\w+)\s*\(", src, re.M))
    return names


def test_library_exports_every_declared_symbol():
    lib = ssa.load()
    names = _declared()
    assert {"ssa_score_topk", "ssa_sparse_attn", "ssa_window_attn"} <= names
    for n in names:
        assert hasattr(lib, n), n
        ctypes.cast(getattr(lib, n), ctypes.c_void_p)
    assert set(_native.EXPORTS) <= names


def test_version_and_status_strings():
    lib = ssa.load()
    assert lib.ssa_version() >= 1
    for s in range(6):
        assert b"unknown" not in lib.ssa_status_string(s)
    assert b"unknown" in lib.ssa_status_string(99)


def test_workspace_size_rules():
    f = ssa.score_topk_workspace_size
    assert f(1, 8, 131072, 131072, 64, 512, 1) > 0
    assert f(1, 1, 16, 16, 48, 4, 0) == 0          # unsupported P
    assert f(1, 1, 16, 16, 64, 4096, 0) == 0       # k too large
    assert f(1, 1, 16, 16, 64, 0, 0) == 0          # k < 1
    assert f(0, 1, 16, 16, 64, 4, 0) > 0           # empty problem: a token size


V = ctypes.c_void_p


def test_host_validation_without_gpu():
    lib = ssa.load()
    ok_ptr = V(4096)           # aligned, never dereferenced: validation fails first
    bad_ptr = V(4100)
    # score_topk: null idx, unsupported P, k too large, misaligned input, workspace too small
    assert lib.ssa_score_topk(ok_ptr, ok_ptr, 1, 1, 1, 8, 8, 64, 4, 0, 0.0, None, None, ok_ptr,
                              1 << 20, None, None) == _native.SSA_ERR_INVALID
    assert lib.ssa_score_topk(ok_ptr, ok_ptr, 1, 1, 1, 8, 8, 48, 4, 0, 0.0, ok_ptr, None, ok_ptr,
                              1 << 20, None, None) == _native.SSA_ERR_UNSUPPORTED
    assert lib.ssa_score_topk(ok_ptr, ok_ptr, 1, 1, 1, 8, 8, 64, 4096, 0, 0.0, ok_ptr, None,
                              ok_ptr, 1 << 20, None, None) == _native.SSA_ERR_UNSUPPORTED
    assert lib.ssa_score_topk(bad_ptr, ok_ptr, 1, 1, 1, 8, 8, 64, 4, 0, 0.0, ok_ptr, None, ok_ptr,
                              1 << 20, None, None) == _native.SSA_ERR_INVALID
    assert lib.ssa_score_topk(ok_ptr, ok_ptr, 1, 1, 1, 8, 8, 64, 4, 0, 0.0, ok_ptr, None, ok_ptr,
                              16, None, None) == _native.SSA_ERR_WORKSPACE
    assert lib.ssa_score_topk(ok_ptr, ok_ptr, 7, 1, 1, 8, 8, 64, 4, 0, 0.0, ok_ptr, None, ok_ptr,
                              1 << 20, None, None) == _native.SSA_ERR_INVALID
    # empty problem: nothing to do, nothing launched
    assert lib.ssa_score_topk(None, None, 1, 0, 1, 8, 8, 64, 4, 0, 0.0, None, None, None, 0,
                              None, None) == _native.SSA_OK
    # sparse_attn: unsupported D, null idx, misaligned O, bad out dtype
    assert lib.ssa_sparse_attn(ok_ptr, ok_ptr, ok_ptr, 1, 1, 1, 8, 8, 96, ok_ptr, 4, 0.0, ok_ptr,
                               1, None, None) == _native.SSA_ERR_UNSUPPORTED
    assert lib.ssa_sparse_attn(ok_ptr, ok_ptr, ok_ptr, 1, 1, 1, 8, 8, 64, None, 4, 0.0, ok_ptr,
                               1, None, None) == _native.SSA_ERR_INVALID
    assert lib.ssa_sparse_attn(ok_ptr, ok_ptr, ok_ptr, 1, 1, 1, 8, 8, 64, ok_ptr, 4, 0.0, bad_ptr,
                               1, None, None) == _native.SSA_ERR_INVALID
    assert lib.ssa_sparse_attn(ok_ptr, ok_ptr, ok_ptr, 1, 1, 1, 8, 8, 64, ok_ptr, 4, 0.0, ok_ptr,
                               5, None, None) == _native.SSA_ERR_INVALID
    # window_attn: negative radius, unsupported D
    assert lib.ssa_window_attn(ok_ptr, ok_ptr, ok_ptr, 1, 1, 1, 8, 64, -1, 2, 0.0, ok_ptr, 1,
                               None, None) == _native.SSA_ERR_INVALID
    assert lib.ssa_window_attn(ok_ptr, ok_ptr, ok_ptr, 1, 1, 1, 8, 32, 1, 2, 0.0, ok_ptr, 1,
                               None, None) == _native.SSA_ERR_UNSUPPORTED


def test_python_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        ssa.ssa_score_topk(x, x, 4, False)
    with pytest.raises(ValueError):
        ssa.ssa_window_attn(x, x, x, 2)


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(OSError):
        _native.load(str(tmp_path / "libssa.so"))


def test_host_validation_of_the_later_calls():
    """ssa_lowrank_project, ssa_sparse_attn_grouped, ssa_score_topk_smooth:
    bad arguments are refused on the host before any launch."""
    lib = ssa.load()
    ok_ptr = V(4096)
    bad_ptr = V(4100)
    BF16, F32 = _native.SSA_BF16, _native.SSA_F32
    # projection: d_model not a multiple of 64, P not 64/128, fp32, misaligned x, empty
    assert lib.ssa_lowrank_project(ok_ptr, ok_ptr, BF16, 8, 100, 64, ok_ptr, None, None) == \
        _native.SSA_ERR_UNSUPPORTED
    assert lib.ssa_lowrank_project(ok_ptr, ok_ptr, BF16, 8, 128, 32, ok_ptr, None, None) == \
        _native.SSA_ERR_UNSUPPORTED
    assert lib.ssa_lowrank_project(ok_ptr, ok_ptr, F32, 8, 128, 64, ok_ptr, None, None) == \
        _native.SSA_ERR_UNSUPPORTED
    assert lib.ssa_lowrank_project(bad_ptr, ok_ptr, BF16, 8, 128, 64, ok_ptr, None, None) == \
        _native.SSA_ERR_INVALID
    assert lib.ssa_lowrank_project(ok_ptr, ok_ptr, BF16, -1, 128, 64, ok_ptr, None, None) == \
        _native.SSA_ERR_INVALID
    assert lib.ssa_lowrank_project(None, None, BF16, 0, 128, 64, None, None, None) == _native.SSA_OK
    # grouped attention: H_kv or H_idx not dividing H, zero groups, unsupported D
    args = lambda H, H_kv, H_idx, D: (ok_ptr, ok_ptr, ok_ptr, BF16, 1, H, H_kv, 8, 8, D,   # noqa: E731
                                      ok_ptr, H_idx, 4, 0.0, ok_ptr, BF16, None, None)
    assert lib.ssa_sparse_attn_grouped(*args(4, 3, 1, 64)) == _native.SSA_ERR_INVALID
    assert lib.ssa_sparse_attn_grouped(*args(4, 2, 3, 64)) == _native.SSA_ERR_INVALID
    assert lib.ssa_sparse_attn_grouped(*args(4, 0, 1, 64)) == _native.SSA_ERR_INVALID
    assert lib.ssa_sparse_attn_grouped(*args(4, 2, 2, 96)) == _native.SSA_ERR_UNSUPPORTED
    # smoothing: k + 1 beyond the largest k, k < 1, workspace too small
    assert lib.ssa_score_topk_smooth(ok_ptr, ok_ptr, BF16, 1, 1, 8, 8, 64, 2048, 0, 0.0, 0.5,
                                     ok_ptr, None, ok_ptr, 1 << 20, None, None) == \
        _native.SSA_ERR_UNSUPPORTED
    assert lib.ssa_score_topk_smooth(ok_ptr, ok_ptr, BF16, 1, 1, 8, 8, 64, 0, 0, 0.0, 0.5,
                                     ok_ptr, None, ok_ptr, 1 << 20, None, None) == \
        _native.SSA_ERR_INVALID
    assert lib.ssa_score_topk_smooth(ok_ptr, ok_ptr, BF16, 1, 1, 8, 8, 64, 4, 0, 0.0, 0.5,
                                     ok_ptr, None, ok_ptr, 16, None, None) == \
        _native.SSA_ERR_WORKSPACE


def test_smooth_workspace_covers_the_larger_selection():
    """The smoothing call needs the workspace of a (k+1) selection plus room
    for its scores; k + 1 beyond the largest supported k has no size."""
    for (B, H, Tq, Tk, P, k) in [(1, 2, 1000, 1000, 64, 64), (1, 8, 4096, 4096, 64, 511),
                                 (2, 3, 77, 400, 16, 40)]:
        a = ssa.score_topk_workspace_size(B, H, Tq, Tk, P, k + 1, True)
        s = ssa.score_topk_smooth_workspace_size(B, H, Tq, Tk, P, k, True)
        assert s >= a + B * H * Tq * (k + 1) * 4
    assert ssa.score_topk_smooth_workspace_size(1, 1, 8, 8, 64, 2048, True) == 0


def test_row_counts_beyond_32_bit_coordinates():
    """The TMA paths address rows with 32-bit coordinates: a projection of
    2^31 rows is refused, and a top-k with 2^31 scorer rows sizes (and would
    run) the row-wise path instead of the tensor-core one."""
    lib = ssa.load()
    ok_ptr = V(4096)
    assert lib.ssa_lowrank_project(ok_ptr, ok_ptr, _native.SSA_BF16, 1 << 31, 128, 64, ok_ptr,
                                   None, None) == _native.SSA_ERR_UNSUPPORTED
    big = ssa.score_topk_workspace_size(1, 32768, 65536, 64, 64, 64, True)   # 2^31 query rows
    rowwise = 1024 * 64 * 4                                                    # 1024 slots of Tk keys
    assert big == rowwise
    assert ssa.score_topk_workspace_size(1, 32767, 65536, 64, 64, 64, True) > rowwise


@pytest.mark.parametrize("bad", [float("nan"), float("inf"), float("-inf")])
def test_non_finite_scale_is_refused(bad):
    """A NaN or infinite scale (or a NaN smoothing threshold) is an invalid
    argument for every call that takes one; nothing is launched."""
    lib = ssa.load()
    ok = V(4096)
    BF16, INV = _native.SSA_BF16, _native.SSA_ERR_INVALID
    assert lib.ssa_score_topk(ok, ok, BF16, 1, 1, 8, 8, 64, 4, 0, bad, ok, None, ok, 1 << 20,
                              None, None) == INV
    assert lib.ssa_score_topk_noalloc(ok, ok, BF16, 1, 1, 8, 8, 64, 4, 0, bad, ok, None, None,
                                      None) == INV
    assert lib.ssa_lowrank_scores(ok, ok, BF16, 1, 1, 8, 8, 64, 0, bad, ok, None, None) == INV
    assert lib.ssa_score_topk_smooth(ok, ok, BF16, 1, 1, 8, 8, 64, 4, 0, bad, 0.5, ok, None, ok,
                                     1 << 20, None, None) == INV
    assert lib.ssa_sparse_attn(ok, ok, ok, BF16, 1, 1, 8, 8, 64, ok, 4, bad, ok, BF16, None,
                               None) == INV
    assert lib.ssa_sparse_attn_grouped(ok, ok, ok, BF16, 1, 4, 2, 8, 8, 64, ok, 1, 4, bad, ok,
                                       BF16, None, None) == INV
    assert lib.ssa_window_attn(ok, ok, ok, BF16, 1, 1, 8, 64, 2, 2, bad, ok, BF16, None,
                               None) == INV
    if bad != bad:   # NaN threshold
        assert lib.ssa_score_topk_smooth(ok, ok, BF16, 1, 1, 8, 8, 64, 4, 0, 0.0, bad, ok, None,
                                         ok, 1 << 20, None, None) == INV


def test_smoothing_k_at_the_int_limit_is_unsupported():
    """k + 1 must not overflow: the largest int k is refused as too large."""
    lib = ssa.load()
    ok = V(4096)
    assert lib.ssa_score_topk_smooth(ok, ok, _native.SSA_BF16, 1, 1, 8, 8, 64, 2 ** 31 - 1, 0,
                                     0.0, 0.5, ok, None, ok, 1 << 20, None, None) == \
        _native.SSA_ERR_UNSUPPORTED
    assert ssa.score_topk_smooth_workspace_size(1, 1, 8, 8, 64, 2 ** 31 - 1, True) == 0


def test_host_validation_of_the_backward_calls():
    """ssa_sparse_attn_bwd / ssa_scorer_bwd refuse bad arguments on the host."""
    lib = ssa.load()
    ok, bad = V(4096), V(4100)
    BF16 = _native.SSA_BF16
    INV, UNS, WS = _native.SSA_ERR_INVALID, _native.SSA_ERR_UNSUPPORTED, _native.SSA_ERR_WORKSPACE
    big = 1 << 30

    def attn(D=64, Tq=8, k=4, scale=0.0, Q=ok, O=ok, wbytes=big, dt=BF16):
        return lib.ssa_sparse_attn_bwd(Q, ok, ok, ok, dt, 1, 1, Tq, 16, D, ok, k, scale, O, ok, ok,
                                       ok, None, ok, wbytes, None, None)

    assert attn(D=96) == UNS
    assert attn(Tq=1 << 20, k=4096) == UNS          # Tq * k beyond 32-bit pair ids
    assert attn(scale=float("nan")) == INV
    assert attn(Q=None) == INV                      # query rows but no Q
    assert attn(O=bad) == INV                       # misaligned dQ
    assert attn(dt=7) == INV
    assert attn(wbytes=16) == WS
    assert lib.ssa_sparse_attn_bwd(None, None, None, None, BF16, 0, 1, 8, 16, 64, None, 4, 0.0,
                                   None, None, None, None, None, None, 0, None, None) == _native.SSA_OK
    assert lib.ssa_sparse_attn_bwd_workspace_size(1, 1, 8, 16, 0) == 0

    def scorer(P=64, scale=0.0, dS=ok, wbytes=big):
        return lib.ssa_scorer_bwd(ok, ok, BF16, 1, 1, 8, 16, P, ok, 4, dS, scale, ok, ok, ok, wbytes,
                                  None, None)

    assert scorer(P=48) == UNS
    assert scorer(scale=float("inf")) == INV
    assert scorer(dS=None) == INV
    assert scorer(wbytes=16) == WS
    assert lib.ssa_scorer_bwd_workspace_size(1, 1, 8, 16, -1) == 0


def test_host_validation_of_the_grouped_backward_calls():
    lib = ssa.load()
    ok = V(4096)
    BF16, INV, UNS = _native.SSA_BF16, _native.SSA_ERR_INVALID, _native.SSA_ERR_UNSUPPORTED

    def attn(H=4, H_kv=2, H_idx=1, D=64, Tq=8, k=4):
        return lib.ssa_sparse_attn_grouped_bwd(ok, ok, ok, ok, BF16, 1, H, H_kv, Tq, 16, D, ok, H_idx,
                                               k, 0.0, ok, ok, ok, ok, None, ok, 1 << 30, None, None)

    assert attn(H_kv=3) == INV            # does not divide H
    assert attn(H_idx=0) == INV
    assert attn(D=96) == UNS
    assert attn(H=8, H_kv=1, Tq=1 << 20, k=512) == UNS   # 8 query heads' pair ids overflow 32 bits
    assert lib.ssa_sparse_attn_grouped_bwd_workspace_size(1, 4, 3, 8, 16, 4) == 0
    assert (lib.ssa_sparse_attn_grouped_bwd_workspace_size(1, 4, 4, 8, 16, 4) ==
            lib.ssa_sparse_attn_bwd_workspace_size(1, 4, 8, 16, 4))

    def scorer(H=4, H_idx=1, P=64):
        return lib.ssa_scorer_grouped_bwd(ok, ok, BF16, 1, H, H_idx, 8, 16, P, ok, 4, ok, 0.0, ok,
                                          ok, ok, 1 << 30, None, None)

    assert scorer(H_idx=3) == INV
    assert scorer(P=48) == UNS
    # one scorer head shared by 4 query heads needs room for the summed pair gradients
    assert (lib.ssa_scorer_grouped_bwd_workspace_size(1, 4, 1, 8, 16, 4) >
            lib.ssa_scorer_grouped_bwd_workspace_size(1, 1, 1, 8, 16, 4))


def test_host_validation_of_the_wait_limit_selftest():
    lib = ssa.load()
    INV = _native.SSA_ERR_INVALID
    assert lib.ssa_selftest_wait_limit(None, 1000, None) == INV        # no status word
    assert lib.ssa_selftest_wait_limit(V(4098), 1000, None) == INV     # misaligned
    assert lib.ssa_selftest_wait_limit(V(4096), 0, None) == INV        # no limit
    assert lib.ssa_selftest_wait_limit(V(4096), 2 * 10 ** 9, None) == INV   # over a second


def test_host_validation_of_the_device_status_reader():
    lib = ssa.load()
    INV = _native.SSA_ERR_INVALID
    assert lib.ssa_device_status(None, None, None) == INV       # no status word
    assert lib.ssa_device_status(V(4098), None, None) == INV    # misaligned
    # the status codes keep the values the boundary defines
    assert (_native.SSA_ERR_TIMEOUT, _native.SSA_ERR_WORKSPACE) == (4, 5)
    assert b"wait" in lib.ssa_status_string(_native.SSA_ERR_TIMEOUT)
    assert b"workspace" in lib.ssa_status_string(_native.SSA_ERR_WORKSPACE)
