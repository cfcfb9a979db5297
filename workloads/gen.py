"""Seeded synthetic inputs for dynamic top-k sparse attention.

This module holds no arithmetic of the method itself: it only turns
(seed, tensor id, element index) into numbers, so that the CUDA path, the CPU
oracle, the tests and the benchmark all see the same inputs. It runs with
plain torch ops on either the CPU or a CUDA device and produces identical
integers on both; normal variates go through float64 Box-Muller and are then
rounded to the tensor's dtype.

Generator: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014). Element ``e`` of the stream
with key ``K`` is the (e+1)-th SplitMix64 output seeded with ``K``:
``mix(K + (e + 1) * GAMMA)``. The stream key of tensor ``tid`` under seed
``s`` is ``mix(s * GAMMA + tid)``. All arithmetic is modulo 2**64, carried in
int64 (torch's int64 multiply wraps); logical right shifts are emulated with a
mask.

Value maps:
  * integer in [-4, 4]: ``((u >> 32) * 9) >> 32`` minus 4 (multiply-shift range
    reduction of the high 32 bits),
  * standard normal: Box-Muller, ``u1 = (hi24 + 1) / 2**24``,
    ``u2 = lo24 / 2**24``, ``z = sqrt(-2 ln u1) * cos(2 pi u2)``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK64 = (1 << 64) - 1


def _s64(x: int) -> int:
    """Reinterpret an unsigned 64-bit integer as int64."""
    x &= _MASK64
    return x - (1 << 64) if x >= (1 << 63) else x


def _lsr(x: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (x >> s) & ((1 << (64 - s)) - 1)


def _mix_t(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _lsr(z, 30)) * _s64(_M1)
    z = (z ^ _lsr(z, 27)) * _s64(_M2)
    return z ^ _lsr(z, 31)


def splitmix64_ref(key: int, e: int) -> int:
    """Pure-Python SplitMix64 output ``e`` of stream ``key`` (unsigned)."""
    z = (key + (e + 1) * GAMMA) & _MASK64
    z = ((z ^ (z >> 30)) * _M1) & _MASK64
    z = ((z ^ (z >> 27)) * _M2) & _MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, tid: int) -> int:
    """Unsigned 64-bit stream key of tensor ``tid`` under ``seed``."""
    z = (seed * GAMMA + tid) & _MASK64
    z = ((z ^ (z >> 30)) * _M1) & _MASK64
    z = ((z ^ (z >> 27)) * _M2) & _MASK64
    return z ^ (z >> 31)


def raw_bits(key: int, start: int, n: int, device) -> torch.Tensor:
    """int64 bit patterns of outputs start..start+n-1 of stream ``key``."""
    e = torch.arange(start + 1, start + n + 1, dtype=torch.int64, device=device)
    z = e * _s64(GAMMA) + _s64(key)
    return _mix_t(z)


def ints_m4_4(bits: torch.Tensor) -> torch.Tensor:
    """Integers uniform on [-4, 4] from 64-bit patterns."""
    return _lsr(_lsr(bits, 32) * 9, 32) - 4


def normals(bits: torch.Tensor) -> torch.Tensor:
    """Standard normal float64 variates from 64-bit patterns."""
    hi = _lsr(bits, 40).to(torch.float64)
    lo = (bits & 0xFFFFFF).to(torch.float64)
    u1 = (hi + 1.0) * (1.0 / 16777216.0)
    u2 = lo * (1.0 / 16777216.0)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


_CHUNK = 1 << 25


def fill(shape, kind: str, seed: int, tid: int, dtype, device) -> torch.Tensor:
    """A tensor of ``shape`` whose flat element e is draw e of stream (seed, tid).

    ``kind`` is "int" (integers in [-4, 4]) or "normal". Generation runs in
    chunks so that int64 intermediates stay small on the device.
    """
    n = 1
    for s in shape:
        n *= int(s)
    out = torch.empty(n, dtype=dtype, device=device)
    key = stream_key(seed, tid)
    for start in range(0, n, _CHUNK):
        m = min(_CHUNK, n - start)
        bits = raw_bits(key, start, m, device)
        if kind == "int":
            v = ints_m4_4(bits)
        elif kind == "normal":
            v = normals(bits)
        else:
            raise ValueError(kind)
        out[start:start + m] = v.to(dtype)
        del bits, v
    return out.view(*shape)


# Tensor ids inside one workload's seed.
TID_QLOW, TID_KLOW, TID_Q, TID_K, TID_V, TID_PLANT_POS, TID_PLANT_GROUP = 1, 2, 3, 4, 5, 6, 7
TID_DO = 8   # the incoming gradient of the attention output (backward workloads)


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, dtype and structure of the inputs."""
    name: str
    B: int
    H: int
    Tq: int
    Tk: int
    D: int
    dtype: str              # "f32" or "bf16"
    P: int = 0              # d_proj of the scorer (0: no scorer, window workload)
    k: int = 0              # selection size
    causal: bool = False
    window: int = -1        # |i - j| <= window (window workload only)
    planted: int = 0        # planted keys per query group (0: none)
    plant_boost: int = 64   # exact dot-product boost of a planted key
    equal_scores: bool = False   # q_low = 0: every score 0 (the all-ties case)
    seed_base: int = 1234
    cfg_id: int = 0
    notes: str = field(default="", compare=False)

    @property
    def seed(self) -> int:
        return self.seed_base + self.cfg_id

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def n_queries(self) -> int:
        return self.B * self.H * self.Tq

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


WORKLOADS = {
    "topk_f32_t1024_k32": Workload(
        "topk_f32_t1024_k32", B=1, H=2, Tq=1024, Tk=1024, D=64, dtype="f32",
        P=16, k=32, causal=False, cfg_id=0,
        notes="fp32, non-causal; integer q_low/k_low; Q/K/V ~ N(0,1)"),
    "window_bf16_t4096_w128": Workload(
        "window_bf16_t4096_w128", B=2, H=8, Tq=4096, Tk=4096, D=64, dtype="bf16",
        window=128, cfg_id=1, notes="sliding window |i-j|<=128 clipped at both ends"),
    "topk_causal_bf16_t32k_k256": Workload(
        "topk_causal_bf16_t32k_k256", B=1, H=16, Tq=32768, Tk=32768, D=128, dtype="bf16",
        P=64, k=256, causal=True, cfg_id=2),
    "topk_causal_bf16_t128k_k512_planted": Workload(
        "topk_causal_bf16_t128k_k512_planted", B=1, H=8, Tq=131072, Tk=131072, D=128,
        dtype="bf16", P=64, k=512, causal=True, planted=16, cfg_id=3,
        notes="16 planted keys per query group, dot product boosted by exactly +64"),
    "topk_causal_bf16_t128k_k512_equal_scores": Workload(
        "topk_causal_bf16_t128k_k512_equal_scores", B=1, H=8, Tq=131072, Tk=131072, D=128,
        dtype="bf16", P=64, k=512, causal=True, equal_scores=True, cfg_id=3,
        notes="the 128K workload with q_low = 0: every score ties, each row selects its "
              "first k_eff keys"),
    "decode_bf16_b32_tk64k_k512": Workload(
        "decode_bf16_b32_tk64k_k512", B=32, H=32, Tq=1, Tk=65536, D=128, dtype="bf16",
        P=64, k=512, causal=False, cfg_id=4, notes="one query per head against 65536 cached keys"),
}


# Planting (integer test data): the last 16 of the 64 scorer dimensions form
# 4 groups of 4. Each query picks a group; a planted key carries the value 4 in
# its group's 4 dimensions, so q_low.k_low gains exactly 4*4*4 = 64 while the
# other 48 dimensions stay uniform integers in [-4, 4].
PLANT_GROUPS = 4
PLANT_DIMS = 4
PLANT_VALUE = 4


def plant_positions(w: Workload, device="cpu") -> torch.Tensor:
    """Planted key positions, int64 [B, H, PLANT_GROUPS, planted].

    Stratified draw: position m lies in stratum m of Tk/planted equal strata,
    so the planted keys of one group are distinct and spread over the sequence.
    """
    n = w.B * w.H * PLANT_GROUPS * w.planted
    bits = raw_bits(stream_key(w.seed, TID_PLANT_POS), 0, n, device)
    width = w.Tk // w.planted
    m = torch.arange(n, device=device) % w.planted
    off = _lsr(_lsr(bits, 32) * width, 32)
    return (m * width + off).view(w.B, w.H, PLANT_GROUPS, w.planted)


def plant_groups(w: Workload, device="cpu") -> torch.Tensor:
    """Group of each query row, int64 [B, H, Tq] in [0, PLANT_GROUPS)."""
    n = w.B * w.H * w.Tq
    bits = raw_bits(stream_key(w.seed, TID_PLANT_GROUP), 0, n, device)
    return _lsr(_lsr(bits, 32) * PLANT_GROUPS, 32).view(w.B, w.H, w.Tq)


def make_scorer_inputs(w: Workload, device="cpu"):
    """(q_low, k_low) in the workload dtype, [B,H,Tq,P] and [B,H,Tk,P]."""
    dt = w.torch_dtype
    q = fill((w.B, w.H, w.Tq, w.P), "int", w.seed, TID_QLOW, dt, device)
    k = fill((w.B, w.H, w.Tk, w.P), "int", w.seed, TID_KLOW, dt, device)
    if w.equal_scores:
        q.zero_()
    elif w.planted:
        base = w.P - PLANT_GROUPS * PLANT_DIMS
        assert base > 0
        q[..., base:] = 0
        k[..., base:] = 0
        grp = plant_groups(w, device)
        pos = plant_positions(w, device)
        for g in range(PLANT_GROUPS):
            lo, hi = base + g * PLANT_DIMS, base + (g + 1) * PLANT_DIMS
            qm = (grp == g).unsqueeze(-1)
            q[..., lo:hi] = torch.where(qm, torch.full_like(q[..., lo:hi], PLANT_VALUE), q[..., lo:hi])
            for b in range(w.B):
                for h in range(w.H):
                    k[b, h, pos[b, h, g], lo:hi] = PLANT_VALUE
    return q, k


def make_attn_inputs(w: Workload, device="cpu"):
    """(Q, K, V) ~ N(0,1) rounded to the workload dtype."""
    dt = w.torch_dtype
    Q = fill((w.B, w.H, w.Tq, w.D), "normal", w.seed, TID_Q, dt, device)
    K = fill((w.B, w.H, w.Tk, w.D), "normal", w.seed, TID_K, dt, device)
    V = fill((w.B, w.H, w.Tk, w.D), "normal", w.seed, TID_V, dt, device)
    return Q, K, V


def make_grad_output(w: Workload, device="cpu"):
    """dO ~ N(0,1) [B,H,Tq,D] in the workload dtype: the gradient reaching the
    attention output in a backward step."""
    return fill((w.B, w.H, w.Tq, w.D), "normal", w.seed, TID_DO, w.torch_dtype, device)


def small(name: str, **kw) -> Workload:
    """A named workload with some fields overridden (small parity cases)."""
    return WORKLOADS[name].with_(**kw)
