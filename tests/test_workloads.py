"""The seeded input generator: SplitMix64 streams and value maps (CPU)."""
import numpy as np
import torch

from workloads import WORKLOADS, fill
from workloads.gen import raw_bits, splitmix64_ref, stream_key


def test_splitmix64_matches_reference():
    # Published first outputs of SplitMix64 seeded with 0 (Steele/Lea/Flood reference code).
    assert splitmix64_ref(0, 0) == 0xE220A8397B1DCDAF
    assert splitmix64_ref(0, 1) == 0x6E789E6AA1B965F4
    assert splitmix64_ref(0, 2) == 0x06C45D188009454F
    for key in [0, 1, stream_key(1234, 3), stream_key(7, 2)]:
        bits = raw_bits(key, 1000, 64, "cpu")
        want = [splitmix64_ref(key, 1000 + e) for e in range(64)]
        got = [int(b) & ((1 << 64) - 1) for b in bits.tolist()]
        assert got == want


def test_value_maps():
    x = fill((200000,), "int", 1, 2, torch.float32, "cpu")
    assert x.min() == -4 and x.max() == 4
    counts = torch.bincount((x + 4).long(), minlength=9).double() / x.numel()
    assert torch.allclose(counts, torch.full((9,), 1 / 9, dtype=torch.float64), atol=5e-3)
    z = fill((400000,), "normal", 1, 3, torch.float64, "cpu")
    assert abs(z.mean().item()) < 0.01 and abs(z.std().item() - 1.0) < 0.01
    # chunked generation equals one-shot generation
    a = fill((3, 5, 7), "normal", 9, 4, torch.bfloat16, "cpu")
    b = fill((105,), "normal", 9, 4, torch.bfloat16, "cpu")
    assert torch.equal(a.flatten(), b)


def test_workload_shapes():
    w = WORKLOADS["topk_causal_bf16_t128k_k512_planted"]
    assert (w.B, w.H, w.Tq, w.D, w.P, w.k, w.causal) == (1, 8, 131072, 128, 64, 512, True)
    assert WORKLOADS["decode_bf16_b32_tk64k_k512"].n_queries == 1024
