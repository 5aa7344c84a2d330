"""The seeded input generator (CPU only)."""
import math

import torch

from exact_io_aware_34_gb300 import inputs


def test_deterministic_and_bf16():
    a = inputs.make_random(1, 2, 64, 64, seed=7)
    b = inputs.make_random(1, 2, 64, 64, seed=7)
    c = inputs.make_random(1, 2, 64, 64, seed=8)
    for x, y in zip(a, b):
        assert x.dtype == torch.bfloat16 and x.shape == (1, 2, 64, 64)
        assert torch.equal(x, y)
    assert not torch.equal(a[0], c[0])
    assert inputs.sha256_of(*a) == inputs.sha256_of(*b) != inputs.sha256_of(*c)


def test_workload_table():
    assert [w.N for w in inputs.WORKLOADS] == [256, 1024, 4096, 8192, 32768]
    assert [w.d for w in inputs.WORKLOADS] == [64, 64, 128, 128, 128]
    w = inputs.workload("prefill8k_d128_h32")
    assert (w.B, w.H) == (1, 32) and w.v_dist == "uniform"
    assert w.flops == 4 * 32 * 8192 ** 2 * 128
    assert abs(w.scale - 1 / math.sqrt(128)) < 1e-15
    assert inputs.workload(4) is w


def test_distributions():
    q, k, v = inputs.make_random(1, 4, 4096, 64, seed=3, q_dist="normal3", v_dist="uniform")
    assert abs(q.float().std().item() - 3.0) < 0.05
    assert abs(k.float().std().item() - 1.0) < 0.02
    assert v.float().min().item() >= -1.0 and v.float().max().item() <= 1.0


def test_spikes():
    """1% of key rows of each head are scaled by exactly 8 (exact in bf16)."""
    B, H, N, d = 1, 3, 1000, 16
    q0, k0, v0 = inputs.make_random(B, H, N, d, seed=5)
    q1, k1, v1 = inputs.make_random(B, H, N, d, seed=5, spike_frac=0.01)
    assert torch.equal(q0, q1) and torch.equal(v0, v1)
    for h in range(H):
        changed = (k0[0, h] != k1[0, h]).any(dim=1)
        assert int(changed.sum()) == 10
        assert torch.equal(k1[0, h][changed].float(), k0[0, h][changed].float() * 8)
