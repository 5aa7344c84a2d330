"""Backward pass on the GPU against the float64 backward oracle, through the C ABI
(needs a GB300).

The O and LSE inputs of every call come from the forward oracle (O rounded to
bf16, LSE to float32); dO is drawn by ``inputs.make_grad``.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_34_gb300 import fa, inputs
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from exact_io_aware_34_gb300 import build
    build.build()
    fa.load_library()


def _column_sum_properties(dk, dv, do):
    """Rows of P sum to one, so sum_j dV_j = sum_i dO_i for every (b, h, column).
    The bf16 rounding of P (2^-9 relative) and of dV bound the gap by
    2^-8 (sum_i |dO_i| + sum_j |dV_j|); 1e-2 of that mass is allowed. (sum_j dK_j = 0 holds only
    when D equals rowsum(P * dP) exactly; with D taken from a bf16 O, as the
    recomputation does, it is off by scale * sum_i delta_i q_i, so it is not
    checked.)"""
    dk, dv, do = (x.double() for x in (dk, dv, do))
    assert torch.isfinite(dk).all() and torch.isfinite(dv).all()
    mass = dv.abs().sum(2) + do.abs().sum(2)
    assert bool(((dv.sum(2) - do.sum(2)).abs() <= 1e-2 * mass + 1e-6).all())


# --- shapes: ragged tails, several blocks, B*H > 1 ---------------------------------
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 2, 64, 127, 128, 129, 255, 256, 300, 513, 1000])
def test_bwd_shapes(N, d):
    q, k, v = inputs.make_random(2, 3, N, d, seed=N * 11 + d)
    do = inputs.make_grad(2, 3, N, d, seed=N * 11 + d)
    err, got = parity.check_bwd_full(q, k, v, do, 1 / math.sqrt(d), two_x_rule=N >= 64)
    _column_sum_properties(got[1], got[2], do)
    print(N, d, {n: (e["max"], e.get("naive_max")) for n, e in err.items()})


# --- the named workloads that the oracle evaluates whole -------------------------
@pytest.mark.parametrize("name", ["n256_d64", "n1024_d64_b4h16"])
def test_bwd_workload_full(name):
    w = inputs.workload(name)
    q, k, v, s = inputs.make_inputs(w)
    do = inputs.make_grad(w.B, w.H, w.N, w.d, w.seed)
    err, _ = parity.check_bwd_full(q, k, v, do, s)
    print(name, err)


# --- full-size workloads: whole heads checked, properties everywhere -------------
@pytest.mark.parametrize("name,heads", [
    ("n4096_d128_b2h16", [(0, 0), (1, 15)]),
    ("prefill8k_d128_h32", [(0, 0), (0, 31)]),
])
def test_bwd_workload_full_size(name, heads):
    w = inputs.workload(name)
    q, k, v, s = inputs.make_inputs(w)
    do = inputs.make_grad(w.B, w.H, w.N, w.d, w.seed)
    o, lse = parity.oracle_forward_inputs(q, k, v, s)
    dq, dk, dv = parity.run_gpu_bwd(q, k, v, o, do, lse, s)
    _column_sum_properties(dk, dv, do)
    Q, K, V, dO = (parity.to64(x) for x in (q, k, v, do))
    refs = oracle.attention_bwd_heads(Q, K, V, dO, s, heads)
    naives = oracle.naive_bf16_attention_bwd(Q, K, V, dO, s, heads=heads)
    for (b, h), ref, naive in zip(heads, refs, naives):
        err = parity.bwd_errors((dq[b, h], dk[b, h], dv[b, h]), ref, naive)
        parity.assert_bwd_within(err)
        print(name, (b, h), {n: (e["max"], e["naive_max"]) for n, e in err.items()})


# --- value distributions and degenerate cases -----------------------------------
def test_bwd_spiky_logits():
    """Large logits (Q, K ~ N(0, 9), 1% of key rows x8): probabilities far from uniform."""
    q, k, v = inputs.make_random(1, 2, 2048, 128, seed=77, q_dist="normal3", k_dist="normal3", spike_frac=0.01)
    do = inputs.make_grad(1, 2, 2048, 128, seed=77)
    err, _ = parity.check_bwd_full(q, k, v, do, 1 / math.sqrt(128))
    print(err)


def test_bwd_scale_zero():
    """scale = 0: P is uniform (1/N); dQ = dK = 0 exactly in the oracle."""
    q, k, v = inputs.make_random(1, 2, 300, 64, seed=78)
    do = inputs.make_grad(1, 2, 300, 64, seed=78)
    err, got = parity.check_bwd_full(q, k, v, do, 0.0, two_x_rule=False)
    assert float(got[0].abs().max()) == 0.0 and float(got[1].abs().max()) == 0.0


def test_bwd_constant_v_gives_zero_dq_dk():
    """Every value row equal: O does not depend on the weights, so dQ = dK = 0
    (up to rounding of dP - D, which cancel exactly in real arithmetic)."""
    q, k, _ = inputs.make_random(1, 2, 257, 128, seed=79)
    v = torch.ones(1, 2, 257, 128, dtype=torch.bfloat16) * 0.5
    do = inputs.make_grad(1, 2, 257, 128, seed=79)
    o, lse = parity.oracle_forward_inputs(q, k, v, 1 / math.sqrt(128))
    dq, dk, dv = parity.run_gpu_bwd(q, k, v, o, do, lse, 1 / math.sqrt(128))
    assert float(dq.abs().max()) < 1e-3 and float(dk.abs().max()) < 1e-3


def test_bwd_deterministic_and_on_a_side_stream():
    """No atomics: two calls give identical bits, also on a non-default stream."""
    q, k, v = inputs.make_random(2, 4, 1000, 128, seed=80)
    do = inputs.make_grad(2, 4, 1000, 128, seed=80)
    o, lse = parity.oracle_forward_inputs(q, k, v, 0.1)
    a = parity.run_gpu_bwd(q, k, v, o, do, lse, 0.1)
    side = torch.cuda.Stream()
    b = parity.run_gpu_bwd(q, k, v, o, do, lse, 0.1, stream=side)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_bwd_outputs_fully_written_and_guard_bands_untouched():
    """Every output element is written; bytes around the outputs are not."""
    B, H, N, d = 1, 2, 200, 64
    q, k, v = inputs.make_random(B, H, N, d, seed=81)
    do = inputs.make_grad(B, H, N, d, seed=81)
    o, lse = parity.oracle_forward_inputs(q, k, v, 0.125)
    dev = "cuda:0"
    n = B * H * N * d
    pad = 4096
    bufs = [torch.full((n + 2 * pad,), float("nan"), dtype=torch.bfloat16, device=dev) for _ in range(3)]
    outs = [b[pad:pad + n].view(B, H, N, d) for b in bufs]
    args = [x.to(dev) for x in (q, k, v, o, do, lse)]
    fa.fa_bwd(*args, dq=outs[0], dk=outs[1], dv=outs[2], scale=0.125)
    torch.cuda.synchronize()
    for b, x in zip(bufs, outs):
        assert torch.isfinite(x.float()).all()
        assert torch.isnan(b[:pad].float()).all() and torch.isnan(b[pad + n:].float()).all()


def test_bwd_small_workspace_rejected():
    q, k, v = (x.cuda() for x in inputs.make_random(1, 1, 256, 64, seed=82))
    o = torch.zeros_like(q)
    lse = torch.zeros(1, 1, 256, device="cuda")
    ws = torch.empty(fa.fa_bwd_workspace_bytes(1, 1, 256) - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError):
        fa.fa_bwd(q, k, v, o, torch.zeros_like(q), lse, workspace=ws)


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_negative_scale(d):
    """scale < 0: P = exp(scale Q K^T - LSE) and the scale factors of dQ and dK
    carry the sign."""
    q, k, v = inputs.make_random(1, 3, 500, d, seed=90 + d)
    do = inputs.make_grad(1, 3, 500, d, seed=90 + d)
    err, got = parity.check_bwd_full(q, k, v, do, -1 / math.sqrt(d))
    _column_sum_properties(got[1], got[2], do)
    print(d, err)
