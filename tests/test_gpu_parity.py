"""CUDA path vs the float64 oracle, through the C ABI (needs a GB300)."""
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


# --- the five named workloads -------------------------------------------------
def test_workload_n256_d64_full():
    q, k, v, s = inputs.make_inputs(inputs.workload("n256_d64"))
    err, _, _ = parity.check_full(q, k, v, s)
    print(err)


def test_workload_n1024_d64_b4h16_full():
    q, k, v, s = inputs.make_inputs(inputs.workload("n1024_d64_b4h16"))
    err, _, _ = parity.check_full(q, k, v, s)
    print(err)


@pytest.mark.parametrize("name", ["n4096_d128_b2h16", "prefill8k_d128_h32", "long32k_d128_h16_spiky"])
def test_workload_full_size_every_row(name, tmp_path):
    """Every one of the B*H*N output rows of the full-size workload, in the
    launch configuration the benchmark times, against the float64 oracle (O
    max-abs, O relative Frobenius, LSE max-abs over all rows, and the 2x rule
    against the bf16 materialise-path reference over all rows)."""
    q, k, v, s = inputs.make_inputs(inputs.workload(name))
    err = parity.check_full_parallel(q, k, v, s, tmp_path)
    print(name, f"{err['rows_checked']} of {err['rows_total']} rows checked", err)


def test_workload_n4096_full_one_head():
    """Every row of one full-size head (first batch, head 0) of the N=4096 workload."""
    q, k, v, s = inputs.make_inputs(inputs.workload("n4096_d128_b2h16"))
    o, lse = parity.run_gpu(q, k, v, s)
    Q, K, V = (parity.to64(x[:1, :1]) for x in (q, k, v))
    O_ref, L_ref = oracle.attention(Q, K, V, s)
    err = parity.errors(o[:1, :1], lse[:1, :1], O_ref, L_ref)
    assert err["o_max"] <= parity.TOL_O_MAX and err["o_fro"] <= parity.TOL_O_FRO
    assert err["lse_max"] <= parity.TOL_LSE_MAX, err


# --- shapes: ragged tails, several tiles, B*H > 1 -----------------------------------
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 2, 7, 64, 127, 128, 129, 200, 255, 256, 257, 383, 384, 513, 1000])
def test_shapes(N, d):
    q, k, v = inputs.make_random(2, 3, N, d, seed=N * 7 + d)
    err, _, _ = parity.check_full(q, k, v, 1 / math.sqrt(d), two_x_rule=N >= 64)
    print(N, d, err)


@pytest.mark.parametrize("d", [64, 128])
def test_many_heads_small_n(d):
    q, k, v = inputs.make_random(3, 40, 96, d, seed=5)
    parity.check_full(q, k, v, 1 / math.sqrt(d))


# --- degenerate cases --------------------------------------------------------------
@pytest.mark.parametrize("d", [64, 128])
def test_scale_zero_gives_uniform_weights(d):
    """scale = 0: every weight is 1/N, O = mean of V, LSE = ln N."""
    N = 300
    q, k, v = inputs.make_random(1, 2, N, d, seed=9)
    o, lse = parity.run_gpu(q, k, v, 0.0)
    mean = v.float().mean(dim=2, keepdim=True).expand_as(o)
    assert torch.allclose(o.float(), mean, atol=1e-2, rtol=0)
    assert torch.allclose(lse, torch.full_like(lse, math.log(N)), atol=1e-4, rtol=0)


@pytest.mark.parametrize("d", [64, 128])
def test_constant_v_rows(d):
    """Every value row equal to v: O = v for every query."""
    N = 777
    q, k, _ = inputs.make_random(1, 2, N, d, seed=10, q_dist="normal3", k_dist="normal3")
    vrow = torch.randn(d, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    v = vrow.expand(1, 2, N, d).contiguous()
    o, _ = parity.run_gpu(q, k, v, 1 / math.sqrt(d))
    assert torch.allclose(o.float(), v.float(), atol=2e-2, rtol=1e-2)


def test_zero_q_and_equal_keys():
    q, k, v = inputs.make_random(2, 2, 333, 128, seed=11, q_dist="zeros")
    parity.check_full(q, k, v, 0.3, two_x_rule=False)
    q, _, v = inputs.make_random(2, 2, 333, 128, seed=12)
    k = q[:, :, :1].expand(-1, -1, 333, -1).contiguous()
    parity.check_full(q, k, v, 0.3, two_x_rule=False)


def test_large_scale_near_hardmax():
    """A large scale concentrates each row on its best key; the running max moves a lot."""
    q, k, v = inputs.make_random(1, 2, 640, 64, seed=13)
    parity.check_full(q, k, v, 2.0, two_x_rule=False)


def test_spiky_keys_small():
    """The long-context stress pattern (std-3 logits, 1% of keys x8) at a size the
    oracle evaluates in full."""
    q, k, v = inputs.make_random(1, 4, 2048, 128, seed=14, q_dist="normal3", k_dist="normal3",
                                 spike_frac=0.01)
    err, _, _ = parity.check_full(q, k, v, 1 / math.sqrt(128))
    print(err)


def test_rising_maximum_forces_rescales():
    """Scores that grow key block by key block make the running maximum move on
    every block, exercising the O rescale path on each one."""
    N, d = 1024, 64
    q, k, v = inputs.make_random(1, 1, N, d, seed=15)
    ramp = torch.linspace(0.2, 4.0, N).view(1, 1, N, 1)
    k = (q[:, :, :1].float() * ramp).to(torch.bfloat16)   # every key aligned with query 0, growing
    parity.check_full(q, k, v, 1.0, two_x_rule=False)


# --- buffers, streams, repeatability -------------------------------------------------
def test_guard_bands_untouched():
    """O and LSE are written exactly in place: sentinels around them survive."""
    B, H, N, d = 1, 2, 300, 128
    q, k, v = inputs.make_random(B, H, N, d, seed=16)
    dev = "cuda:0"
    pad = 256
    o_buf = torch.full((pad + B * H * N * d + pad,), 7.0, dtype=torch.bfloat16, device=dev)
    l_buf = torch.full((pad + B * H * N + pad,), -3.0, dtype=torch.float32, device=dev)
    o = o_buf[pad:pad + B * H * N * d].view(B, H, N, d)
    lse = l_buf[pad:pad + B * H * N].view(B, H, N)
    fa.fa_fwd(q.to(dev), k.to(dev), v.to(dev), o, lse, scale=1 / math.sqrt(d))
    torch.cuda.synchronize()
    assert bool((o_buf[:pad] == 7.0).all()) and bool((o_buf[-pad:] == 7.0).all())
    assert bool((l_buf[:pad] == -3.0).all()) and bool((l_buf[-pad:] == -3.0).all())
    O_ref, L_ref = oracle.attention(*(parity.to64(x) for x in (q, k, v)), 1 / math.sqrt(d))
    err = parity.errors(o.cpu(), lse.cpu(), O_ref, L_ref)
    assert err["o_max"] <= parity.TOL_O_MAX and err["lse_max"] <= parity.TOL_LSE_MAX


def test_side_stream_and_determinism():
    q, k, v = inputs.make_random(2, 4, 1111, 64, seed=17)
    qd, kd, vd = (x.cuda() for x in (q, k, v))
    o1, l1 = fa.fa_fwd(qd, kd, vd)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o2, l2 = fa.fa_fwd(qd, kd, vd, stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert fa.fa_get_device_status()[0] == fa.FA_OK


def test_no_device_allocation_by_library():
    """With O and LSE preallocated, a call allocates no device memory."""
    q, k, v = (x.cuda() for x in inputs.make_random(1, 8, 2048, 128, seed=18))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    fa.fa_fwd(q, k, v, o, lse)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    before = torch.cuda.memory_allocated()
    for _ in range(3):
        fa.fa_fwd(q, k, v, o, lse)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == before
    assert abs(free1 - free0) < (2 << 20)


def test_python_binding_checks():
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        fa.fa_fwd(q.float(), q, q)
    with pytest.raises(ValueError):
        fa.fa_fwd(q, q[:, :, :4], q)
    with pytest.raises(ValueError):
        fa.fa_fwd(q.transpose(2, 3), q.transpose(2, 3), q.transpose(2, 3))
    with pytest.raises(fa.FaError) as ei:
        fa.fa_fwd(torch.zeros(1, 1, 8, 96, dtype=torch.bfloat16, device="cuda"),
                  torch.zeros(1, 1, 8, 96, dtype=torch.bfloat16, device="cuda"),
                  torch.zeros(1, 1, 8, 96, dtype=torch.bfloat16, device="cuda"))
    assert ei.value.status == fa.FA_ERR_UNSUPPORTED


def test_lse_rebuilds_probabilities():
    """LSE is the value a backward pass needs: exp(scale*q.k - LSE) sums to 1 per row."""
    q, k, v = inputs.make_random(1, 2, 500, 128, seed=19)
    s = 1 / math.sqrt(128)
    _, lse = parity.run_gpu(q, k, v, s)
    S = s * (parity.to64(q) @ np.swapaxes(parity.to64(k), -1, -2))
    rows = np.exp(S - parity.to64(lse)[..., None]).sum(-1)
    assert np.abs(rows - 1).max() < 2e-3


# --- negative scale ----------------------------------------------------------------
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("scale", [-0.1, -0.125, -1.5])
def test_negative_scale(d, scale):
    """scale < 0 puts the most weight on the keys least aligned with each query;
    the kernel has the tensor core form -S and runs with |scale|."""
    q, k, v = inputs.make_random(2, 3, 700, d, seed=20 + d)
    err, _, _ = parity.check_full(q, k, v, scale, two_x_rule=abs(scale) <= 0.2)
    print(d, scale, err)


@pytest.mark.parametrize("d", [64, 128])
def test_negative_scale_equals_negated_keys(d):
    """scale * Q K^T = |scale| * Q (-K)^T: negating the scale or the keys gives
    the same scores (negation is exact), so the two calls agree bit for bit."""
    q, k, v = inputs.make_random(1, 2, 513, d, seed=23 + d)
    o1, l1 = parity.run_gpu(q, k, v, -0.09)
    o2, l2 = parity.run_gpu(q, -k, v, 0.09)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


# --- units shared by CTA pairs (the split last round) ----------------------------
@pytest.mark.parametrize("d", [64, 128])
def test_whole_rounds_then_split_tail(d):
    """40 heads of 1024 rows are 160 units of 256 rows: one whole round on the
    SMs, then 8 units each shared by a pair of CTAs (half of the 8 key blocks
    each, merged through distributed shared memory). Every row against the
    oracle."""
    q, k, v = inputs.make_random(1, 40, 1024, d, seed=50 + d)
    err, _, _ = parity.check_full(q, k, v, 1 / math.sqrt(d))
    print(d, err)


@pytest.mark.parametrize("d", [64, 128])
def test_long_sequence_sampled_rows(d):
    """131000 rows and keys per head (1024 key blocks per unit, the last one
    ragged; 512 units of which the last is partial): sampled rows against the
    oracle, every row finite and inside the range of V."""
    q, k, v = inputs.make_random(1, 2, 131000, d, seed=80 + d)
    err = parity.check_sampled(q, k, v, 1 / math.sqrt(d), n_rows=96, seed=d)
    print(d, err)


def _sweep_shapes():
    """24 seeded shapes: odd lengths, both head sizes, both signs of scale, and
    half of them with a unit count (B*H*ceil(N/256)) whose leftover after the
    whole rounds on 152 SMs is 1-76 units, so that CTA pairs share the last
    round (with 4 or more key blocks)."""
    rng = np.random.default_rng(2024)
    shapes = []
    while len(shapes) < 24:
        d = int(rng.choice([64, 128]))
        scale = float(rng.uniform(0.02, 0.2) * rng.choice([-1, 1]))
        if len(shapes) % 2 == 0:
            N = int(rng.integers(1, 3000))
            B, H = int(rng.integers(1, 4)), int(rng.integers(1, 24))
        else:
            N = int(rng.integers(513, 2600))            # 3-11 units per head, >= 5 key blocks
            qb = (N + 255) // 256
            target = 152 * int(rng.integers(1, 3)) + int(rng.integers(1, 77))
            H = max(1, target // qb)
            B = 1
        shapes.append((B, H, N, d, scale))
    return shapes


@pytest.mark.parametrize("B,H,N,d,scale", _sweep_shapes())
def test_seeded_shape_sweep(B, H, N, d, scale):
    q, k, v = inputs.make_random(B, H, N, d, seed=B * 7919 + H * 104729 + N * 13 + d)
    err = parity.check_sampled(q, k, v, scale, n_rows=48, seed=N, two_x_rule=N >= 64)
    print(B, H, N, d, scale, fa.fa_fwd_launch_shape(B, H, N, d), err["o_max"], err["lse_max"])


def test_launch_shapes_of_the_workloads():
    """The launch the benchmark workloads get on a 152-SM GB300: the 4096-row
    shape (512 units) and the spiky 32k shape (2048 units) share their last
    round in CTA pairs; the 8k prefill (1024 units, 112 left over) and the
    1024-row d = 64 shape (256 units, 104 left over) run every unit whole,
    since their leftovers are more than half the grid; the 256-row shape
    runs 16 units; 40 heads of 1024 rows (160 units) share 8."""
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the expected shapes are those of a 152-SM device")
    assert fa.fa_fwd_launch_shape(2, 16, 4096, 128) == (152, 2, 456)
    assert fa.fa_fwd_launch_shape(1, 16, 32768, 128) == (152, 2, 1976)
    assert fa.fa_fwd_launch_shape(1, 32, 8192, 128) == (152, 1, 1024)
    assert fa.fa_fwd_launch_shape(4, 16, 1024, 64) == (152, 1, 256)
    assert fa.fa_fwd_launch_shape(1, 16, 256, 64) == (16, 1, 16)
    assert fa.fa_fwd_launch_shape(1, 40, 1024, 128) == (152, 2, 152)


def test_split_units_with_ragged_keys_and_negative_scale():
    """Split units where the second half ends in a ragged key block, with a
    negative scale (the scores negated on the tensor core)."""
    q, k, v = inputs.make_random(2, 3, 777, 128, seed=53)
    err, _, _ = parity.check_full(q, k, v, -0.07)
    print(err)
