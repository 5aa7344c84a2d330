"""Device-side wait limits: a K/V tile that never arrives ends the kernel with a
timeout status instead of a hang, and the context stays usable (needs a GB300).

The failure is made without faulting the GPU: the test hook tells the
producer to skip one TMA load, so its consumer's wait runs out after a short
limit. Every role then stops, waits for its own copies and MMAs in flight,
frees tensor memory and returns.
"""
import math

import pytest
import torch

import oracle
from exact_io_aware_34_gb300 import fa, inputs
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("drop", [0, 1, 2, 5])
def test_dropped_load_times_out_cleanly(d, drop):
    B, H, N = 1, 2, 700
    q, k, v = inputs.make_random(B, H, N, d, seed=20 + drop)
    qd, kd, vd = (x.cuda() for x in (q, k, v))
    o = torch.zeros_like(qd)
    lse = torch.zeros(B, H, N, dtype=torch.float32, device="cuda")
    st = fa.fa_fwd_fault_test(qd, kd, vd, o, lse, 1 / math.sqrt(d), drop, 20_000_000)   # 20 ms
    assert st == fa.FA_OK
    st, info = fa.fa_get_device_status()
    assert st == fa.FA_ERR_TIMEOUT, (st, info)
    assert info[0] in (1, 2, 3)
    assert fa.fa_get_device_status()[0] == fa.FA_OK          # the status word was cleared
    # the context is still usable and the next call is correct
    s = 1 / math.sqrt(d)
    o2, lse2 = fa.fa_fwd(qd, kd, vd, scale=s)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status()[0] == fa.FA_OK
    O_ref, L_ref = oracle.attention(*(parity.to64(x) for x in (q, k, v)), s)
    err = parity.errors(o2.cpu(), lse2.cpu(), O_ref, L_ref)
    assert err["o_max"] <= parity.TOL_O_MAX and err["lse_max"] <= parity.TOL_LSE_MAX, err


def test_drop_beyond_last_load_is_harmless():
    q, k, v = (x.cuda() for x in inputs.make_random(1, 1, 256, 128, seed=30))
    o = torch.empty_like(q)
    lse = torch.empty(1, 1, 256, dtype=torch.float32, device="cuda")
    assert fa.fa_fwd_fault_test(q, k, v, o, lse, 0.1, 10_000, 20_000_000) == fa.FA_OK
    assert fa.fa_get_device_status()[0] == fa.FA_OK


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("drop", [0, 1, 3, 6])
def test_backward_dropped_load_times_out_cleanly(d, drop):
    """The same for fa_bwd: one K/V load of every dQ CTA and the Q/dO loads of
    one block in every dK/dV CTA never arrive; the launch ends with a timeout
    status, and the next backward call in the same context is correct."""
    B, H, N = 1, 2, 700
    s = 1 / math.sqrt(d)
    q, k, v = inputs.make_random(B, H, N, d, seed=40 + drop)
    do = inputs.make_grad(B, H, N, d, seed=40 + drop)
    o, lse = parity.oracle_forward_inputs(q, k, v, s)
    args = [x.cuda() for x in (q, k, v, o, do, lse)]
    grads = [torch.zeros_like(args[0]) for _ in range(3)]
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N), dtype=torch.uint8, device="cuda")
    st = fa.fa_bwd_fault_test(*args, *grads, s, ws, drop, 20_000_000)   # 20 ms
    assert st == fa.FA_OK
    st, info = fa.fa_get_device_status()
    assert st == fa.FA_ERR_TIMEOUT, (st, info)
    assert info[0] in (4, 5, 6, 7, 8, 9)
    assert fa.fa_get_device_status()[0] == fa.FA_OK
    got = parity.run_gpu_bwd(q, k, v, o, do, lse, s)
    ref = oracle.attention_bwd(*(parity.to64(x) for x in (q, k, v, do)), s)
    err = parity.bwd_errors(got, ref)
    parity.assert_bwd_within(err, two_x_rule=False)


def test_backward_fault_hook_rejects_zero_timeout():
    q, k, v = (x.cuda() for x in inputs.make_random(1, 1, 128, 64, seed=49))
    lse = torch.zeros(1, 1, 128, device="cuda")
    ws = torch.empty(fa.fa_bwd_workspace_bytes(1, 1, 128), dtype=torch.uint8, device="cuda")
    g = [torch.zeros_like(q) for _ in range(3)]
    assert fa.fa_bwd_fault_test(q, k, v, q.clone(), q.clone(), lse, *g, 0.125, ws, 0, 0) == fa.FA_ERR_INVALID_ARG


def test_dropped_load_in_a_split_unit_times_out_cleanly():
    """160 units (40 heads of 1024 rows): one whole round, then 8 units shared by
    CTA pairs. Load 20 of a CTA is a K/V tile of its shared unit, so that
    CTA's wait runs out, its partner's waits for the exchange run out too, and
    both still meet at the closing cluster barrier: the launch ends with a
    timeout status and the next call is correct."""
    B, H, N, d = 1, 40, 1024, 128
    q, k, v = inputs.make_random(B, H, N, d, seed=60)
    qd, kd, vd = (x.cuda() for x in (q, k, v))
    o = torch.zeros_like(qd)
    lse = torch.zeros(B, H, N, dtype=torch.float32, device="cuda")
    assert fa.fa_fwd_fault_test(qd, kd, vd, o, lse, 1 / math.sqrt(d), 20, 20_000_000) == fa.FA_OK
    st, info = fa.fa_get_device_status()
    assert st == fa.FA_ERR_TIMEOUT, (st, info)
    assert info[0] in (1, 2, 3)
    s = 1 / math.sqrt(d)
    o2, lse2 = fa.fa_fwd(qd, kd, vd, scale=s)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status()[0] == fa.FA_OK
    O_ref, L_ref = oracle.attention(*(parity.to64(x) for x in (q, k, v)), s)
    err = parity.errors(o2.cpu(), lse2.cpu(), O_ref, L_ref)
    assert err["o_max"] <= parity.TOL_O_MAX and err["lse_max"] <= parity.TOL_LSE_MAX, err
