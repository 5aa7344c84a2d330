"""The standard-attention comparator (S and P materialised in HBM) vs the oracle
(needs a GB300)."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_34_gb300 import fa, inputs
from tests import parity

pytestmark = pytest.mark.gpu


def emulated_lse(Q, K, scale):
    """LSE of the bf16 score matrix as the materialise path computes it."""
    out = np.empty(Q.shape[:3])
    for b in range(Q.shape[0]):
        for h in range(Q.shape[1]):
            S = oracle.bf16_round(oracle.bf16_round(Q[b, h].astype(np.float32) @ K[b, h].astype(np.float32).T)
                                  * np.float32(scale)).astype(np.float64)
            m = S.max(axis=1)
            out[b, h] = m + np.log(np.exp(S - m[:, None]).sum(axis=1))
    return out


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [7, 128, 129, 300, 1000])
def test_naive_matches_bf16_emulation(N, d):
    q, k, v = inputs.make_random(2, 3, N, d, seed=40 + N + d)
    s = 1 / math.sqrt(d)
    o, lse = fa.fa_naive_fwd(q.cuda(), k.cuda(), v.cuda(), scale=s)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status()[0] == fa.FA_OK
    Q, K, V = (parity.to64(x) for x in (q, k, v))
    On = oracle.naive_bf16_attention(Q, K, V, s)
    og = parity.to64(o.cpu())
    O_ref, L_ref = oracle.attention(Q, K, V, s)
    d_emul = np.abs(og - On)
    err_gpu = np.abs(og - O_ref).max()
    err_emul = np.abs(On - O_ref).max()
    lse_diff = np.abs(parity.to64(lse.cpu()) - emulated_lse(Q, K, s)).max()
    print(f"N={N} d={d}: max|O-emul| {d_emul.max():.2e}, equal {np.mean(d_emul == 0):.3f}, "
          f"err vs fp64 {err_gpu:.2e} (emulation {err_emul:.2e}), max|LSE-emul| {lse_diff:.2e}")
    # The tensor-core fp32 sums may differ from numpy's in the last bit; a flipped
    # bf16 rounding of one score moves that key's weight by about 2^-8, so O may
    # differ from the emulation by a few bf16 ulps where that key dominates.
    assert np.mean(d_emul == 0) > 0.8
    assert d_emul.max() <= 1e-2
    assert lse_diff <= 5e-3
    # and it is attention, with the materialise path's own accuracy
    assert err_gpu <= 1.5 * err_emul + 2e-3
    assert np.linalg.norm(og - O_ref) / np.linalg.norm(O_ref) <= 2e-2


def test_naive_prefill_head_sampled():
    """The 8k prefill workload (first 2 heads) on the comparator, sampled rows vs the emulation."""
    w = inputs.workload("prefill8k_d128_h32")
    q, k, v, s = inputs.make_inputs(w)
    q, k, v = (x[:, :2].contiguous() for x in (q, k, v))
    o, lse = fa.fa_naive_fwd(q.cuda(), k.cuda(), v.cuda(), scale=s)
    torch.cuda.synchronize()
    rows = parity.sample_rows(1, 2, w.N, 64, seed=3)
    On = oracle.naive_bf16_attention(parity.to64(q), parity.to64(k), parity.to64(v), s, rows)
    og = parity.to64(o.cpu())[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert np.abs(og - On).max() <= 2 * np.abs(On).max() * 2 ** -7
    O_ref, L_ref = oracle.attention_rows(parity.to64(q), parity.to64(k), parity.to64(v), s, rows)
    assert np.abs(og - O_ref).max() < 5e-2


def test_naive_rejects_small_workspace():
    q = torch.zeros(1, 1, 256, 64, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(fa.fa_naive_workspace_bytes(1, 1, 256) - 128, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError) as ei:
        fa.fa_naive_fwd(q, q.clone(), q.clone(), workspace=ws)
    assert ei.value.status == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("d", [64, 128])
def test_naive_negative_scale(d):
    """scale < 0: the comparator's scores are bf16(scale * bf16(Q K^T)) with the
    sign carried through; the result is attention with the materialise path's
    accuracy."""
    q, k, v = inputs.make_random(1, 3, 400, d, seed=70 + d)
    s = -1 / math.sqrt(d)
    o, lse = fa.fa_naive_fwd(q.cuda(), k.cuda(), v.cuda(), scale=s)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status()[0] == fa.FA_OK
    Q, K, V = (parity.to64(x) for x in (q, k, v))
    On = oracle.naive_bf16_attention(Q, K, V, s)
    O_ref, _ = oracle.attention(Q, K, V, s)
    og = parity.to64(o.cpu())
    assert np.abs(og - On).max() <= 1e-2
    assert np.abs(og - O_ref).max() <= 1.5 * np.abs(On - O_ref).max() + 2e-3
    assert np.abs(parity.to64(lse.cpu()) - emulated_lse(Q, K, s)).max() <= 5e-3
