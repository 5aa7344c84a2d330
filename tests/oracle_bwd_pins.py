"""Checks that pin the backward oracle to facts that do not come from it.

Each ``pin_*`` takes a backward implementation ``bwd(Q, K, V, dO, scale) ->
(dQ, dK, dV)`` (float64 numpy, [B,H,N,d]) and raises AssertionError when it
disagrees with: central finite differences of the forward oracle (itself
pinned to closed forms and 50-digit arithmetic), torch's float64 autograd of
scaled_dot_product_attention, the closed forms for N = 1 and for equal keys,
or the column sums that the softmax rows summing to one force. The same
pins are run on deliberately broken backwards in ``test_oracle_bwd_pins.py``.
"""
from __future__ import annotations

import numpy as np

import oracle


def _rng(seed):
    return np.random.default_rng(seed)


def _loss(Q, K, V, dO, s):
    O, _ = oracle.attention(Q, K, V, s)
    return float(np.sum(O * dO))


def pin_bwd_finite_difference(bwd):
    """Every gradient entry against a central difference of <dO, O(Q, K, V)>."""
    r = _rng(31)
    h = 1e-5
    for (N, d, s) in [(1, 2, 0.7), (2, 1, 1.3), (3, 2, 0.5), (5, 3, 0.9), (4, 4, 0.0)]:
        Q, K, V, dO = (r.standard_normal((1, 2, N, d)) for _ in range(4))
        grads = bwd(Q, K, V, dO, s)
        for X, G in zip((Q, K, V), grads):
            for idx in np.ndindex(X.shape):
                old = X[idx]
                X[idx] = old + h
                fp = _loss(Q, K, V, dO, s)
                X[idx] = old - h
                fm = _loss(Q, K, V, dO, s)
                X[idx] = old
                fd = (fp - fm) / (2 * h)
                assert abs(G[idx] - fd) <= 1e-7 * max(1.0, abs(fd)), (N, d, s, idx, G[idx], fd)


def pin_bwd_n1(bwd):
    """N = 1: P = 1 whatever the scores, so dV = dO and dQ = dK = 0."""
    r = _rng(32)
    Q, K, V, dO = (r.standard_normal((2, 3, 1, 8)) for _ in range(4))
    dQ, dK, dV = bwd(Q, K, V, dO, 0.4)
    np.testing.assert_allclose(dV, dO, rtol=0, atol=1e-14)
    np.testing.assert_allclose(dQ, 0.0, rtol=0, atol=1e-14)
    np.testing.assert_allclose(dK, 0.0, rtol=0, atol=1e-14)


def pin_bwd_equal_keys(bwd):
    """All keys equal: P is uniform (1/N), so dV_j = (1/N) sum_i dO_i for every
    j, dQ = 0 (no score depends on q), and
    dK_j = (scale/N) sum_i (dO_i . (v_j - mean(v))) q_i."""
    r = _rng(33)
    N, d, s = 7, 5, 0.6
    Q, V, dO = (r.standard_normal((1, 1, N, d)) for _ in range(3))
    K = np.broadcast_to(r.standard_normal(d), (1, 1, N, d)).copy()
    dQ, dK, dV = bwd(Q, K, V, dO, s)
    np.testing.assert_allclose(dV[0, 0], np.broadcast_to(dO[0, 0].sum(0) / N, (N, d)), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dQ, 0.0, rtol=0, atol=1e-13)
    vbar = V[0, 0].mean(0)
    expect = np.stack([(s / N) * ((dO[0, 0] @ (V[0, 0, j] - vbar))[:, None] * Q[0, 0]).sum(0) for j in range(N)])
    np.testing.assert_allclose(dK[0, 0], expect, rtol=1e-12, atol=1e-13)


def pin_bwd_column_sums(bwd):
    """Rows of P sum to one: sum_j dK_j = 0 (shifting every key by one vector
    leaves the softmax unchanged) and sum_j dV_j = sum_i dO_i."""
    r = _rng(34)
    Q, K, V, dO = (r.standard_normal((2, 2, 37, 16)) * 1.5 for _ in range(4))
    dQ, dK, dV = bwd(Q, K, V, dO, 0.3)
    np.testing.assert_allclose(dK.sum(axis=2), 0.0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dV.sum(axis=2), dO.sum(axis=2), rtol=1e-12, atol=1e-12)


def pin_bwd_library_autograd(bwd):
    """Agreement with torch float64 autograd of scaled_dot_product_attention."""
    import torch
    r = _rng(35)
    for (B, H, N, d, s) in [(1, 1, 1, 3, 0.3), (2, 3, 45, 16, 0.25), (1, 2, 130, 64, 0.125), (1, 1, 9, 2, 0.0)]:
        Q, K, V, dO = (r.standard_normal((B, H, N, d)) * 2 for _ in range(4))
        tq, tk, tv = (torch.from_numpy(x.copy()).requires_grad_(True) for x in (Q, K, V))
        out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=s)
        out.backward(torch.from_numpy(dO))
        dQ, dK, dV = bwd(Q, K, V, dO, s)
        for mine, t in ((dQ, tq), (dK, tk), (dV, tv)):
            np.testing.assert_allclose(mine, t.grad.numpy(), rtol=1e-10, atol=1e-11)


ALL_BWD_PINS = [pin_bwd_finite_difference, pin_bwd_n1, pin_bwd_equal_keys, pin_bwd_column_sums,
                pin_bwd_library_autograd]


# --- the bf16 materialise-path backward (the "twice the baseline" reference) ----
def _torch_bf16_autograd(q, k, v, do, s):
    """torch's own bf16 CPU autograd of standard attention: S = q k^T (bf16),
    S * scale (bf16), a bf16 softmax (float32 inside, bf16 out), O = P v (bf16),
    then O.backward(dO). Returns (dQ, dK, dV) as float64 numpy."""
    import torch
    tq, tk, tv = (x.clone().requires_grad_(True) for x in (q, k, v))
    O = torch.softmax((tq @ tk.transpose(-1, -2)) * s, dim=-1) @ tv
    O.backward(do)
    return tuple(t.grad.float().numpy().astype(np.float64) for t in (tq, tk, tv))


def pin_naive_bwd_torch_bf16_autograd(naive_bwd):
    """``naive_bwd(Q, K, V, dO, scale)`` against torch's bf16 autograd of the
    materialise path, element by element. Both store the same intermediates in
    bf16 and sum in float32, so almost every element is identical; a float32
    summation order that differs flips a bf16 rounding now and then (one ulp of
    P, dS or a gradient element, seen large only where dQ cancels to near zero).
    So: at least 98% identical elements, and every element within 2^-6 of its
    own size plus 2^-9 of the gradient's largest element."""
    import torch
    g = torch.Generator().manual_seed(46)
    for (B, H, N, d, s) in [(1, 2, 96, 64, 0.125), (1, 1, 200, 32, 0.3), (2, 1, 130, 16, 1.7)]:
        q, k, v, do = (torch.randn(B, H, N, d, generator=g).to(torch.bfloat16) for _ in range(4))
        want = _torch_bf16_autograd(q, k, v, do, s)
        got = naive_bwd(*(x.float().numpy().astype(np.float64) for x in (q, k, v, do)), s)
        for name, T, M in zip(("dQ", "dK", "dV"), want, got):
            same = float(np.mean(T == M))
            assert same >= 0.98, (name, N, d, s, same)
            bound = 2.0 ** -6 * np.abs(T) + 2.0 ** -9 * np.abs(T).max()
            assert np.all(np.abs(T - M) <= bound), (name, N, d, s, float(np.abs(T - M).max()))
