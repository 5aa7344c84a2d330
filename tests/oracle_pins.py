"""Checks that pin the CPU oracle to what the pages and mathematics fix.

Each ``pin_*`` takes an attention implementation ``attn(Q, K, V, scale) ->
(O, LSE)`` (float64 numpy, [B,H,N,d] and [B,H,N]) and raises AssertionError
when it disagrees with a fact that does not come from the oracle itself:
closed forms, high-precision brute force, invariants of the safe softmax
("Flash Attention (FA1)", naive attention analysis: subtracting the row max
does not change the result), or a library routine. The same pins are run on
deliberately broken implementations in ``test_oracle_pins.py`` to show that
a plausible mistake fails at least one of them.
"""
from __future__ import annotations

import math

import numpy as np


def _rng(seed):
    return np.random.default_rng(seed)


def pin_n1(attn):
    """N = 1: the softmax of one score is 1, so O = V_0 and LSE = scale * q.k."""
    r = _rng(1)
    for d in (1, 3, 64):
        Q, K, V = (r.standard_normal((2, 3, 1, d)) for _ in range(3))
        s = 0.37
        O, L = attn(Q, K, V, s)
        np.testing.assert_allclose(O, V, rtol=0, atol=1e-13)
        expect = s * np.einsum("bhnd,bhnd->bhn", Q, K)
        np.testing.assert_allclose(L, expect, rtol=0, atol=1e-13)


def pin_n2_logistic(attn):
    """N = 2: weights are the logistic function of the score difference."""
    r = _rng(2)
    for trial in range(20):
        d = int(r.integers(1, 5))
        q = r.standard_normal(d) * 2
        k = r.standard_normal((2, d)) * 2
        v = r.standard_normal((2, d))
        s = float(r.uniform(0.1, 2.0))
        s0 = s * math.fsum(q[i] * k[0, i] for i in range(d))
        s1 = s * math.fsum(q[i] * k[1, i] for i in range(d))
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        w1 = 1.0 / (1.0 + math.exp(s0 - s1))
        o = w0 * v[0] + w1 * v[1]
        lse = max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1)))
        O, L = attn(q.reshape(1, 1, 1, d), k.reshape(1, 1, 2, d), v.reshape(1, 1, 2, d), s)
        np.testing.assert_allclose(O[0, 0, 0], o, rtol=1e-12, atol=1e-13)
        assert abs(L[0, 0, 0] - lse) <= 1e-12 * max(1.0, abs(lse))


def pin_bruteforce_mp(attn):
    """Tiny inputs (N <= 4, d <= 2) against 50-digit arithmetic."""
    import mpmath
    mpmath.mp.dps = 50
    r = _rng(3)
    for trial in range(30):
        N = int(r.integers(1, 5))
        d = int(r.integers(1, 3))
        Q = r.standard_normal((1, 2, N, d)) * 3
        K = r.standard_normal((1, 2, N, d)) * 3
        V = r.standard_normal((1, 2, N, d))
        s = float(r.uniform(0.05, 1.5))
        O, L = attn(Q, K, V, s)
        for h in range(2):
            for i in range(N):
                sc = [mpmath.mpf(s) * mpmath.fsum(mpmath.mpf(Q[0, h, i, t]) * mpmath.mpf(K[0, h, j, t])
                                                  for t in range(d)) for j in range(N)]
                z = mpmath.fsum(mpmath.e ** x for x in sc)
                for t in range(d):
                    o = mpmath.fsum(mpmath.e ** sc[j] * mpmath.mpf(V[0, h, j, t]) for j in range(N)) / z
                    assert abs(float(o) - O[0, h, i, t]) <= 1e-13 * max(1.0, abs(float(o))), (N, d, h, i, t)
                assert abs(float(mpmath.log(z)) - L[0, h, i]) <= 1e-13 * max(1.0, abs(float(mpmath.log(z))))


def pin_constant_v(attn):
    """Every row of V equal to v gives O = v whatever the weights are."""
    r = _rng(4)
    Q = r.standard_normal((2, 2, 37, 8)) * 4
    K = r.standard_normal((2, 2, 37, 8)) * 4
    v = r.standard_normal(8)
    V = np.broadcast_to(v, (2, 2, 37, 8)).copy()
    O, _ = attn(Q, K, V, 0.5)
    np.testing.assert_allclose(O, V, rtol=1e-13, atol=1e-13)


def pin_uniform(attn):
    """Q = 0 gives uniform weights: O = mean of V, LSE = ln N.
    Equal key rows give uniform weights too, with LSE = scale*q.k + ln N."""
    r = _rng(5)
    N, d = 29, 6
    V = r.standard_normal((1, 3, N, d))
    K = r.standard_normal((1, 3, N, d))
    O, L = attn(np.zeros((1, 3, N, d)), K, V, 0.9)
    np.testing.assert_allclose(O, np.broadcast_to(V.mean(axis=2, keepdims=True), O.shape), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L, np.full(L.shape, math.log(N)), rtol=0, atol=1e-13)
    Q = r.standard_normal((1, 3, N, d))
    krow = r.standard_normal(d)
    Ke = np.broadcast_to(krow, (1, 3, N, d)).copy()
    O, L = attn(Q, Ke, V, 0.9)
    np.testing.assert_allclose(O, np.broadcast_to(V.mean(axis=2, keepdims=True), O.shape), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L, 0.9 * (Q @ krow) + math.log(N), rtol=0, atol=1e-12)


def pin_shift_via_inputs(attn):
    """Adding c_r to every score of row r leaves O unchanged and moves LSE by c_r.
    Realised through the inputs: Q gets an extra column c_r/scale, K an extra column of ones."""
    r = _rng(6)
    B, H, N, d = 1, 2, 23, 5
    Q, K, V = (r.standard_normal((B, H, N, d)) for _ in range(3))
    s = 0.7
    c = r.uniform(-30, 30, size=(B, H, N))
    Q2 = np.concatenate([Q, (c / s)[..., None]], axis=-1)
    K2 = np.concatenate([K, np.ones((B, H, N, 1))], axis=-1)
    O1, L1 = attn(Q, K, V, s)
    O2, L2 = attn(Q2, K2, V, s)
    np.testing.assert_allclose(O2, O1, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(L2, L1 + c, rtol=1e-12, atol=1e-11)


def pin_permutations(attn):
    """Jointly permuting key/value rows leaves O unchanged; permuting queries permutes O."""
    r = _rng(7)
    B, H, N, d = 2, 2, 31, 4
    Q, K, V = (r.standard_normal((B, H, N, d)) for _ in range(3))
    O, L = attn(Q, K, V, 0.6)
    p = r.permutation(N)
    O2, L2 = attn(Q, K[:, :, p], V[:, :, p], 0.6)
    np.testing.assert_allclose(O2, O, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L2, L, rtol=1e-13, atol=1e-13)
    O3, L3 = attn(Q[:, :, p], K, V, 0.6)
    np.testing.assert_allclose(O3, O[:, :, p], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(L3, L[:, :, p], rtol=1e-13, atol=1e-14)
    # heads and batches are independent problems
    O4, _ = attn(Q[:, ::-1], K[:, ::-1], V[:, ::-1], 0.6)
    np.testing.assert_allclose(O4, O[:, ::-1], rtol=1e-13, atol=1e-14)


def pin_linear_in_v(attn):
    """O is linear in V for fixed Q and K."""
    r = _rng(8)
    Q, K, V1, V2 = (r.standard_normal((1, 2, 19, 7)) for _ in range(4))
    a, b = 1.75, -0.4
    O1, _ = attn(Q, K, V1, 0.8)
    O2, _ = attn(Q, K, V2, 0.8)
    O12, _ = attn(Q, K, a * V1 + b * V2, 0.8)
    np.testing.assert_allclose(O12, a * O1 + b * O2, rtol=1e-11, atol=1e-12)


def pin_hardmax(attn):
    """A very large scale with a unique row maximum puts all weight on it."""
    r = _rng(9)
    N, d = 17, 6
    Q, K, V = (r.standard_normal((1, 1, N, d)) for _ in range(3))
    s = 1e4
    O, L = attn(Q, K, V, s)
    S = Q[0, 0] @ K[0, 0].T
    j = S.argmax(axis=1)
    gap = np.sort(S, axis=1)[:, -1] - np.sort(S, axis=1)[:, -2]
    assert np.all(gap * s > 50), "test data needs a clear maximum"
    np.testing.assert_allclose(O[0, 0], V[0, 0][j], rtol=0, atol=1e-12)
    np.testing.assert_allclose(L[0, 0], s * S.max(axis=1), rtol=1e-14, atol=0)


def pin_library_sdpa(attn):
    """Agreement with torch's scaled_dot_product_attention and logsumexp in float64 (CPU)."""
    import torch
    r = _rng(10)
    for (B, H, N, d, s) in [(1, 1, 1, 3, 0.3), (2, 3, 45, 16, 0.25), (1, 2, 130, 64, 0.125), (1, 1, 9, 2, 0.0)]:
        Q = r.standard_normal((B, H, N, d)) * 2
        K = r.standard_normal((B, H, N, d)) * 2
        V = r.standard_normal((B, H, N, d))
        O, L = attn(Q, K, V, s)
        tq, tk, tv = (torch.from_numpy(x) for x in (Q, K, V))
        Ot = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=s)
        Lt = torch.logsumexp(s * (tq @ tk.transpose(-1, -2)), dim=-1)
        np.testing.assert_allclose(O, Ot.numpy(), rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(L, Lt.numpy(), rtol=1e-12, atol=1e-12)


ALL_PINS = [pin_n1, pin_n2_logistic, pin_bruteforce_mp, pin_constant_v, pin_uniform,
            pin_shift_via_inputs, pin_permutations, pin_linear_in_v, pin_hardmax, pin_library_sdpa]
