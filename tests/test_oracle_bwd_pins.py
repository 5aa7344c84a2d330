"""The backward oracle against what the mathematics fixes (CPU only)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from tests import oracle_bwd_pins as pins


def _recompute(Q, K, V, dO, s):
    """The recomputation form fed with the forward oracle's exact O and LSE."""
    O, L = oracle.attention(Q, K, V, s)
    return oracle.attention_bwd_recompute(Q, K, V, O, dO, L, s)


@pytest.mark.parametrize("impl", [oracle.attention_bwd, _recompute], ids=["definition", "recompute"])
@pytest.mark.parametrize("pin", pins.ALL_BWD_PINS, ids=lambda p: p.__name__)
def test_bwd_pins(impl, pin):
    pin(impl)


def test_heads_matches_full():
    r = np.random.default_rng(40)
    Q, K, V, dO = (r.standard_normal((2, 3, 70, 16)) for _ in range(4))
    full = oracle.attention_bwd(Q, K, V, dO, 0.25)
    heads = [(1, 2), (0, 0), (1, 0)]
    for (b, h), got in zip(heads, oracle.attention_bwd_heads(Q, K, V, dO, 0.25, heads)):
        for X, g in zip(full, got):
            np.testing.assert_array_equal(X[b, h], g)


def test_row_chunking_does_not_change_result():
    r = np.random.default_rng(41)
    Q, K, V, dO = (r.standard_normal((1, 2, 300, 8)) for _ in range(4))
    a = oracle.attention_bwd(Q, K, V, dO, 0.4, row_chunk=4096)
    b = oracle.attention_bwd(Q, K, V, dO, 0.4, row_chunk=64)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-13)
    O, L = oracle.attention(Q, K, V, 0.4)
    c = oracle.attention_bwd_recompute(Q, K, V, O, dO, L, 0.4, row_chunk=64)
    for x, y in zip(a, c):
        np.testing.assert_allclose(x, y, rtol=1e-11, atol=1e-12)


def test_recompute_uses_the_stored_o_and_lse():
    """The recomputation form reads D from O and P from LSE: feeding it a
    shifted LSE scales every P by e^{-c}, so dV scales by e^{-c}."""
    r = np.random.default_rng(42)
    Q, K, V, dO = (r.standard_normal((1, 1, 20, 4)) for _ in range(4))
    O, L = oracle.attention(Q, K, V, 0.5)
    _, _, dV0 = oracle.attention_bwd_recompute(Q, K, V, O, dO, L, 0.5)
    _, _, dV1 = oracle.attention_bwd_recompute(Q, K, V, O, dO, L + 0.7, 0.5)
    np.testing.assert_allclose(dV1, dV0 * np.exp(-0.7), rtol=1e-12, atol=1e-14)


# --- the bf16 materialise-path backward ---------------------------------------
def test_naive_bf16_bwd_n1_exact():
    """N = 1: P = 1 exactly, so dV = dO (bf16 inputs) and dQ = dK = 0 exactly."""
    r = np.random.default_rng(43)
    Q, K, V, dO = (oracle.bf16_round(r.standard_normal((1, 2, 1, 16))).astype(np.float64) for _ in range(4))
    dQ, dK, dV = oracle.naive_bf16_attention_bwd(Q, K, V, dO, 0.3)
    np.testing.assert_array_equal(dV, dO)
    assert not dQ.any() and not dK.any()


def test_naive_bf16_bwd_error_is_bf16_sized():
    r = np.random.default_rng(44)
    Q, K, V, dO = (oracle.bf16_round(r.standard_normal((1, 2, 256, 64))).astype(np.float64) for _ in range(4))
    exact = oracle.attention_bwd(Q, K, V, dO, 0.125)
    naive = oracle.naive_bf16_attention_bwd(Q, K, V, dO, 0.125)
    for X, Y in zip(exact, naive):
        err = np.abs(X - Y).max()
        assert 1e-6 < err < 3e-2 * np.abs(X).max(), err


def test_naive_bf16_bwd_matches_torch_bf16_autograd():
    """The reference agrees with torch's bf16 CPU autograd of the materialise
    path element by element (rare one-ulp flips from float32 summation order)."""
    pins.pin_naive_bwd_torch_bf16_autograd(oracle.naive_bf16_attention_bwd)


def _naive_bwd_variant(change):
    """The bf16 materialise-path backward written out again with one planted
    change, for checking that the torch-autograd pin sees it."""
    def bwd(Q, K, V, dO, scale):
        s32 = np.float32(scale)
        rnd = oracle.bf16_round

        def one(q, k, v, do):
            S = rnd(rnd(q @ k.T) * s32)
            m = S.max(axis=1, keepdims=True)
            e = np.exp(S - m, dtype=np.float32)
            P32 = e / e.sum(axis=1, keepdims=True, dtype=np.float32)
            P = rnd(P32)
            dv = rnd(P.T @ do)
            dP = do @ v.T if change == "dp_not_rounded" else rnd(do @ v.T)
            Pb = P32 if change == "p_unrounded_in_softmax_grad" else P
            if change == "d_from_o":
                D = np.sum(do * rnd(P @ v), axis=1, keepdims=True, dtype=np.float32)
            else:
                D = np.sum(Pb * dP, axis=1, keepdims=True, dtype=np.float32)
            dS = rnd(Pb * (dP - D))
            if change != "scale_missing_from_ds":
                dS = rnd(dS * s32)
            return rnd(dS @ k), rnd(dS.T @ q), dv

        Qf, Kf, Vf, dOf = (np.asarray(x, dtype=np.float32) for x in (Q, K, V, dO))
        out = [np.empty(Qf.shape) for _ in range(3)]
        for b in range(Qf.shape[0]):
            for h in range(Qf.shape[1]):
                for X, g in zip(out, one(Qf[b, h], Kf[b, h], Vf[b, h], dOf[b, h])):
                    X[b, h] = g
        return out
    return bwd


def test_naive_bwd_variant_without_change_passes():
    pins.pin_naive_bwd_torch_bf16_autograd(_naive_bwd_variant(None))


@pytest.mark.parametrize("change", ["scale_missing_from_ds", "dp_not_rounded", "d_from_o",
                                    "p_unrounded_in_softmax_grad"])
def test_planted_naive_bwd_mistake_is_caught(change):
    with pytest.raises(AssertionError):
        pins.pin_naive_bwd_torch_bf16_autograd(_naive_bwd_variant(change))


def test_naive_bf16_bwd_heads_matches_full():
    r = np.random.default_rng(45)
    Q, K, V, dO = (oracle.bf16_round(r.standard_normal((2, 2, 40, 8))).astype(np.float64) for _ in range(4))
    full = oracle.naive_bf16_attention_bwd(Q, K, V, dO, 0.3)
    for (b, h), got in zip([(1, 1), (0, 1)], oracle.naive_bf16_attention_bwd(Q, K, V, dO, 0.3, heads=[(1, 1), (0, 1)])):
        for X, g in zip(full, got):
            np.testing.assert_array_equal(X[b, h], g)


# --- planted mistakes fail at least one pin -----------------------------------
def _mutants():
    def per_head(fn):
        def bwd(Q, K, V, dO, s):
            out = [np.empty_like(Q), np.empty_like(K), np.empty_like(V)]
            for b in range(Q.shape[0]):
                for h in range(Q.shape[1]):
                    S = s * Q[b, h] @ K[b, h].T
                    P, _, _ = oracle.safe_softmax(S)
                    for X, g in zip(out, fn(Q[b, h], K[b, h], V[b, h], dO[b, h], s, P)):
                        X[b, h] = g
            return out
        bwd.__name__ = fn.__name__
        return bwd

    @per_head
    def dropped_d(q, k, v, do, s, P):
        dS = P * (do @ v.T)
        return s * dS @ k, s * dS.T @ q, P.T @ do

    @per_head
    def transposed_p(q, k, v, do, s, P):
        dP = do @ v.T
        dS = P * (dP - np.sum(P * dP, 1)[:, None])
        return s * dS @ k, s * dS.T @ q, P @ do

    @per_head
    def unscaled_dq(q, k, v, do, s, P):
        dP = do @ v.T
        dS = P * (dP - np.sum(P * dP, 1)[:, None])
        return dS @ k, s * dS.T @ q, P.T @ do

    @per_head
    def dk_without_transpose(q, k, v, do, s, P):
        dP = do @ v.T
        dS = P * (dP - np.sum(P * dP, 1)[:, None])
        return s * dS @ k, s * dS @ q, P.T @ do

    @per_head
    def sign_flip(q, k, v, do, s, P):
        dP = do @ v.T
        dS = P * (np.sum(P * dP, 1)[:, None] - dP)
        return s * dS @ k, s * dS.T @ q, P.T @ do

    @per_head
    def d_over_columns(q, k, v, do, s, P):
        dP = do @ v.T
        dS = P * (dP - np.sum(P * dP, 0)[None, :])
        return s * dS @ k, s * dS.T @ q, P.T @ do

    return [dropped_d, transposed_p, unscaled_dq, dk_without_transpose, sign_flip, d_over_columns]


@pytest.mark.parametrize("mutant", _mutants(), ids=lambda f: f.__name__)
def test_planted_bwd_mistake_is_caught(mutant):
    caught = []
    for pin in pins.ALL_BWD_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mutant)
        except (AssertionError, FloatingPointError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught {mutant.__name__}"
