"""The shared-K/V-head and split-key oracle against facts that do not come from it (CPU only)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle


def _rand(seed, *shape, s=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * s


# --- pins of attention_gqa ---------------------------------------------------------
def pin_gqa_reduces_to_plain(fn):
    """H_kv = H is the plain (pinned) definition."""
    Q, K, V = _rand(1, 2, 3, 17, 8), _rand(2, 2, 3, 23, 8), _rand(3, 2, 3, 23, 8)
    O, L = fn(Q, K, V, 0.4)
    O2, L2 = oracle.attention(Q, K, V, 0.4)
    np.testing.assert_allclose(O, O2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(L, L2, rtol=1e-13, atol=1e-14)


def pin_gqa_library(fn):
    """torch float64 SDPA with each K/V head repeated for its G query heads."""
    for (B, H, Hkv, Nq, Nkv, d, s) in [(1, 8, 2, 5, 33, 16, 0.25), (2, 6, 3, 1, 70, 8, 0.5), (1, 4, 1, 9, 9, 4, 0.0)]:
        Q, K, V = _rand(4, B, H, Nq, d, s=2), _rand(5, B, Hkv, Nkv, d, s=2), _rand(6, B, Hkv, Nkv, d)
        O, L = fn(Q, K, V, s)
        G = H // Hkv
        tk = torch.from_numpy(K).repeat_interleave(G, dim=1)
        tv = torch.from_numpy(V).repeat_interleave(G, dim=1)
        tq = torch.from_numpy(Q)
        Ot = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=s)
        Lt = torch.logsumexp(s * (tq @ tk.transpose(-1, -2)), dim=-1)
        np.testing.assert_allclose(O, Ot.numpy(), rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(L, Lt.numpy(), rtol=1e-12, atol=1e-12)


def pin_gqa_groups_independent(fn):
    """Changing K/V head 1 changes only query heads 2 and 3 (G = 2); heads of
    one group with equal queries give equal outputs."""
    Q, K, V = _rand(7, 1, 4, 6, 5), _rand(8, 1, 2, 11, 5), _rand(9, 1, 2, 11, 5)
    Q[0, 1] = Q[0, 0]
    O, _ = fn(Q, K, V, 0.7)
    K2, V2 = K.copy(), V.copy()
    K2[0, 1] += 1.0
    V2[0, 1] *= -1.0
    O2, _ = fn(Q, K2, V2, 0.7)
    np.testing.assert_array_equal(O[0, :2], O2[0, :2])
    assert np.abs(O[0, 2:] - O2[0, 2:]).min() > 0
    np.testing.assert_array_equal(O[0, 0], O[0, 1])


GQA_PINS = [pin_gqa_reduces_to_plain, pin_gqa_library, pin_gqa_groups_independent]


@pytest.mark.parametrize("pin", GQA_PINS, ids=lambda p: p.__name__)
def test_gqa_pins(pin):
    pin(oracle.attention_gqa)


def test_gqa_rows_matches_full():
    Q, K, V = _rand(10, 2, 6, 4, 8), _rand(11, 2, 3, 19, 8), _rand(12, 2, 3, 19, 8)
    O, L = oracle.attention_gqa(Q, K, V, 0.3)
    for (b, h), (o, l) in zip([(1, 5), (0, 2)], oracle.attention_gqa_rows(Q, K, V, 0.3, [(1, 5), (0, 2)])):
        np.testing.assert_array_equal(O[b, h], o)
        np.testing.assert_array_equal(L[b, h], l)


# --- pins of the merge ----------------------------------------------------------------
def pin_merge_partition(merge):
    """Merging attention over the parts of any partition of the keys gives the
    attention over all keys (the online-softmax combination of two states)."""
    rng = np.random.default_rng(13)
    Q, K, V = _rand(14, 1, 2, 7, 6, s=3), _rand(15, 1, 2, 50, 6, s=3), _rand(16, 1, 2, 50, 6)
    O_full, L_full = oracle.attention(Q, K, V, 0.5)
    for bounds in ([0, 50], [0, 1, 50], [0, 25, 50], [0, 3, 4, 17, 49, 50], [0] + sorted(rng.choice(np.arange(1, 50), 9, replace=False).tolist()) + [50]):
        parts = [oracle.attention(Q, K[:, :, a:b], V[:, :, a:b], 0.5) for a, b in zip(bounds[:-1], bounds[1:])]
        O, L = merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        np.testing.assert_allclose(O, O_full, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(L, L_full, rtol=1e-13, atol=1e-13)


def pin_merge_closed_form(merge):
    """Two parts: LSE = logaddexp(L1, L2), O = sigmoid(L1 - L2) O1 + sigmoid(L2 - L1) O2;
    very large LSEs do not overflow."""
    O1, O2 = _rand(17, 3, 4), _rand(18, 3, 4)
    for L1, L2 in [(np.array([0.1, -2.0, 5.0]), np.array([0.3, 1.0, -5.0])),
                   (np.array([800.0, -900.0, 1e4]), np.array([799.0, -901.0, 1e4 + 1]))]:
        O, L = merge(np.stack([O1, O2]), np.stack([L1, L2]))
        np.testing.assert_allclose(L, np.logaddexp(L1, L2), rtol=1e-14, atol=1e-12)
        w1 = 1.0 / (1.0 + np.exp(L2 - L1))
        np.testing.assert_allclose(O, w1[:, None] * O1 + (1 - w1)[:, None] * O2, rtol=1e-13, atol=1e-14)


MERGE_PINS = [pin_merge_partition, pin_merge_closed_form]


@pytest.mark.parametrize("pin", MERGE_PINS, ids=lambda p: p.__name__)
def test_merge_pins(pin):
    pin(oracle.merge_partials)


def test_attention_split_equals_whole():
    Q, K, V = _rand(19, 2, 8, 3, 16), _rand(20, 2, 2, 300, 16), _rand(21, 2, 2, 300, 16)
    O, L = oracle.attention_gqa(Q, K, V, 0.25)
    for bounds in ([0, 128, 256, 300], [0, 300], [0, 1, 299, 300]):
        O2, L2 = oracle.attention_split(Q, K, V, 0.25, bounds)
        np.testing.assert_allclose(O2, O, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(L2, L, rtol=1e-13, atol=1e-13)


# --- planted mistakes -----------------------------------------------------------------
def _gqa_mutants():
    from oracle.attention import _attention_one_head

    def modulo_grouping(Q, K, V, s):   # h % H_kv instead of h // G
        B, H, Nq, _ = Q.shape
        Hkv = K.shape[1]
        O = np.empty((B, H, Nq, V.shape[-1])); L = np.empty((B, H, Nq))
        for b in range(B):
            for h in range(H):
                O[b, h], L[b, h] = _attention_one_head(Q[b, h], K[b, h % Hkv], V[b, h % Hkv], s)
        return O, L

    def shared_first_head(Q, K, V, s):
        B, H, Nq, _ = Q.shape
        O = np.empty((B, H, Nq, V.shape[-1])); L = np.empty((B, H, Nq))
        for b in range(B):
            for h in range(H):
                O[b, h], L[b, h] = _attention_one_head(Q[b, h], K[b, 0], V[b, 0], s)
        return O, L

    return [modulo_grouping, shared_first_head]


def _merge_mutants():
    def unweighted(Op, Lp):
        return Op.mean(axis=0), np.log(np.exp(Lp).sum(axis=0))

    def no_max(Op, Lp):
        w = np.exp(Lp)
        return np.einsum("s...,s...d->...d", w / w.sum(axis=0), Op), np.log(w.sum(axis=0))

    def max_instead_of_sum(Op, Lp):
        i = Lp.argmax(axis=0)
        return np.take_along_axis(Op, i[None, ..., None], axis=0)[0], Lp.max(axis=0)

    return [unweighted, no_max, max_instead_of_sum]


@pytest.mark.parametrize("mutant", _gqa_mutants(), ids=lambda f: f.__name__)
def test_planted_gqa_mistake_is_caught(mutant):
    caught = []
    for pin in GQA_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught


@pytest.mark.parametrize("mutant", _merge_mutants(), ids=lambda f: f.__name__)
def test_planted_merge_mistake_is_caught(mutant):
    caught = []
    for pin in MERGE_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mutant)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught
