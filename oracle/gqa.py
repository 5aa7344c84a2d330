"""Oracle for shared key/value heads and split key ranges: plain, float64, CPU.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it. It shares no code with the
CUDA path.

What the pages fix, and the reading taken where they stop:

* Shared key/value heads -- "FlashAttention：IO 感知的精确注意力"
  (inference.xph.ink kp-015), "与其他知识点的关系": grouped K/V heads (GQA)
  shrink the K/V volume and combine with the exact, IO-aware kernel. The page
  gives no formula. Reading: H query heads and H_kv key/value heads with H a
  multiple of H_kv; query head h attends to K/V head h // (H / H_kv), the
  usual grouping of consecutive query heads. Everything else is the
  definition of :func:`oracle.attention.attention`.
* Short queries against a long key/value cache -- the same page, "常见误区" and
  "自测题": decode (generation) is bandwidth-bound, unlike prefill. Reading:
  N_q query rows (often 1) attend to all N_kv keys, no mask; the definition
  does not depend on N_q.
* Combining partial results over disjoint key ranges -- "Flash Attention (FA1)"
  (languisher.top), derivation steps 4-5: two softmax states (m1, l1, O1) and
  (m2, l2, O2) over disjoint key sets combine through m = max(m1, m2),
  l = e^{m1-m} l1 + e^{m2-m} l2, O = (e^{m1-m} l1 O1 + e^{m2-m} l2 O2) / l.
  With LSE_s = m_s + ln l_s that is LSE = ln sum_s e^{LSE_s} and
  O = sum_s e^{LSE_s - LSE} O_s (:func:`merge_partials`, which takes the steps
  in that order: the maximum first, then the rescaled sums).

Parity status: pinned by ``tests/test_oracle_gqa_pins.py`` (reduction to the
pinned plain attention at H_kv = H, torch float64 with repeated heads,
independence of groups, merges of arbitrary partitions equal to the whole,
planted mistakes); none is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

from .attention import _attention_one_head

__all__ = ["attention_gqa", "attention_gqa_rows", "merge_partials", "attention_split"]


def attention_gqa(Q, K, V, scale: float):
    """O and LSE for Q [B, H, N_q, d] against K, V [B, H_kv, N_kv, d].

    Query head h uses K/V head h // (H // H_kv). Returns O [B, H, N_q, d]
    and LSE [B, H, N_q], float64.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    B, H, Nq, _ = Q.shape
    Hkv = K.shape[1]
    if H % Hkv:
        raise ValueError("H must be a multiple of H_kv")
    G = H // Hkv
    O = np.empty((B, H, Nq, V.shape[-1]))
    L = np.empty((B, H, Nq))
    for b in range(B):
        for h in range(H):
            O[b, h], L[b, h] = _attention_one_head(Q[b, h], K[b, h // G], V[b, h // G], scale)
    return O, L


def attention_gqa_rows(Q, K, V, scale: float, heads):
    """The same for selected query heads: ``heads`` is a list of (b, h);
    returns a list of (O [N_q, d], LSE [N_q])."""
    G = Q.shape[1] // K.shape[1]
    out = []
    for b, h in heads:
        q, k, v = (np.asarray(x, dtype=np.float64) for x in (Q[b, h], K[b, h // G], V[b, h // G]))
        out.append(_attention_one_head(q, k, v, scale))
    return out


def merge_partials(O_parts, LSE_parts):
    """Combine S partial results over disjoint key ranges.

    O_parts [S, ..., d] (each normalised by its own l_s), LSE_parts [S, ...].
    Returns (O, LSE) with LSE = ln sum_s e^{LSE_s} and
    O = sum_s e^{LSE_s - LSE} O_s, evaluated with the maximum taken first.
    """
    O_parts = np.asarray(O_parts, dtype=np.float64)
    LSE_parts = np.asarray(LSE_parts, dtype=np.float64)
    m = LSE_parts.max(axis=0)                         # the largest partial log-sum-exp
    w = np.exp(LSE_parts - m)                         # e^{LSE_s - m}, at most 1
    total = w.sum(axis=0)
    LSE = m + np.log(total)
    O = np.einsum("s...,s...d->...d", w / total, O_parts)
    return O, LSE


def attention_split(Q, K, V, scale: float, bounds):
    """Attention over the key ranges [bounds[s], bounds[s+1]) computed
    separately (with :func:`attention_gqa`) and merged with :func:`merge_partials`."""
    parts = [attention_gqa(Q, K[:, :, a:b], V[:, :, a:b], scale) for a, b in zip(bounds[:-1], bounds[1:])]
    return merge_partials(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
