"""Exact-attention backward oracle: plain, slow, float64, CPU.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it. It shares no code with the
CUDA path (no kernels, headers, helpers or constants).

What the pages fix, and the reading taken where they stop:

* "01 · 注意力为什么是 IO 瓶颈" (ai-reference-codex) §7, third item: the
  backward of the fused method keeps only O and the per-row LSE from the
  forward and rebuilds the probabilities P from them, instead of reading back
  a stored N x N matrix as standard attention does. The pages print no
  gradient formulas (they point to a chapter that is not among them).
* Reading: the backward computes the gradients of the scalar L = <dO, O>
  (dO, the incoming gradient of O, is an input) with respect to Q, K and V
  for O = softmax(scale Q K^T) V, one softmax per query row. The chain rule
  gives, per (batch, head):
      S  = scale Q K^T,   P = softmax(S) row-wise
      dV = P^T dO
      dP = dO V^T
      dS = P * (dP - D[:, None]),   D_i = sum_j P_ij dP_ij
           (the Jacobian of a row softmax applied to dP)
      dQ = scale dS K,   dK = scale dS^T Q
  :func:`attention_bwd` writes exactly that, with P from the safe softmax.
* The recomputation form (:func:`attention_bwd_recompute`) is what §7
  describes: P_ij = exp(S_ij - LSE_i) from the stored LSE, and D_i = dO_i . O_i
  from the stored O. Both equal the definition's values when O and LSE are
  exact, because O_i = sum_j P_ij V_j gives sum_j P_ij dP_ij = dO_i . O_i.
* The bf16 materialise path (:func:`naive_bf16_attention_bwd`) is the
  standard-attention backward as a bf16 framework would run it, the
  "PyTorch baseline" of §7's error rule; its rounding points are a reading,
  stated in its docstring.

All arrays are numpy; shapes are [B, H, N, d] for Q, K, V, O, dO and the
gradients, [B, H, N] for LSE.

Parity status: every function here is pinned by ``tests/test_oracle_bwd_pins.py``
(finite differences of the pinned forward oracle, torch float64 autograd,
closed forms for N = 1 and equal keys, and column-sum invariants); none is
"parity unpinned".
"""
from __future__ import annotations

import numpy as np

from .attention import bf16_round, safe_softmax

__all__ = ["attention_bwd", "attention_bwd_recompute", "attention_bwd_heads", "naive_bf16_attention_bwd"]


def _bwd_one_head(q, k, v, do, scale, row_chunk):
    """Definition for one head: q [r, d], k/v [n, d], do [r, dv] -> (dq, dk, dv)."""
    dq = np.empty_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for r0 in range(0, q.shape[0], row_chunk):
        r1 = min(q.shape[0], r0 + row_chunk)
        S = scale * (q[r0:r1] @ k.T)                  # scaled scores
        P, _, _ = safe_softmax(S)                     # probabilities, one softmax per row
        dv += P.T @ do[r0:r1]                         # dV = P^T dO
        dP = do[r0:r1] @ v.T                          # dP = dO V^T
        D = np.sum(P * dP, axis=1)                    # D_i = sum_j P_ij dP_ij
        dS = P * (dP - D[:, None])                    # softmax Jacobian
        dq[r0:r1] = scale * (dS @ k)                  # dQ = scale dS K
        dk += scale * (dS.T @ q[r0:r1])               # dK = scale dS^T Q
    return dq, dk, dv


def attention_bwd(Q, K, V, dO, scale: float, row_chunk: int = 2048):
    """Gradients (dQ, dK, dV) of <dO, softmax(scale Q K^T) V>, float64.

    Q, K, V, dO: [B, H, N, d]. Query rows are processed ``row_chunk`` at a time
    only to bound the materialised N x N matrices; dK and dV sum over all of them.
    """
    Q, K, V, dO = (np.asarray(x, dtype=np.float64) for x in (Q, K, V, dO))
    B, H = Q.shape[:2]
    dQ = np.empty_like(Q)
    dK = np.empty_like(K)
    dV = np.empty_like(V)
    for b in range(B):
        for h in range(H):
            dQ[b, h], dK[b, h], dV[b, h] = _bwd_one_head(Q[b, h], K[b, h], V[b, h], dO[b, h], scale, row_chunk)
    return dQ, dK, dV


def attention_bwd_heads(Q, K, V, dO, scale: float, heads, row_chunk: int = 2048):
    """The definition evaluated for selected heads only.

    ``heads`` is a list of (b, h) pairs; returns a list of (dq, dk, dv) triples,
    each [N, d] float64, in that order.
    """
    out = []
    for b, h in heads:
        q, k, v, do = (np.asarray(x[b, h], dtype=np.float64) for x in (Q, K, V, dO))
        out.append(_bwd_one_head(q, k, v, do, scale, row_chunk))
    return out


def attention_bwd_recompute(Q, K, V, O, dO, LSE, scale: float, row_chunk: int = 2048):
    """Recomputation form: P rebuilt from LSE, D from O (the pages' §7 scheme).

    P_ij = exp(scale q_i . k_j - LSE_i),  D_i = dO_i . O_i; then dV, dP, dS,
    dQ and dK as in :func:`attention_bwd`. O and LSE are inputs (the forward's
    outputs); with exact O and LSE the result equals the definition's.
    """
    Q, K, V, O, dO = (np.asarray(x, dtype=np.float64) for x in (Q, K, V, O, dO))
    LSE = np.asarray(LSE, dtype=np.float64)
    B, H, N, _ = Q.shape
    dQ = np.empty_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    for b in range(B):
        for h in range(H):
            q, k, v, o, do, lse = Q[b, h], K[b, h], V[b, h], O[b, h], dO[b, h], LSE[b, h]
            for r0 in range(0, N, row_chunk):
                r1 = min(N, r0 + row_chunk)
                P = np.exp(scale * (q[r0:r1] @ k.T) - lse[r0:r1, None])   # rebuilt probabilities
                D = np.sum(do[r0:r1] * o[r0:r1], axis=1)                  # D_i = dO_i . O_i
                dV[b, h] += P.T @ do[r0:r1]
                dS = P * (do[r0:r1] @ v.T - D[:, None])
                dQ[b, h, r0:r1] = scale * (dS @ k)
                dK[b, h] += scale * (dS.T @ q[r0:r1])
    return dQ, dK, dV


def naive_bf16_attention_bwd(Q, K, V, dO, scale: float, heads=None):
    """Standard-attention backward with bf16 storage of every intermediate.

    Reading of the rounding points of a bf16 framework running the
    materialise-path attention ("01 · 注意力为什么是 IO 瓶颈" §3) through its
    autograd; every product is summed in float32 and stored in bf16:
      forward (as in the bf16 forward reference):
        S = bf16(scale * bf16(Q K^T)),  P = bf16(softmax(S) in float32)
      backward:
        dV = bf16(P^T dO)
        dP = bf16(dO V^T)
        dS = bf16(P * (dP - rowsum(P * dP))), evaluated in float32
        dS' = bf16(scale * dS)            (the gradient through S = scale * .)
        dQ = bf16(dS' K),   dK = bf16(dS'^T Q)
    Returns (dQ, dK, dV) float64 holding bf16 values. ``heads`` optionally
    selects (b, h) pairs; then a list of (dq, dk, dv) triples is returned.
    """
    s32 = np.float32(scale)

    def one(q, k, v, do):
        S = bf16_round(q @ k.T)
        S = bf16_round(S * s32)
        m = S.max(axis=1, keepdims=True)
        e = np.exp(S - m, dtype=np.float32)
        P = bf16_round(e / e.sum(axis=1, keepdims=True, dtype=np.float32))
        dv = bf16_round(P.T @ do)
        dP = bf16_round(do @ v.T)
        D = np.sum(P * dP, axis=1, keepdims=True, dtype=np.float32)
        dS = bf16_round(P * (dP - D))
        dS = bf16_round(dS * s32)
        dq = bf16_round(dS @ k)
        dk = bf16_round(dS.T @ q)
        return dq.astype(np.float64), dk.astype(np.float64), dv.astype(np.float64)

    Qf, Kf, Vf, dOf = (np.asarray(x, dtype=np.float32) for x in (Q, K, V, dO))
    if heads is not None:
        return [one(Qf[b, h], Kf[b, h], Vf[b, h], dOf[b, h]) for b, h in heads]
    B, H = Qf.shape[:2]
    dQ = np.empty(Qf.shape)
    dK = np.empty(Kf.shape)
    dV = np.empty(Vf.shape)
    for b in range(B):
        for h in range(H):
            dQ[b, h], dK[b, h], dV[b, h] = one(Qf[b, h], Kf[b, h], Vf[b, h], dOf[b, h])
    return dQ, dK, dV
