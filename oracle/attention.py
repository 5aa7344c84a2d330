"""Exact-attention oracle: plain, slow, float64, CPU.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it. It shares no code with the
CUDA path (no kernels, headers, helpers or constants).

What it computes, and where each step comes from (page title, then section):

* Safe softmax -- "Flash Attention (FA1)" (languisher.top), section
  "Naive Attention 问题分析" (naive attention analysis): for a vector x,
  m(x) = max_i x_i and softmax(x) = [e^{x_i - m(x)}] / sum_j e^{x_j - m(x)}.
* Standard attention O = softmax(QK^T) V, one independent softmax per query
  row -- "01 · 注意力为什么是 IO 瓶颈" (ai-reference-codex) §1 and §5, and
  "Flash Attention (FA1)", "Online Softmax in FlashAttention" (each row is its
  own softmax). The pages print the score formula without a scale (the
  standard-attention formula itself was lost in extraction); this oracle
  reads it as S = scale * Q K^T with the caller's scale.
* The log-sum-exp output, one float32 per query row -- "01 · 注意力为什么是
  IO 瓶颈" §4 (the fused kernel writes O and LSE) and §6 (softmax_lse, one
  float32 per row). Reading: LSE = m + ln l of the *scaled* scores, the value
  the backward recomputation (§7 of the same page) needs to rebuild P.
* Tiling -- "Flash Attention (FA1)", "Tiling in FlashAttention": Q split into
  Tr = ceil(N/Br) row blocks, K and V into Tc = ceil(N/Bc) blocks, K/V in the
  outer loop and Q/O in the inner loop. "01 · 注意力为什么是 IO 瓶颈" §5 sketches
  the other order (Q outer, K/V inner); both orders are provided.
* The online-softmax state update -- "Flash Attention (FA1)", "核心局部状态计算
  和更新公式推导" (derivation of the local state and its update), steps 1-5
  and the boxed O_new equation, restated in "总结" (summary).
* The FlashAttention-2 arrangement (fewer non-matmul operations: keep O
  unnormalised and divide once at the end, parallel over query blocks) --
  "FlashAttention：IO 感知的精确注意力" (inference.xph.ink kp-015), core
  concepts, last item.
* The materialise-then-softmax bf16 path used by the "error no larger than
  twice the PyTorch baseline" rule -- "01 · 注意力为什么是 IO 瓶颈" §3 (three
  kernels, S and P written to HBM) and §7 (the tolerance rule). The pages do
  not fix its rounding points; the reading used here is stated in
  :func:`naive_bf16_attention`.

All arrays are numpy; float inputs are converted exactly to float64 (bf16
values are exactly representable). Shapes are [B, H, N, d] for Q, K, V and O,
[B, H, N] for LSE, row-major, as the fused kernel's interface uses.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, high-precision brute force, invariants and a library routine);
none is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_round",
    "safe_softmax",
    "attention",
    "attention_rows",
    "flash_fa1",
    "flash_fa2",
    "naive_bf16_attention",
]


# ---------------------------------------------------------------------------
# bf16 rounding (used only by the naive materialise-path reference)
# ---------------------------------------------------------------------------
def bf16_round(x) -> np.ndarray:
    """Round to the nearest bfloat16 value, ties to even; returns float32.

    bfloat16 is the upper 16 bits of an IEEE float32. Rounding to nearest-even
    adds 0x7FFF plus the lowest kept bit, then truncates the low 16 bits.
    The sum stays below 2^32 for every non-NaN bit pattern (the largest,
    -inf = 0xFF800000, reaches 0xFF807FFF), so 32-bit unsigned arithmetic is
    exact. NaN is passed through unchanged.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    keep_lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + (np.uint32(0x7FFF) + keep_lsb)) & np.uint32(0xFFFF0000)
    out = r.view(np.float32)
    return np.where(np.isnan(x), x, out)


# ---------------------------------------------------------------------------
# Safe softmax, row-wise ("Flash Attention (FA1)", naive attention analysis)
# ---------------------------------------------------------------------------
def safe_softmax(S: np.ndarray):
    """Row-wise safe softmax of a float64 matrix S [..., n].

    Returns (P, m, l) with m = row max, l = sum_j e^{S_j - m}, P = e^{S - m}/l.
    """
    S = np.asarray(S, dtype=np.float64)
    m = S.max(axis=-1)
    e = np.exp(S - m[..., None])
    l = e.sum(axis=-1)
    return e / l[..., None], m, l


# ---------------------------------------------------------------------------
# Plain definition: materialise S in float64, safe softmax, multiply by V
# ---------------------------------------------------------------------------
def _attention_one_head(q, k, v, scale):
    """q [r, d], k [n, d], v [n, d] float64 -> (O [r, d], LSE [r])."""
    S = scale * (q @ k.T)                 # scores, float64
    P, m, l = safe_softmax(S)             # safe softmax per query row
    O = P @ v                             # weighted sum of value rows
    lse = m + np.log(l)                   # natural log-sum-exp of the scaled scores
    return O, lse


def attention(Q, K, V, scale: float, row_chunk: int = 2048):
    """O = softmax(scale * Q K^T) V and LSE for every (batch, head, row).

    Q, K, V: [B, H, N, d]. Returns O [B, H, N, d] float64 and LSE [B, H, N]
    float64. Query rows are independent softmaxes, so they are evaluated
    ``row_chunk`` rows at a time only to bound the size of the materialised S.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    B, H, N, _ = Q.shape
    dv = V.shape[-1]
    O = np.empty((B, H, N, dv), dtype=np.float64)
    LSE = np.empty((B, H, N), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            for r0 in range(0, N, row_chunk):
                r1 = min(N, r0 + row_chunk)
                O[b, h, r0:r1], LSE[b, h, r0:r1] = _attention_one_head(
                    Q[b, h, r0:r1], K[b, h], V[b, h], scale)
    return O, LSE


def attention_rows(Q, K, V, scale: float, rows):
    """The same definition evaluated only at sampled query rows.

    ``rows`` is an integer array [R, 3] of (b, h, r) triples. Returns
    O [R, d] and LSE [R] float64 for those rows, in the given order.
    """
    rows = np.asarray(rows, dtype=np.int64).reshape(-1, 3)
    O = np.empty((rows.shape[0], V.shape[-1]), dtype=np.float64)
    LSE = np.empty((rows.shape[0],), dtype=np.float64)
    # group by head so K and V of a head are converted once
    heads = {}
    for idx, (b, h, r) in enumerate(rows):
        heads.setdefault((int(b), int(h)), []).append((idx, int(r)))
    for (b, h), items in heads.items():
        k = np.asarray(K[b, h], dtype=np.float64)
        v = np.asarray(V[b, h], dtype=np.float64)
        idxs = np.array([i for i, _ in items])
        rr = np.array([r for _, r in items])
        q = np.asarray(Q[b, h][rr], dtype=np.float64)
        O[idxs], LSE[idxs] = _attention_one_head(q, k, v, scale)
    return O, LSE


# ---------------------------------------------------------------------------
# The pages' tiled online-softmax recurrence
# ---------------------------------------------------------------------------
def _tile_bounds(n: int, block: int):
    """Row ranges of the ceil(n/block) tiles ("Tiling in FlashAttention")."""
    t = -(-n // block)
    return [(i * block, min(n, (i + 1) * block)) for i in range(t)]


def flash_fa1(Q, K, V, scale: float, Br: int, Bc: int, order: str = "kv_outer"):
    """FlashAttention-1 recurrence with O kept normalised after every tile.

    Follows "Flash Attention (FA1)", derivation steps 1-5 (and the summary):
      1. local state:  m~ = rowmax(S_ij), P~ = exp(S_ij - m~), l~ = rowsum(P~)
      2. running state: m_new = max(m_i, m~),
                        l_new = l_i e^{m_i - m_new} + l~ e^{m~ - m_new}
      3. tile numerator: O~ = P~ V_j
      4-5. O_new = diag(l_new)^{-1} (diag(l_i e^{m_i - m_new}) O_i
                                       + e^{m~ - m_new} O~)
    Initial state (the algorithm figure was lost; reading): m = -inf, l = 0,
    O = 0, so the first update reduces to (m~, l~, O~/l~).

    ``order`` = "kv_outer" is the page's loop order (K/V outer, Q/O inner);
    "q_outer" is the order sketched in "01 · 注意力为什么是 IO 瓶颈" §5.
    Returns (O, LSE) with LSE = m + ln l.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    B, H, N, _ = Q.shape
    d = V.shape[-1]
    O_all = np.zeros((B, H, N, d))
    LSE_all = np.zeros((B, H, N))
    q_tiles = _tile_bounds(N, Br)
    kv_tiles = _tile_bounds(K.shape[2], Bc)
    if order == "kv_outer":
        pairs = [(i, j) for j in range(len(kv_tiles)) for i in range(len(q_tiles))]
    elif order == "q_outer":
        pairs = [(i, j) for i in range(len(q_tiles)) for j in range(len(kv_tiles))]
    else:
        raise ValueError(order)
    for b in range(B):
        for h in range(H):
            O = np.zeros((N, d))
            l = np.zeros(N)
            m = np.full(N, -np.inf)
            for i, j in pairs:
                r0, r1 = q_tiles[i]
                c0, c1 = kv_tiles[j]
                S_ij = scale * (Q[b, h, r0:r1] @ K[b, h, c0:c1].T)
                # step 1: local statistics of this tile
                m_t = S_ij.max(axis=1)
                P_t = np.exp(S_ij - m_t[:, None])
                l_t = P_t.sum(axis=1)
                # step 2: running max and normaliser
                m_i, l_i = m[r0:r1], l[r0:r1]
                m_new = np.maximum(m_i, m_t)
                old_w = np.where(np.isneginf(m_i), 0.0, np.exp(m_i - m_new))
                new_w = np.exp(m_t - m_new)
                l_new = l_i * old_w + l_t * new_w
                # step 3: this tile's numerator
                O_t = P_t @ V[b, h, c0:c1]
                # steps 4-5: rescale history, merge, renormalise
                Phi = (l_i * old_w)[:, None] * O[r0:r1]
                Delta = new_w[:, None] * O_t
                O[r0:r1] = (Phi + Delta) / l_new[:, None]
                m[r0:r1], l[r0:r1] = m_new, l_new
            O_all[b, h] = O
            LSE_all[b, h] = m + np.log(l)
    return O_all, LSE_all


def flash_fa2(Q, K, V, scale: float, Br: int, Bc: int):
    """FlashAttention-2 arrangement of the same recurrence.

    Q blocks outer, K/V blocks inner; O is kept as the unnormalised numerator
    and divided by l once after the last tile ("FlashAttention：IO 感知的精确
    注意力", core concepts: fewer non-matmul operations). Per tile, with
    m_new = max(m, rowmax(S_ij)) and alpha = e^{m - m_new}:
        l   <- alpha l + rowsum(e^{S_ij - m_new})
        acc <- alpha acc + e^{S_ij - m_new} V_j
    which is steps 2-5 of "Flash Attention (FA1)" with the exponentials of
    step 1 taken against m_new directly (e^{S - m~} e^{m~ - m_new} = e^{S - m_new}).
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    B, H, N, _ = Q.shape
    d = V.shape[-1]
    O_all = np.zeros((B, H, N, d))
    LSE_all = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            for r0, r1 in _tile_bounds(N, Br):
                acc = np.zeros((r1 - r0, d))
                l = np.zeros(r1 - r0)
                m = np.full(r1 - r0, -np.inf)
                for c0, c1 in _tile_bounds(K.shape[2], Bc):
                    S = scale * (Q[b, h, r0:r1] @ K[b, h, c0:c1].T)
                    m_new = np.maximum(m, S.max(axis=1))
                    alpha = np.where(np.isneginf(m), 0.0, np.exp(m - m_new))
                    P = np.exp(S - m_new[:, None])
                    l = alpha * l + P.sum(axis=1)
                    acc = alpha[:, None] * acc + P @ V[b, h, c0:c1]
                    m = m_new
                O_all[b, h, r0:r1] = acc / l[:, None]
                LSE_all[b, h, r0:r1] = m + np.log(l)
    return O_all, LSE_all


# ---------------------------------------------------------------------------
# Materialise-path reference in bf16 (for the "twice the baseline" rule)
# ---------------------------------------------------------------------------
def naive_bf16_attention(Q, K, V, scale: float, rows=None):
    """Standard three-step attention with bf16 storage of S, P and O.

    "01 · 注意力为什么是 IO 瓶颈" §3 and §5: S = QK^T is written out, P =
    softmax(S) is written out, then O = PV. The pages only say the fused
    result must be no worse than twice the error of the PyTorch baseline
    (§7). Reading of that baseline's rounding points, as a bf16 framework
    would run it:
      S = bf16(sum of float32 products of the bf16 Q and K values)
      S = bf16(scale * S)
      P = bf16(softmax of S evaluated in float32)
      O = bf16(sum of float32 products of P and V)
    Returns O as float64 (holding bf16 values). ``rows`` optionally selects
    (b, h, r) triples as in :func:`attention_rows`; then O is [R, d].
    """
    Qf = np.asarray(Q, dtype=np.float32)
    Kf = np.asarray(K, dtype=np.float32)
    Vf = np.asarray(V, dtype=np.float32)
    s32 = np.float32(scale)

    def one(q, k, v):
        S = bf16_round(q @ k.T)
        S = bf16_round(S * s32)
        m = S.max(axis=1, keepdims=True)
        e = np.exp(S - m, dtype=np.float32)
        P = bf16_round(e / e.sum(axis=1, keepdims=True, dtype=np.float32))
        return bf16_round(P @ v).astype(np.float64)

    if rows is None:
        B, H, N, d = Qf.shape
        O = np.empty((B, H, N, d))
        for b in range(B):
            for h in range(H):
                for r0 in range(0, N, 2048):
                    r1 = min(N, r0 + 2048)
                    O[b, h, r0:r1] = one(Qf[b, h, r0:r1], Kf[b, h], Vf[b, h])
        return O
    rows = np.asarray(rows, dtype=np.int64).reshape(-1, 3)
    O = np.empty((rows.shape[0], Qf.shape[-1]))
    heads = {}
    for idx, (b, h, r) in enumerate(rows):
        heads.setdefault((int(b), int(h)), []).append((idx, int(r)))
    for (b, h), items in heads.items():
        idxs = np.array([i for i, _ in items])
        rr = np.array([r for _, r in items])
        O[idxs] = one(Qf[b, h][rr], Kf[b, h], Vf[b, h])
    return O
