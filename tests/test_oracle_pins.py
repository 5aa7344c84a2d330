"""The oracle against what the pages and mathematics fix (CPU only)."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from tests import oracle_pins as pins


def _full(Q, K, V, s):
    return oracle.attention(Q, K, V, s)


# --- the plain definition --------------------------------------------------
@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pins(pin):
    if pin is pins.pin_bruteforce_mp:
        pytest.importorskip("mpmath")
    pin(_full)


# --- the pages' tiled recurrence obeys the same pins ------------------------
@pytest.mark.parametrize("impl", ["fa1_kv_outer", "fa1_q_outer", "fa2"])
@pytest.mark.parametrize("pin", [pins.pin_n1, pins.pin_n2_logistic, pins.pin_constant_v, pins.pin_uniform,
                                 pins.pin_shift_via_inputs, pins.pin_library_sdpa],
                         ids=lambda p: p.__name__)
def test_recurrence_pins(impl, pin):
    if impl == "fa2":
        f = lambda Q, K, V, s: oracle.flash_fa2(Q, K, V, s, 5, 3)   # noqa: E731
    else:
        order = "kv_outer" if impl.endswith("kv_outer") else "q_outer"
        f = lambda Q, K, V, s: oracle.flash_fa1(Q, K, V, s, 5, 3, order)  # noqa: E731
    pin(f)


_BLOCKS = [1, 2, 3, 5, 16, 64, 128, None]   # None = the whole sequence


@pytest.mark.parametrize("Br", _BLOCKS)
@pytest.mark.parametrize("Bc", _BLOCKS)
def test_recurrence_equals_full_softmax(Br, Bc):
    """'Flash Attention (FA1)', online softmax: tile-by-tile updates equal the global
    softmax exactly (up to float64 rounding) for every block size, including block
    sizes that do not divide N (ragged last tile, T = ceil(N/B))."""
    r = np.random.default_rng(11)
    N, d = 133, 8
    Q = r.standard_normal((1, 2, N, d)) * 3
    K = r.standard_normal((1, 2, N, d)) * 3
    V = r.standard_normal((1, 2, N, d))
    s = 1 / math.sqrt(d)
    O, L = oracle.attention(Q, K, V, s)
    br = Br or N
    bc = Bc or N
    for order in ("kv_outer", "q_outer"):
        O1, L1 = oracle.flash_fa1(Q, K, V, s, br, bc, order)
        np.testing.assert_allclose(O1, O, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(L1, L, rtol=1e-12, atol=1e-12)
    O2, L2 = oracle.flash_fa2(Q, K, V, s, br, bc)
    np.testing.assert_allclose(O2, O, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(L2, L, rtol=1e-12, atol=1e-12)


def test_recurrence_spiky_rows():
    """Rows whose maximum jumps by large amounts from tile to tile (the long-context
    stress pattern) still agree: the running-max rescale of step 2 is exact."""
    r = np.random.default_rng(12)
    N, d = 300, 16
    Q = r.standard_normal((1, 1, N, d)) * 3
    K = r.standard_normal((1, 1, N, d)) * 3
    K[0, 0, r.permutation(N)[:3]] *= 8
    K[0, 0, -1] *= 20          # the largest score arrives in the very last tile
    s = 1 / math.sqrt(d)
    O, L = oracle.attention(Q, K, Q * 0 + r.standard_normal((1, 1, N, d)), s)
    V = Q * 0 + r.standard_normal((1, 1, N, d))
    O, L = oracle.attention(Q, K, V, s)
    for br, bc in [(16, 16), (7, 128), (128, 13)]:
        O2, L2 = oracle.flash_fa2(Q, K, V, s, br, bc)
        np.testing.assert_allclose(O2, O, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(L2, L, rtol=1e-13, atol=1e-11)
        O1, L1 = oracle.flash_fa1(Q, K, V, s, br, bc)
        np.testing.assert_allclose(O1, O, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(L1, L, rtol=1e-13, atol=1e-11)


# --- safe softmax -------------------------------------------------------------
def test_rows_of_p_sum_to_one():
    r = np.random.default_rng(13)
    S = r.standard_normal((50, 77)) * 20
    P, m, l = oracle.safe_softmax(S)
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(P >= 0)
    np.testing.assert_array_equal(m, S.max(axis=1))
    assert np.all(l >= 1.0)          # the max term contributes e^0 = 1


def test_softmax_shift_invariance():
    """Subtracting (or adding) a per-row constant does not change P; m moves by it."""
    r = np.random.default_rng(14)
    S = r.standard_normal((40, 33)) * 5
    c = r.uniform(-100, 100, size=40)
    P, m, l = oracle.safe_softmax(S)
    P2, m2, l2 = oracle.safe_softmax(S + c[:, None])
    np.testing.assert_allclose(P2, P, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(m2, m + c, rtol=1e-14, atol=1e-12)
    np.testing.assert_allclose(l2, l, rtol=1e-12)


def test_softmax_no_overflow():
    """The max subtraction keeps huge scores finite (the reason for 'safe' softmax)."""
    S = np.array([[1000.0, 999.0, -1000.0], [-1e300, -1e300, -1e300]])
    P, m, l = oracle.safe_softmax(S)
    assert np.all(np.isfinite(P))
    np.testing.assert_allclose(P[0, :2], [1 / (1 + math.exp(-1)), math.exp(-1) / (1 + math.exp(-1))], rtol=1e-14)
    np.testing.assert_allclose(P[1], [1 / 3] * 3, rtol=1e-14)


# --- sampled rows equal the full evaluation ---------------------------------------
def test_attention_rows_matches_full():
    r = np.random.default_rng(15)
    Q, K, V = (r.standard_normal((2, 3, 70, 16)) for _ in range(3))
    O, L = oracle.attention(Q, K, V, 0.25, row_chunk=16)
    rows = np.array([[1, 2, 69], [0, 0, 0], [1, 0, 33], [0, 2, 5], [1, 2, 0]])
    Os, Ls = oracle.attention_rows(Q, K, V, 0.25, rows)
    for i, (b, h, n) in enumerate(rows):
        np.testing.assert_allclose(Os[i], O[b, h, n], rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(Ls[i], L[b, h, n], rtol=1e-15, atol=1e-15)


# --- bf16 rounding and the materialise-path reference ------------------------------
def test_bf16_round_matches_torch():
    """RNE to bf16 agrees bit for bit with torch's float32 -> bfloat16 conversion."""
    r = np.random.default_rng(16)
    x = np.concatenate([
        r.standard_normal(100000).astype(np.float32) * np.float32(10) ** r.integers(-30, 30, 100000).astype(np.float32),
        # exact ties: low 16 bits = 0x8000, with even and odd kept bits
        (np.arange(1, 2000, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, 1e-45, -1e-45], dtype=np.float32),
    ])
    # a stride through every 32-bit pattern, and the largest finite values and
    # infinities of both signs (where a 32-bit sum would come closest to wrapping)
    sweep = np.arange(0, 1 << 32, 65537, dtype=np.uint64).astype(np.uint32)
    edges = np.array([0x7F7FFFFF, 0xFF7FFFFF, 0x7F7F8000, 0xFF7F8000, 0x7F800000, 0xFF800000, 0x7F7F7FFF,
                      0xFF7F7FFF], dtype=np.uint32)
    bits = np.concatenate([sweep, edges]).view(np.float32)
    x = np.concatenate([x, bits[~np.isnan(bits)]])
    mine = oracle.bf16_round(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(mine.view(np.uint32), ref.view(np.uint32))
    assert np.isnan(oracle.bf16_round(np.array([np.nan], dtype=np.float32)))[0]


def test_naive_bf16_n1_exact():
    """N = 1: P = 1 exactly, so the bf16 materialise path returns V exactly."""
    r = np.random.default_rng(17)
    V = oracle.bf16_round(r.standard_normal((1, 2, 1, 16))).astype(np.float64)
    Q = r.standard_normal((1, 2, 1, 16))
    O = oracle.naive_bf16_attention(Q, Q, V, 0.3)
    np.testing.assert_array_equal(O, V)


def test_naive_bf16_matches_torch_bf16_pipeline():
    """The reference agrees with torch's own bf16 CPU pipeline (matmul -> scale ->
    softmax -> matmul, each result stored in bf16) except for rare one-ulp flips
    caused by a different float32 summation order."""
    g = torch.Generator().manual_seed(18)
    q, k, v = (torch.randn(1, 2, 96, 64, generator=g).to(torch.bfloat16) for _ in range(3))
    s = 0.125
    S = (q @ k.transpose(-1, -2)) * s
    P = torch.softmax(S.float(), dim=-1).to(torch.bfloat16)
    Ot = (P @ v).float().numpy().astype(np.float64)
    On = oracle.naive_bf16_attention(q.float().numpy(), k.float().numpy(), v.float().numpy(), s)
    same = np.mean(On == Ot)
    assert same > 0.97, same
    ulp = np.abs(Ot) * 2.0 ** -7 + 1e-30
    assert np.all(np.abs(On - Ot) <= 2 * ulp + 2 ** -133)


def test_naive_bf16_error_is_bf16_sized():
    """Its error against the float64 definition is of bf16 size: nonzero, and
    well under a percent of the output scale."""
    r = np.random.default_rng(19)
    Q, K, V = (oracle.bf16_round(r.standard_normal((1, 2, 256, 64))).astype(np.float64) for _ in range(3))
    O, _ = oracle.attention(Q, K, V, 0.125)
    On = oracle.naive_bf16_attention(Q, K, V, 0.125)
    err = np.abs(On - O).max()
    assert 1e-5 < err < 2e-2 * np.abs(O).max()


# --- planted mistakes fail at least one pin -----------------------------------------
def _mutants():
    def no_max(Q, K, V, s):
        S = s * np.einsum("bhid,bhjd->bhij", Q, K)
        e = np.exp(S)
        l = e.sum(-1)
        return np.einsum("bhij,bhjd->bhid", e / l[..., None], V), np.log(l)

    def transposed(Q, K, V, s):
        S = s * np.einsum("bhid,bhjd->bhji", Q, K)
        P, m, l = oracle.safe_softmax(S)
        return np.einsum("bhij,bhjd->bhid", P, V), m + np.log(l)

    def no_scale(Q, K, V, s):
        return oracle.attention(Q, K, V, 1.0)

    def lse_without_max(Q, K, V, s):
        O, L = oracle.attention(Q, K, V, s)
        S = s * np.einsum("bhid,bhjd->bhij", Q, K)
        return O, L - S.max(-1)

    def unnormalised(Q, K, V, s):
        S = s * np.einsum("bhid,bhjd->bhij", Q, K)
        m = S.max(-1, keepdims=True)
        e = np.exp(S - m)
        return np.einsum("bhij,bhjd->bhid", e, V), (m[..., 0] + np.log(e.sum(-1)))

    def wrong_axis(Q, K, V, s):
        S = s * np.einsum("bhid,bhjd->bhij", Q, K)
        m = S.max(-2, keepdims=True)
        e = np.exp(S - m)
        P = e / e.sum(-2, keepdims=True)
        return np.einsum("bhij,bhjd->bhid", P, V), np.log(np.exp(S).sum(-1))

    def log2_lse(Q, K, V, s):
        O, L = oracle.attention(Q, K, V, s)
        return O, L / math.log(2)

    def fa1_dropped_history(Q, K, V, s):
        # step 4 dropped: history not rescaled by e^{m - m_new}
        B, H, N, d = Q.shape
        O = np.zeros_like(Q)
        Ls = np.zeros(Q.shape[:3])
        for b in range(B):
            for h in range(H):
                o = np.zeros((N, d)); l = np.zeros(N); m = np.full(N, -np.inf)
                for c0 in range(0, N, 4):
                    S = s * Q[b, h] @ K[b, h, c0:c0 + 4].T
                    mt = S.max(1); Pt = np.exp(S - mt[:, None]); lt = Pt.sum(1)
                    mn = np.maximum(m, mt)
                    ln = l + lt * np.exp(mt - mn)
                    o = (l[:, None] * o + np.exp(mt - mn)[:, None] * (Pt @ V[b, h, c0:c0 + 4])) / ln[:, None]
                    m, l = mn, ln
                O[b, h] = o
                Ls[b, h] = m + np.log(l)
        return O, Ls

    return [no_max, transposed, no_scale, lse_without_max, unnormalised, wrong_axis, log2_lse,
            fa1_dropped_history]


@pytest.mark.parametrize("mutant", _mutants(), ids=lambda f: f.__name__)
def test_planted_mistake_is_caught(mutant):
    pytest.importorskip("mpmath")
    caught = []
    for pin in pins.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mutant)
        except (AssertionError, FloatingPointError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught {mutant.__name__}"
