"""Seeded synthetic inputs for the attention forward pass.

This module holds no attention arithmetic: it only draws Q, K and V. It is
the one module that both the oracle side (tests, CPU baseline) and the CUDA
side (tests, bench) use, so that both see the identical bf16 bits.

Recipe (the pages name no dataset; every input is synthetic):
  * the backward pass's incoming gradient dO: standard normal, bf16, from a
    generator of its own (``make_grad``);
  * shapes with shared K/V heads (``make_kv``): Q [B, H, N_q, d] then K and V
    [B, H_kv, N_kv, d], standard normal, in that order;
  * a ``torch.Generator`` on the CPU, seeded with ``seed``;
  * Q, K, V drawn in that order in float32 with the distribution the workload
    names, then rounded to bf16 (round-to-nearest-even, torch's conversion);
  * for the long-context stress workload, 1% of the key rows of each (b, h)
    (``round(0.01 * N)`` distinct positions from a seeded permutation, heads
    in (b, h) order) are multiplied by 8 after rounding; x8 is exact in bf16.

The named workloads are the five shapes the forward pass is specified on:
N = 256 (d 64), 1024 (d 64), 4096 (d 128), the 8k-context prefill shape
(B=1, H=32, N=8192, d=128, V uniform in [-1, 1]) and a 32k long-context
stress shape with spiky logits.
"""
from __future__ import annotations

import hashlib
import math
from dataclasses import dataclass

import torch

__all__ = ["Workload", "WORKLOADS", "workload", "make_inputs", "make_random", "make_grad", "KvWorkload",
           "KV_WORKLOADS", "kv_workload", "make_kv", "sha256_of"]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    q_dist: str = "normal"      # "normal" | "normal3" (std 3) | "uniform"
    k_dist: str = "normal"
    v_dist: str = "normal"
    spike_frac: float = 0.0     # fraction of key rows scaled by spike_mult
    spike_mult: float = 8.0
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> float:
        """Forward FLOPs counted as 4*B*H*N^2*d (the two N x N x d products)."""
        return 4.0 * self.B * self.H * self.N * self.N * self.d

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "H": self.H, "N": self.N, "d": self.d,
                "q": self.q_dist, "k": self.k_dist, "v": self.v_dist,
                "spike_frac": self.spike_frac, "seed": self.seed,
                "scale": "1/sqrt(d)", "causal": False}


WORKLOADS = [
    Workload("n256_d64", 1, 1, 256, 64, seed=1001),
    Workload("n1024_d64_b4h16", 4, 16, 1024, 64, seed=1002),
    Workload("n4096_d128_b2h16", 2, 16, 4096, 128, seed=1003),
    Workload("prefill8k_d128_h32", 1, 32, 8192, 128, v_dist="uniform", seed=1004),
    Workload("long32k_d128_h16_spiky", 1, 16, 32768, 128, q_dist="normal3",
             k_dist="normal3", spike_frac=0.01, seed=1005),
]


def workload(name_or_index) -> Workload:
    """Look a workload up by name or by 1-based position in ``WORKLOADS``."""
    if isinstance(name_or_index, int):
        return WORKLOADS[name_or_index - 1]
    for w in WORKLOADS:
        if w.name == name_or_index:
            return w
    raise KeyError(name_or_index)


def _draw(gen: torch.Generator, shape, dist: str) -> torch.Tensor:
    if dist == "normal":
        x = torch.randn(shape, generator=gen, dtype=torch.float32)
    elif dist == "normal3":
        x = torch.randn(shape, generator=gen, dtype=torch.float32) * 3.0
    elif dist == "uniform":
        x = torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    elif dist == "zeros":
        x = torch.zeros(shape, dtype=torch.float32)
    else:
        raise ValueError(dist)
    return x.to(torch.bfloat16)


def make_random(B: int, H: int, N: int, d: int, seed: int, q_dist="normal", k_dist="normal",
                v_dist="normal", spike_frac: float = 0.0, spike_mult: float = 8.0):
    """Draw bf16 Q, K, V [B, H, N, d] on the CPU from ``seed`` (recipe above)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed))
    shape = (B, H, N, d)
    q = _draw(gen, shape, q_dist)
    k = _draw(gen, shape, k_dist)
    v = _draw(gen, shape, v_dist)
    n_spikes = int(round(spike_frac * N))
    if n_spikes > 0:
        for b in range(B):
            for h in range(H):
                pos = torch.randperm(N, generator=gen)[:n_spikes]
                k[b, h, pos] = (k[b, h, pos].float() * spike_mult).to(torch.bfloat16)
    return q, k, v


def make_inputs(w: Workload):
    """Q, K, V (bf16, CPU) and the scale for a named workload."""
    q, k, v = make_random(w.B, w.H, w.N, w.d, w.seed, w.q_dist, w.k_dist, w.v_dist,
                          w.spike_frac, w.spike_mult)
    return q, k, v, w.scale


def make_grad(B: int, H: int, N: int, d: int, seed: int) -> torch.Tensor:
    """The incoming gradient dO of the backward pass: bf16 [B, H, N, d], standard
    normal, drawn on the CPU from its own generator seeded with ``seed + 7919``
    (so that it never repeats the Q, K, V stream of the same seed)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed) + 7919)
    return _draw(gen, (B, H, N, d), "normal")


@dataclass(frozen=True)
class KvWorkload:
    """A shape with shared K/V heads: Q [B, H, N_q, d], K/V [B, H_kv, N_kv, d]."""
    name: str
    B: int
    H: int
    H_kv: int
    N_q: int
    N_kv: int
    d: int
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def kv_bytes(self) -> int:
        """Bytes of K and V, read once by an exact kernel: the decode shape's traffic."""
        return 2 * self.B * self.H_kv * self.N_kv * self.d * 2

    @property
    def flops(self) -> float:
        return 4.0 * self.B * self.H * self.N_q * self.N_kv * self.d

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "H": self.H, "H_kv": self.H_kv, "N_q": self.N_q,
                "N_kv": self.N_kv, "d": self.d, "q": "normal", "k": "normal", "v": "normal", "seed": self.seed,
                "scale": "1/sqrt(d)", "causal": False}


# Decode against a long K/V cache with grouped heads (32 query heads on 8 K/V
# heads), one new token per sequence, batch 4.
KV_WORKLOADS = [
    KvWorkload("decode32k_gqa8_b4", 4, 32, 8, 1, 32768, 128, seed=2001),
]


def kv_workload(name: str) -> KvWorkload:
    for w in KV_WORKLOADS:
        if w.name == name:
            return w
    raise KeyError(name)


def make_kv(B: int, H: int, H_kv: int, N_q: int, N_kv: int, d: int, seed: int):
    """Q [B, H, N_q, d] and K, V [B, H_kv, N_kv, d], bf16, standard normal, drawn
    in that order on the CPU from ``seed``."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed))
    q = _draw(gen, (B, H, N_q, d), "normal")
    k = _draw(gen, (B, H_kv, N_kv, d), "normal")
    v = _draw(gen, (B, H_kv, N_kv, d), "normal")
    return q, k, v


def sha256_of(*tensors: torch.Tensor) -> str:
    """SHA-256 over the raw bytes of the given tensors, in order."""
    h = hashlib.sha256()
    for t in tensors:
        h.update(t.contiguous().view(torch.uint8).numpy().tobytes()
                 if t.dtype != torch.bfloat16 else
                 t.contiguous().view(torch.int16).numpy().tobytes())
    return h.hexdigest()
