"""The sequence-split exchange (exact_io_aware_34_gb300.cp) across two gloo ranks on
the CPU: each rank takes its key shard, computes its partial result, the ranks
all-gather, and the merge reproduces attention over all keys. The partial and
merge steps are the oracle here (the CUDA kernels need a GPU); the shard
bookkeeping and the collective are the product code."""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from exact_io_aware_34_gb300 import cp, inputs


def test_shard_bounds_cover_the_sequence():
    for n_kv in (1, 2, 127, 128, 129, 1000, 8192, 32768 + 5):
        for world in (1, 2, 3, 4, 8):
            if n_kv < world:
                with pytest.raises(ValueError):
                    cp.shard_bounds(n_kv, world, 0)
                continue
            b = [cp.shard_bounds(n_kv, world, r) for r in range(world)]
            assert b[0][0] == 0 and b[-1][1] == n_kv
            assert all(b[r][1] == b[r + 1][0] for r in range(world - 1))
            assert all(e > s for s, e in b)
            if (n_kv + 127) // 128 >= world:   # whole blocks except the last shard's end
                assert all(s % 128 == 0 for s, _ in b)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_partial(q, k, v, scale):
    O, L = oracle.attention_gqa(q.double().numpy(), k.double().numpy(), v.double().numpy(), scale)
    return torch.from_numpy(O), torch.from_numpy(L)


def _oracle_merge(o_parts, lse_parts):
    O, L = oracle.merge_partials(o_parts.double().numpy(), lse_parts.double().numpy())
    return torch.from_numpy(O), torch.from_numpy(L)


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q, k, v = inputs.make_kv(1, 8, 2, 5, 700, 64, seed=909)
        s0, s1 = cp.shard_bounds(700, world, rank)
        o, lse = cp.fa_fwd_cp(q.float(), k[:, :, s0:s1].float(), v[:, :, s0:s1].float(), scale=0.125,
                              partial_fn=_oracle_partial, merge_fn=_oracle_merge)
        O_ref, L_ref = oracle.attention_gqa(q.double().numpy(), k.double().numpy(), v.double().numpy(), 0.125)
        out[rank] = float(max(np.abs(o.numpy() - O_ref).max(), np.abs(lse.numpy() - L_ref).max()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_sequence_split_across_gloo_ranks(world):
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
    assert sorted(out.keys()) == list(range(world))
    # the partial O travel as float32 (the exchange format), so the agreement is float32-sized
    assert max(out.values()) < 1e-6, dict(out)
