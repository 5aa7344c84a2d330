"""Sequence split of the keys and values across devices (context parallelism).

Every rank of a process group holds all query rows and one contiguous shard
of the keys and values, for example a long sequence whose K/V cache does not
fit one device. The exchange step is the one the online softmax allows
("Flash Attention (FA1)", derivation steps 4-5):
  1. each rank computes the exact attention of its queries over its own key
     shard, a partial result (O_r normalised by its own l_r, and LSE_r);
  2. the ranks all-gather the partial results (one collective per output);
  3. each rank merges them, LSE = ln sum_r e^{LSE_r} and
     O = sum_r e^{LSE_r - LSE} O_r, into the attention over all keys.
Step 1 is fa_fwd_kv_f32 (O stays float32, so the exchange carries it
unrounded) and step 3 fa_merge_partials (which rounds O to bf16 once), both
CUDA kernels of this library; step 2 is torch.distributed: NCCL between GPUs,
or gloo, which gathers through host copies of the partial results. Nothing
here touches the data outside those calls.
"""
from __future__ import annotations

import math

import torch

__all__ = ["shard_bounds", "fa_fwd_cp"]


def shard_bounds(n_kv: int, world: int, rank: int):
    """[start, end) of rank's contiguous key shard: whole 128-key blocks, as
    even as the block count allows; every rank gets at least one key."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank / world size")
    if n_kv < world:
        raise ValueError(f"cannot split {n_kv} keys over {world} ranks")
    blocks = (n_kv + 127) // 128
    if blocks >= world:
        per, extra = divmod(blocks, world)
        start_blk = rank * per + min(rank, extra)
        end_blk = start_blk + per + (1 if rank < extra else 0)
        return min(n_kv, 128 * start_blk), min(n_kv, 128 * end_blk)
    per, extra = divmod(n_kv, world)          # fewer blocks than ranks: split keys evenly
    start = rank * per + min(rank, extra)
    return start, start + per + (1 if rank < extra else 0)


def _partial_cuda(q, k, v, scale):
    from . import fa
    return fa.fa_fwd_kv_f32(q, k, v, scale=scale)


def _merge_cuda(o_parts, lse_parts):
    from . import fa
    return fa.fa_merge_partials(o_parts, lse_parts)


def fa_fwd_cp(q, k_shard, v_shard, scale: float | None = None, group=None, partial_fn=None, merge_fn=None):
    """O and LSE of q over the keys of all ranks of ``group``.

    q: [B, H, N_q, d] (the same on every rank); k_shard, v_shard: this rank's
    [B, H_kv, N_kv_r, d] slice of the keys and values, in rank order along
    the sequence (see :func:`shard_bounds`). ``partial_fn(q, k, v, scale) ->
    (o, lse)`` and ``merge_fn(o_parts, lse_parts) -> (o, lse)`` default to the
    CUDA kernels; they are parameters only so that the exchange logic can be
    exercised on CPU process groups.
    """
    import torch.distributed as dist
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    world = dist.get_world_size(group)
    o_r, lse_r = (partial_fn or _partial_cuda)(q, k_shard, v_shard, scale)
    if o_r.dtype != torch.float32 and o_r.dtype != torch.float64:
        raise TypeError(f"partial O must stay float32 for the exchange, got {o_r.dtype}")
    o_r, lse_r = o_r.contiguous(), lse_r.contiguous()
    device = o_r.device
    # gloo gathers host tensors only: the partial results cross through host memory.
    via_host = device.type == "cuda" and dist.get_backend(group) == "gloo"
    if via_host:
        o_r, lse_r = o_r.cpu(), lse_r.cpu()
    o_list = [torch.empty_like(o_r) for _ in range(world)]
    l_list = [torch.empty_like(lse_r) for _ in range(world)]
    dist.all_gather(o_list, o_r, group=group)
    dist.all_gather(l_list, lse_r, group=group)
    o_parts, l_parts = torch.stack(o_list), torch.stack(l_list)
    if via_host:
        o_parts, l_parts = o_parts.to(device), l_parts.to(device)
    return (merge_fn or _merge_cuda)(o_parts, l_parts)
