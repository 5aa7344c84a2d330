"""Shared K/V heads and short query blocks (fa_fwd_kv) against the oracle, through
the C ABI (needs a GB300).

Reference: ``oracle.attention_gqa`` (query head h attends to K/V head
h // (H / H_kv)); the "twice the baseline" rule compares with the bf16
materialise-path reference evaluated on K/V repeated per query head.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_34_gb300 import fa, inputs
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from exact_io_aware_34_gb300 import build
    build.build()
    fa.load_library()


def run_kv(q, k, v, scale, num_splits=0):
    o, lse = fa.fa_fwd_kv(q.cuda(), k.cuda(), v.cuda(), scale=scale, num_splits=num_splits)
    torch.cuda.synchronize()
    st, info = fa.fa_get_device_status()
    assert st == fa.FA_OK, (fa.fa_status_string(st), info)
    return o.cpu(), lse.cpu()


def check_kv(q, k, v, scale, num_splits=0, two_x_rule=True):
    o, lse = run_kv(q, k, v, scale, num_splits)
    Q, K, V = (parity.to64(x) for x in (q, k, v))
    O_ref, L_ref = oracle.attention_gqa(Q, K, V, scale)
    err = parity.errors(o, lse, O_ref, L_ref)
    assert err["finite"], err
    assert err["o_max"] <= parity.TOL_O_MAX, err
    assert err["o_fro"] <= parity.TOL_O_FRO, err
    assert err["lse_max"] <= parity.TOL_LSE_MAX, err
    if two_x_rule:
        G = q.shape[1] // k.shape[1]
        On = oracle.naive_bf16_attention(Q, np.repeat(K, G, axis=1), np.repeat(V, G, axis=1), scale)
        err["naive_o_max"] = float(np.abs(On - O_ref).max())
        assert err["o_max"] <= 2 * err["naive_o_max"], err
    return err, o, lse


# --- short query blocks (the packed, split-key kernel) ------------------------------
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N_q,G", [(1, 1), (1, 8), (3, 4), (16, 8), (64, 2), (128, 1), (100, 4)])
@pytest.mark.parametrize("N_kv", [1, 100, 129, 1000])
def test_short_queries(d, N_q, G, N_kv):
    H_kv = 2
    q, k, v = inputs.make_kv(2, G * H_kv, H_kv, N_q, N_kv, d, seed=N_q * 131 + G * 17 + N_kv + d)
    err, _, _ = check_kv(q, k, v, 1 / math.sqrt(d), two_x_rule=N_kv >= 64)
    print(d, N_q, G, N_kv, err)


@pytest.mark.parametrize("num_splits", [1, 2, 3, 7, 64])
def test_forced_splits(num_splits):
    """Every split count gives the oracle's result (the merge of partial results)."""
    q, k, v = inputs.make_kv(1, 16, 4, 5, 4000, 128, seed=300 + num_splits)
    err, o, lse = check_kv(q, k, v, 1 / math.sqrt(128), num_splits=num_splits)
    print(num_splits, fa.fa_fwd_kv_workspace_bytes(1, 16, 4, 5, 4000, 128, num_splits), err)


def test_splits_agree_with_each_other():
    q, k, v = inputs.make_kv(2, 8, 2, 1, 3000, 64, seed=310)
    o1, l1 = run_kv(q, k, v, 0.125, num_splits=1)
    o5, l5 = run_kv(q, k, v, 0.125, num_splits=5)
    assert float((o1.float() - o5.float()).abs().max()) <= 1e-2
    assert float((l1 - l5).abs().max()) <= 1e-4


def test_spiky_keys_with_splits():
    """Large logits and spiky keys, so the splits' maxima differ widely."""
    q, k, v = inputs.make_kv(1, 8, 1, 4, 2048, 128, seed=320)
    q = (q.float() * 3).to(torch.bfloat16)
    k = (k.float() * 3).to(torch.bfloat16)
    k[0, 0, 1500] = (k[0, 0, 1500].float() * 8).to(torch.bfloat16)
    check_kv(q, k, v, 1 / math.sqrt(128), num_splits=6)


# --- long query blocks with shared K/V heads ----------------------------------------
# num_splits = 1 takes the fused forward kernel; 0 (at these few heads) and
# explicit counts take the short-query kernel with 128-row query tiles and a
# key split.
@pytest.mark.parametrize("num_splits", [1, 0, 5])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N_q,N_kv,G", [(300, 300, 4), (1000, 700, 2), (129, 2000, 8), (257, 129, 1)])
def test_long_queries(d, N_q, N_kv, G, num_splits):
    q, k, v = inputs.make_kv(1, 2 * G, 2, N_q, N_kv, d, seed=N_q + N_kv + G + d)
    check_kv(q, k, v, 1 / math.sqrt(d), num_splits=num_splits)


def test_long_query_split_is_chosen_for_few_heads():
    """A chunk of 512 queries of 8 heads against 32k keys: the automatic
    choice is a key split (the fused kernel would fill 16 SMs)."""
    q, k, v = inputs.make_kv(1, 8, 2, 512, 32768, 128, seed=335)
    splits = fa.fa_fwd_kv_num_splits(1, 8, 2, 512, 32768, 128)
    assert splits > 1
    err, o, lse = check_kv(q, k, v, 1 / math.sqrt(128))
    o1, l1 = run_kv(q, k, v, 1 / math.sqrt(128), num_splits=1)
    assert float((o.float() - o1.float()).abs().max()) <= 1e-2
    assert float((lse - l1).abs().max()) <= 1e-4
    print(splits, err)


def test_kv_heads_equal_reduces_to_fa_fwd():
    """H_kv = H and N_q = N_kv with one split: the same result as fa_fwd, bit for bit."""
    q, k, v = inputs.make_random(1, 4, 700, 128, seed=330)
    o1, l1 = run_kv(q, k, v, 0.09, num_splits=1)
    o2, l2 = parity.run_gpu(q, k, v, 0.09)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


# --- the decode workload the bench times ---------------------------------------------
def test_decode_workload_full():
    w = inputs.kv_workload("decode32k_gqa8_b4")
    q, k, v = inputs.make_kv(w.B, w.H, w.H_kv, w.N_q, w.N_kv, w.d, w.seed)
    err, _, _ = check_kv(q, k, v, w.scale)
    print(w.name, fa.fa_fwd_kv_num_splits(w.B, w.H, w.H_kv, w.N_q, w.N_kv, w.d), err)


def test_decode_million_keys():
    """One query row per head against 1,000,003 keys (7813 key blocks, the
    last ragged) with 4 query heads on one K/V head: every output row against
    the oracle (the key split merges ranges of about 900 blocks)."""
    q, k, v = inputs.make_kv(1, 4, 1, 1, 1_000_003, 128, seed=390)
    err, _, _ = check_kv(q, k, v, 1 / math.sqrt(128), two_x_rule=False)
    print(fa.fa_fwd_kv_num_splits(1, 4, 1, 1, 1_000_003, 128), err)


# --- failure path and rejections ---------------------------------------------------
@pytest.mark.parametrize("N_q", [2, 300])
@pytest.mark.parametrize("drop", [0, 1, 4])
def test_kv_dropped_load_times_out_cleanly(drop, N_q):
    q, k, v = (x.cuda() for x in inputs.make_kv(1, 8, 2, N_q, 2000, 128, seed=340 + drop))
    o = torch.zeros_like(q)
    lse = torch.zeros(1, 8, N_q, device="cuda")
    ws = torch.empty(fa.fa_fwd_kv_workspace_bytes(1, 8, 2, N_q, 2000, 128, 3), dtype=torch.uint8, device="cuda")
    st = fa.fa_fwd_kv_fault_test(q, k, v, o, lse, 0.1, 3, ws, drop, 20_000_000)
    assert st == fa.FA_OK
    st, info = fa.fa_get_device_status()
    assert st == fa.FA_ERR_TIMEOUT, (st, info)
    assert info[0] in (10, 11, 12)
    assert fa.fa_get_device_status()[0] == fa.FA_OK
    check_kv(q.cpu(), k.cpu(), v.cpu(), 0.1, num_splits=3)


def test_kv_small_workspace_rejected():
    q, k, v = (x.cuda() for x in inputs.make_kv(1, 8, 2, 1, 4000, 128, seed=350))
    need = fa.fa_fwd_kv_workspace_bytes(1, 8, 2, 1, 4000, 128, 4)
    ws = torch.empty(need - 128, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError):
        fa.fa_fwd_kv(q, k, v, num_splits=4, workspace=ws)


# --- merging partial results (the exchange step of a sequence split) ----------------
def test_merge_partials_matches_oracle():
    rng = np.random.default_rng(360)
    P, rows, d = 5, 300, 128
    o_parts = torch.from_numpy(rng.standard_normal((P, 3, rows // 3, d)).astype(np.float32))
    lse_parts = torch.from_numpy((rng.standard_normal((P, 3, rows // 3)) * 20).astype(np.float32))
    o, lse = fa.fa_merge_partials(o_parts.cuda(), lse_parts.cuda())
    torch.cuda.synchronize()
    O_ref, L_ref = oracle.merge_partials(o_parts.double().numpy(), lse_parts.double().numpy())
    assert float(np.abs(o.float().cpu().numpy() - O_ref).max()) <= 2 ** -8 * float(np.abs(O_ref).max()) + 1e-6
    assert float(np.abs(lse.cpu().numpy() - L_ref).max()) <= 1e-4


# --- float32 partial results (the exchange format of a sequence split) -------------
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N_q,N_kv,splits", [(1, 1000, 0), (16, 4096, 1), (100, 777, 3), (300, 2000, 2),
                                             (300, 2000, 1)])
def test_kv_f32_partial_result(d, N_q, N_kv, splits):
    """fa_fwd_kv_f32 keeps O in float32: within the parity tolerances of the
    oracle, and, rounded to bf16, bit for bit fa_fwd_kv's O on the same kernel
    path (the short-query kernel with the same key split)."""
    q, k, v = inputs.make_kv(1, 8, 2, N_q, N_kv, d, seed=380 + N_q + d)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    s = 1 / math.sqrt(d)
    o32, l32 = fa.fa_fwd_kv_f32(qd, kd, vd, scale=s, num_splits=splits)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status()[0] == fa.FA_OK
    assert o32.dtype == torch.float32
    O_ref, L_ref = oracle.attention_gqa(*(parity.to64(x) for x in (q, k, v)), s)
    err = parity.errors(o32.cpu(), l32.cpu(), O_ref, L_ref)
    assert err["finite"] and err["o_max"] <= parity.TOL_O_MAX and err["o_fro"] <= parity.TOL_O_FRO, err
    assert err["lse_max"] <= parity.TOL_LSE_MAX, err
    # the same kernel with bf16 output: force the short-query route for long queries
    same_route = splits if (N_q <= 128 or splits != 1) else None
    if same_route is not None:
        o16, l16 = fa.fa_fwd_kv(qd, kd, vd, scale=s, num_splits=same_route)
        torch.cuda.synchronize()
        assert torch.equal(o32.to(torch.bfloat16).view(torch.int16), o16.view(torch.int16))
        assert torch.equal(l32, l16)
    print(d, N_q, N_kv, splits, err)


def _cp_rank(rank, world, port, folder):
    """One rank of a sequence split on the one GPU: its key shard through
    fa_fwd_kv_f32, the gather over gloo through host copies, the merge on the
    GPU (the library's fa_fwd_cp end to end)."""
    import os
    import torch.distributed as dist
    from exact_io_aware_34_gb300 import build, cp
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    build.build()
    fa.load_library()
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q, k, v = inputs.make_kv(1, 8, 2, 300, 5000, 128, seed=390 + world)
        s0, s1 = cp.shard_bounds(5000, world, rank)
        dev = torch.device("cuda", 0)
        o, lse = cp.fa_fwd_cp(q.to(dev), k[:, :, s0:s1].contiguous().to(dev), v[:, :, s0:s1].contiguous().to(dev),
                              scale=0.09)
        torch.cuda.synchronize(dev)
        assert fa.fa_get_device_status()[0] == fa.FA_OK
        torch.save({"o": o.cpu(), "lse": lse.cpu()}, os.path.join(folder, f"rank{rank}.pt"))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_fa_fwd_cp_across_gloo_ranks_on_one_gpu(world, tmp_path):
    """cp.fa_fwd_cp itself, run by ``world`` processes that share the GPU (each
    launches only its own independent kernels; nothing waits on another rank's
    kernel): every rank's merged result equals attention over all keys."""
    import socket
    import torch.multiprocessing as tmp
    from exact_io_aware_34_gb300 import cp  # noqa: F401
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    tmp.start_processes(_cp_rank, args=(world, port, str(tmp_path)), nprocs=world, start_method="spawn", join=True)
    q, k, v = inputs.make_kv(1, 8, 2, 300, 5000, 128, seed=390 + world)
    O_ref, L_ref = oracle.attention_gqa(parity.to64(q), parity.to64(k), parity.to64(v), 0.09)
    first = None
    for r in range(world):
        res = torch.load(tmp_path / f"rank{r}.pt")
        err = parity.errors(res["o"], res["lse"], O_ref, L_ref)
        assert err["finite"] and err["o_max"] <= parity.TOL_O_MAX and err["o_fro"] <= parity.TOL_O_FRO, err
        assert err["lse_max"] <= parity.TOL_LSE_MAX, err
        if first is None:
            first = res
        else:   # every rank merges the same gathered partials
            assert torch.equal(res["o"].view(torch.int16), first["o"].view(torch.int16))
        print(world, r, err)


@pytest.mark.parametrize("world", [2, 3, 8])
def test_sequence_split_emulated_on_one_gpu(world):
    """The ranks of a sequence split, run one after another on one GPU: each
    shard's float32 partial result from fa_fwd_kv_f32, then one
    fa_merge_partials call, against the oracle over all keys."""
    from exact_io_aware_34_gb300 import cp
    q, k, v = inputs.make_kv(1, 8, 2, 300, 5000, 128, seed=370 + world)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    parts = []
    for r in range(world):
        s0, s1 = cp.shard_bounds(5000, world, r)
        parts.append(fa.fa_fwd_kv_f32(qd, kd[:, :, s0:s1].contiguous(), vd[:, :, s0:s1].contiguous(), scale=0.09))
    o, lse = fa.fa_merge_partials(torch.stack([p[0] for p in parts]), torch.stack([p[1] for p in parts]))
    torch.cuda.synchronize()
    O_ref, L_ref = oracle.attention_gqa(parity.to64(q), parity.to64(k), parity.to64(v), 0.09)
    err = parity.errors(o.cpu(), lse.cpu(), O_ref, L_ref)
    assert err["finite"] and err["o_max"] <= parity.TOL_O_MAX and err["o_fro"] <= parity.TOL_O_FRO, err
    assert err["lse_max"] <= parity.TOL_LSE_MAX, err
    print(world, err)


@pytest.mark.parametrize("N_q,N_kv,splits", [(1, 1000, 0), (16, 4096, 3), (300, 700, 1), (300, 5000, 0)])
def test_negative_scale(N_q, N_kv, splits):
    """scale < 0 on both kernels of fa_fwd_kv (short queries with a key split,
    and the fused kernel for long query blocks)."""
    q, k, v = inputs.make_kv(1, 8, 2, N_q, N_kv, 128, seed=60 + N_q)
    err, _, _ = check_kv(q, k, v, -0.11, num_splits=splits)
    print(N_q, N_kv, splits, err)
