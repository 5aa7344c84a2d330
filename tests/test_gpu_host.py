"""The forward pass on host buffers (fa_fwd_host) through the C ABI (needs a GB300).

Each head's result must be fa_fwd's bit for bit (the same kernel runs on every
head group), so the oracle comparison of the fused kernel carries over; one
case is also checked against the oracle directly.
"""
from __future__ import annotations

import math

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


def run_host(q, k, v, scale, num_chunks=0, workspace=None, stream=None):
    qh, kh, vh = (x.contiguous().pin_memory() for x in (q, k, v))
    oh, lh = fa.fa_fwd_host(qh, kh, vh, scale=scale, num_chunks=num_chunks, workspace=workspace, stream=stream)
    torch.cuda.synchronize()
    st, info = fa.fa_get_device_status()
    assert st == fa.FA_OK, (fa.fa_status_string(st), info)
    return oh, lh


def bits_equal(a, b):
    return torch.equal(a.contiguous().view(torch.int16), b.contiguous().view(torch.int16))


@pytest.mark.parametrize("num_chunks", [0, 1, 3, 16])
@pytest.mark.parametrize("B,H,N,d", [(2, 3, 700, 128), (1, 5, 129, 64), (1, 1, 300, 128), (3, 4, 1024, 64)])
def test_host_path_equals_device_path(B, H, N, d, num_chunks):
    q, k, v = inputs.make_random(B, H, N, d, seed=B * 100 + H * 10 + N + d)
    scale = 1 / math.sqrt(d)
    oh, lh = run_host(q, k, v, scale, num_chunks)
    od, ld = parity.run_gpu(q, k, v, scale)
    assert bits_equal(oh, od)
    assert torch.equal(lh, ld)


def test_host_path_matches_oracle():
    q, k, v = inputs.make_random(1, 4, 520, 128, seed=77)
    oh, lh = run_host(q, k, v, 0.09, num_chunks=3)
    O_ref, L_ref = oracle.attention(parity.to64(q), parity.to64(k), parity.to64(v), 0.09)
    err = parity.errors(oh, lh, O_ref, L_ref)
    assert err["finite"] and err["o_max"] <= parity.TOL_O_MAX and err["o_fro"] <= parity.TOL_O_FRO, err
    assert err["lse_max"] <= parity.TOL_LSE_MAX, err


def test_back_to_back_calls_reuse_the_workspace():
    """Two calls on one stream with one workspace: the second call's uploads
    wait for the first call's kernels and downloads."""
    ws = torch.empty(fa.fa_fwd_host_workspace_bytes(2, 4, 2048, 128), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    outs = []
    ins = [inputs.make_random(2, 4, 2048, 128, seed=90 + r) for r in range(2)]
    for q, k, v in ins:
        qh, kh, vh = (x.pin_memory() for x in (q, k, v))
        outs.append(fa.fa_fwd_host(qh, kh, vh, scale=0.1, num_chunks=4, workspace=ws, stream=s))
    s.synchronize()
    for (q, k, v), (oh, lh) in zip(ins, outs):
        od, ld = parity.run_gpu(q, k, v, 0.1)
        assert bits_equal(oh, od)
        assert torch.equal(lh, ld)


def test_host_path_rejects_device_tensors():
    q, k, v = inputs.make_random(1, 1, 128, 64, seed=5)
    with pytest.raises(ValueError):
        fa.fa_fwd_host(q.cuda(), k, v)


def test_pageable_host_buffers():
    """Unpinned host memory: slower copies, the same result."""
    q, k, v = inputs.make_random(1, 3, 333, 64, seed=81)
    oh, lh = fa.fa_fwd_host(q.contiguous(), k.contiguous(), v.contiguous(), scale=0.125, num_chunks=2,
                            oh=torch.empty(q.shape, dtype=torch.bfloat16), lseh=torch.empty((1, 3, 333)))
    torch.cuda.synchronize()
    od, ld = parity.run_gpu(q, k, v, 0.125)
    assert bits_equal(oh, od)
    assert torch.equal(lh, ld)


def test_full_workload_in_the_bench_configuration():
    """prefill8k_d128_h32 through fa_fwd_host with the automatic head groups, as the bench's e2e
    times it: bit for bit fa_fwd's result (which the full-size parity tests check against the
    oracle on sampled rows)."""
    w = inputs.workload("prefill8k_d128_h32")
    q, k, v, scale = inputs.make_inputs(w)
    oh, lh = run_host(q, k, v, scale)
    od, ld = parity.run_gpu(q, k, v, scale)
    assert bits_equal(oh, od)
    assert torch.equal(lh, ld)


def test_concurrent_calls_from_two_threads():
    """Two host threads, each with its own stream and workspace, call at the same
    time (the library serialises its enqueue and reuses its events): every result
    is still fa_fwd's bit for bit."""
    import threading
    cases = [inputs.make_random(1, 6, 900, 128, seed=95 + i) for i in range(2)]
    results = [None, None]
    errors = []

    def worker(i):
        try:
            torch.cuda.set_device(0)
            q, k, v = cases[i]
            s = torch.cuda.Stream()
            ws = torch.empty(fa.fa_fwd_host_workspace_bytes(1, 6, 900, 128), dtype=torch.uint8, device="cuda")
            outs = []
            for _ in range(5):
                outs.append(fa.fa_fwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), scale=0.08, num_chunks=3,
                                           workspace=ws, stream=s))
            s.synchronize()
            results[i] = outs
        except Exception as e:     # surfaced below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i, (q, k, v) in enumerate(cases):
        od, ld = parity.run_gpu(q, k, v, 0.08)
        for oh, lh in results[i]:
            assert bits_equal(oh, od)
            assert torch.equal(lh, ld)


def test_host_path_negative_scale():
    """scale < 0 through the host-buffer entry point: the same bits as fa_fwd."""
    q, k, v = inputs.make_random(1, 4, 600, 128, seed=81)
    oh, lh = run_host(q, k, v, -0.1, num_chunks=2)
    od, ld = parity.run_gpu(q, k, v, -0.1)
    assert bits_equal(oh, od)
    assert torch.equal(lh, ld)


@pytest.mark.parametrize("num_chunks", [3, 7, 16])
def test_host_groups_follow_the_whole_problems_shared_units(num_chunks):
    """40 heads of 1024 rows: fa_fwd runs one whole round of units and has CTA
    pairs share the last 8 (heads 38 and 39). The head groups of fa_fwd_host are
    separate launches with fewer units each; they still share exactly those
    units, so every head's result is fa_fwd's, bit for bit."""
    q, k, v = inputs.make_random(1, 40, 1024, 128, seed=91)
    oh, lh = run_host(q, k, v, 0.088, num_chunks=num_chunks)
    od, ld = parity.run_gpu(q, k, v, 0.088)
    assert bits_equal(oh, od)
    assert torch.equal(lh, ld)
