"""Helpers for comparing the CUDA path with the oracle.

Tolerances (bf16 inputs, fp32 accumulation), measured against the float64
oracle on the identical bf16 inputs:
  O   max |err|                    <= 2e-2
  O   ||err||_F / ||O_ref||_F      <= 1e-2
  LSE max |err|                    <= 1e-3
  O   max |err| <= 2 x the max |err| of the bf16 materialise-path reference
      ("01 · 注意力为什么是 IO 瓶颈" §7: no worse than twice the baseline)
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

TOL_O_MAX = 2e-2
TOL_O_FRO = 1e-2
TOL_LSE_MAX = 1e-3


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def run_gpu(q, k, v, scale, device="cuda:0"):
    from exact_io_aware_34_gb300 import fa
    qd, kd, vd = (x.to(device) for x in (q, k, v))
    o, lse = fa.fa_fwd(qd, kd, vd, scale=scale)
    torch.cuda.synchronize(device)
    st, info = fa.fa_get_device_status()
    assert st == fa.FA_OK, (fa.fa_status_string(st), info)
    return o.cpu(), lse.cpu()


def errors(o_gpu, lse_gpu, O_ref, L_ref):
    og = to64(o_gpu)
    lg = to64(lse_gpu)
    e = og - O_ref
    return {
        "o_max": float(np.abs(e).max()) if e.size else 0.0,
        "o_fro": float(np.linalg.norm(e) / max(np.linalg.norm(O_ref), 1e-300)) if e.size else 0.0,
        "lse_max": float(np.abs(lg - L_ref).max()) if lg.size else 0.0,
        "finite": bool(np.isfinite(og).all() and np.isfinite(lg).all()),
    }


def check_full(q, k, v, scale, two_x_rule=True):
    """Whole-output parity (sizes the oracle evaluates in seconds)."""
    o, lse = run_gpu(q, k, v, scale)
    Q, K, V = (to64(x) for x in (q, k, v))
    O_ref, L_ref = oracle.attention(Q, K, V, scale)
    err = errors(o, lse, O_ref, L_ref)
    assert err["finite"], err
    assert err["o_max"] <= TOL_O_MAX, err
    assert err["o_fro"] <= TOL_O_FRO, err
    assert err["lse_max"] <= TOL_LSE_MAX, err
    if two_x_rule:
        On = oracle.naive_bf16_attention(Q, K, V, scale)
        err["naive_o_max"] = float(np.abs(On - O_ref).max())
        assert err["o_max"] <= 2 * err["naive_o_max"], err
    return err, o, lse


def sample_rows(B, H, N, n, seed=0):
    """(b, h, r) triples: tile edges, the last rows, and random rows."""
    rng = np.random.default_rng(seed)
    picks = set()
    edges = [0, 1, 127, 128, 255, 256, N - 129, N - 128, N - 1]
    for b in range(B):
        for h in (0, H - 1):
            for r in edges:
                if 0 <= r < N:
                    picks.add((b, h, r))
    while len(picks) < n:
        picks.add((int(rng.integers(B)), int(rng.integers(H)), int(rng.integers(N))))
    return np.array(sorted(picks), dtype=np.int64)


def check_sampled(q, k, v, scale, n_rows=256, seed=0, two_x_rule=True):
    """Full-size run on the GPU, compared with the oracle at sampled rows, plus
    properties every row must have (finite; each O row inside the column-wise
    range of V, as a convex combination of value rows)."""
    B, H, N, d = q.shape
    o, lse = run_gpu(q, k, v, scale)
    rows = sample_rows(B, H, N, n_rows, seed)
    O_ref, L_ref = oracle.attention_rows(q.float().numpy(), k.float().numpy(), v.float().numpy(), scale, rows)
    og = o[rows[:, 0], rows[:, 1], rows[:, 2]]
    lg = lse[rows[:, 0], rows[:, 1], rows[:, 2]]
    err = errors(og, lg, O_ref, L_ref)
    assert err["finite"], err
    assert err["o_max"] <= TOL_O_MAX, err
    assert err["o_fro"] <= TOL_O_FRO, err
    assert err["lse_max"] <= TOL_LSE_MAX, err
    if two_x_rule:
        On = oracle.naive_bf16_attention(q.float().numpy(), k.float().numpy(), v.float().numpy(), scale, rows)
        err["naive_o_max"] = float(np.abs(On - O_ref).max())
        assert err["o_max"] <= 2 * err["naive_o_max"], err
    of = o.float()
    assert torch.isfinite(of).all() and torch.isfinite(lse).all()
    vmin = v.float().amin(dim=2, keepdim=True)
    vmax = v.float().amax(dim=2, keepdim=True)
    slack = 1e-2 * (vmax - vmin) + 1e-6
    assert bool((of >= vmin - slack).all()) and bool((of <= vmax + slack).all())
    return err


# --- backward ------------------------------------------------------------------
# Tolerances for dQ, dK, dV (bf16 outputs), against the float64 backward oracle
# on the identical bf16 inputs and the oracle's forward O (rounded to bf16, as
# a forward pass hands it over) and LSE (float32):
#   max |err| <= 2 x the max |err| of the bf16 materialise-path backward
#               (the same "twice the baseline" rule as the forward, §7)
#   ||err||_F <= 1e-2 ||ref||_F + 1e-6 sqrt(size)   (bf16 output rounding is
#               2^-9 relative; the floor covers an all-zero reference, N = 1)
TOL_BWD_FRO = 1e-2


def oracle_forward_inputs(q, k, v, scale):
    """O (bf16) and LSE (float32) from the float64 forward oracle: the
    backward's O/LSE inputs come from the oracle, never from the CUDA path."""
    O, L = oracle.attention(to64(q), to64(k), to64(v), scale)
    return torch.from_numpy(O).to(torch.bfloat16), torch.from_numpy(L).to(torch.float32)


def run_gpu_bwd(q, k, v, o, do, lse, scale, device="cuda:0", stream=None):
    from exact_io_aware_34_gb300 import fa
    args = [x.to(device) for x in (q, k, v, o, do, lse)]
    dq, dk, dv = fa.fa_bwd(*args, scale=scale, stream=stream)
    torch.cuda.synchronize(device)
    st, info = fa.fa_get_device_status()
    assert st == fa.FA_OK, (fa.fa_status_string(st), info)
    return dq.cpu(), dk.cpu(), dv.cpu()


def bwd_errors(got, ref, naive=None):
    """Per-gradient error figures; ``got`` bf16 tensors, ``ref``/``naive`` float64."""
    out = {}
    for name, g, r, nv in zip(("dq", "dk", "dv"), got, ref, naive if naive is not None else (None,) * 3):
        g64 = to64(g) if isinstance(g, torch.Tensor) else g
        e = g64 - r
        out[name] = {
            "max": float(np.abs(e).max()),
            "fro": float(np.linalg.norm(e)),
            "ref_fro": float(np.linalg.norm(r)),
            "ref_max": float(np.abs(r).max()),
            "size": int(r.size),
            "finite": bool(np.isfinite(g64).all()),
        }
        if nv is not None:
            out[name]["naive_max"] = float(np.abs(nv - r).max())
    return out


def assert_bwd_within(err, two_x_rule=True):
    for name, e in err.items():
        assert e["finite"], (name, e)
        assert e["fro"] <= TOL_BWD_FRO * e["ref_fro"] + 1e-6 * np.sqrt(e["size"]), (name, e)
        if two_x_rule and "naive_max" in e:
            assert e["max"] <= 2 * e["naive_max"], (name, e)


def check_bwd_full(q, k, v, do, scale, two_x_rule=True):
    """Whole-gradient parity (sizes the oracle evaluates in seconds)."""
    o, lse = oracle_forward_inputs(q, k, v, scale)
    got = run_gpu_bwd(q, k, v, o, do, lse, scale)
    Q, K, V, dO = (to64(x) for x in (q, k, v, do))
    ref = oracle.attention_bwd(Q, K, V, dO, scale)
    naive = oracle.naive_bf16_attention_bwd(Q, K, V, dO, scale) if two_x_rule else None
    err = bwd_errors(got, ref, naive)
    assert_bwd_within(err, two_x_rule)
    return err, got


# --- whole-output parity at full size -------------------------------------------
# Every output row of a full-size workload against the oracle, evaluated by a
# pool of spawned single-threaded processes (one per host core): the inputs and
# the GPU's O and LSE go to .npy files that every worker maps read-only, and
# each task returns error statistics for one block of query rows of one head.
def _full_rows_task(args):
    folder, b, h, r0, r1, scale, two_x_rule = args
    import os as _os
    load = lambda n: np.load(_os.path.join(folder, n + ".npy"), mmap_mode="r")  # noqa: E731
    q, k, v, o, lse = (load(n) for n in ("q", "k", "v", "o", "lse"))
    Q = np.asarray(q[b:b + 1, h:h + 1, r0:r1], dtype=np.float64)
    K = np.asarray(k[b:b + 1, h:h + 1], dtype=np.float64)
    V = np.asarray(v[b:b + 1, h:h + 1], dtype=np.float64)
    O_ref, L_ref = oracle.attention(Q, K, V, scale)
    og = np.asarray(o[b:b + 1, h:h + 1, r0:r1], dtype=np.float64)
    lg = np.asarray(lse[b:b + 1, h:h + 1, r0:r1], dtype=np.float64)
    e = og - O_ref
    out = {
        "rows": r1 - r0,
        "o_max": float(np.abs(e).max()),
        "err_sq": float(np.sum(e * e)),
        "ref_sq": float(np.sum(O_ref * O_ref)),
        "lse_max": float(np.abs(lg - L_ref).max()),
        "finite": bool(np.isfinite(og).all() and np.isfinite(lg).all()),
    }
    if two_x_rule:
        On = oracle.naive_bf16_attention(Q, K, V, scale)
        out["naive_o_max"] = float(np.abs(On - O_ref).max())
    return out


def check_full_parallel(q, k, v, scale, folder, two_x_rule=True, row_block=1024, workers=None):
    """Full-size run on the GPU, then every output row compared with the
    oracle (and the bf16 materialise-path reference for the 2x rule) by a
    spawned process pool. Asserts the same tolerances as :func:`check_full`
    over all B*H*N rows and returns the aggregated figures."""
    import multiprocessing as mp
    import os
    B, H, N, d = q.shape
    o, lse = run_gpu(q, k, v, scale)
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("lse", lse)):
        np.save(os.path.join(folder, name + ".npy"), t.float().numpy())
    tasks = [(str(folder), b, h, r0, min(N, r0 + row_block), float(scale), two_x_rule)
             for b in range(B) for h in range(H) for r0 in range(0, N, row_block)]
    n = workers or len(os.sched_getaffinity(0))
    saved = {x: os.environ.get(x) for x in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")}
    for x in saved:
        os.environ[x] = "1"
    try:
        with mp.get_context("spawn").Pool(n) as pool:
            parts = pool.map(_full_rows_task, tasks, chunksize=1)
    finally:
        for x, val in saved.items():
            if val is None:
                os.environ.pop(x, None)
            else:
                os.environ[x] = val
    err = {
        "rows_checked": sum(p["rows"] for p in parts),
        "rows_total": B * H * N,
        "o_max": max(p["o_max"] for p in parts),
        "o_fro": float(np.sqrt(sum(p["err_sq"] for p in parts) / max(sum(p["ref_sq"] for p in parts), 1e-300))),
        "lse_max": max(p["lse_max"] for p in parts),
        "finite": all(p["finite"] for p in parts),
        "workers": n,
    }
    assert err["rows_checked"] == err["rows_total"], err
    assert err["finite"], err
    assert err["o_max"] <= TOL_O_MAX, err
    assert err["o_fro"] <= TOL_O_FRO, err
    assert err["lse_max"] <= TOL_LSE_MAX, err
    if two_x_rule:
        err["naive_o_max"] = max(p["naive_o_max"] for p in parts)
        assert err["o_max"] <= 2 * err["naive_o_max"], err
    return err
