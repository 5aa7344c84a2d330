"""Host-side logic of bench.py (CPU only): the max-over-ranks reduction with two
gloo ranks, clock parsing, peaks and the traffic record's source-hash check."""
import json
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    # per-rank summed step time: the job's time is the slowest rank's
    m = bench.reduce_max(10.0 + 5.0 * rank, w)
    out[rank] = m
    bench.barrier(w)
    dist.destroy_process_group()


def test_reduce_max_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as man:
        out = man.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        assert dict(out) == {0: 15.0, 1: 15.0}


def test_reduce_max_single_rank_is_identity():
    assert bench.reduce_max(3.25, 1) == 3.25


def test_clock_summary_parsing():
    c = bench.ClockSampler(0)
    c.out = "\n".join([
        "0, 1900, 2070, 900.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 1950, 2070, 1100.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 2000, 2070, 1200.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
    ])
    s = c.summary()
    assert s["sm_mhz"] == 1950 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 3


def test_peaks_and_traffic(tmp_path, monkeypatch):
    peaks, src = bench.load_peaks()
    assert peaks["bf16_tflops"] > 100 and src in ("measured", "fallback")
    rec = {"prefill8k_d128_h32": {"kernel_source_hash": bench.kernel_source_hash(), "dram_bytes_per_launch": 123}}
    p = tmp_path / "t.json"
    p.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(p))
    assert bench.load_traffic("prefill8k_d128_h32") == 123
    rec["prefill8k_d128_h32"]["kernel_source_hash"] = "stale"
    p.write_text(json.dumps(rec))
    assert bench.load_traffic("prefill8k_d128_h32") is None


def test_warmup_floor():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_clock_summary_nvml_samples():
    c = bench.ClockSampler(0)
    c.samples = [(1900.0, 900.0, 0x4), (1950.0, 1000.0, 0), (2000.0, 1100.0, 0x8)]
    c.max_mhz = 2070.0
    s = c.summary()
    assert s["sm_mhz"] == 1950.0 and s["sm_max_mhz"] == 2070.0 and s["source"] == "nvml"
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"] and s["samples"] == 3


def test_cpu_baselines_of_the_next_rows():
    """The backward and decode oracle timings return well-formed records (tiny samples)."""
    import bench
    rb = bench.cpu_baseline_bwd("n256_d64", target_s=0.5)
    assert rb["kind"] == "oracle" and rb["unit"] == "TFLOP/s" and rb["value"] > 0 and rb["cores"] >= 1
    rd = bench.cpu_baseline_decode("decode32k_gqa8_b4")
    assert rd["kind"] == "oracle" and rd["unit"] == "GB/s" and rd["value"] > 0


def test_cpu_baseline_single_core():
    """The one-core oracle timing of a small configuration is a well-formed record."""
    import bench
    r = bench.cpu_baseline_single_core("n256_d64", target_s=0.2)
    assert r["kind"] == "oracle" and r["cores"] == 1 and r["unit"] == "TFLOP/s" and r["value"] > 0
    assert r["workload"] == "n256_d64"


def test_source_hash_ignores_comments_only():
    """The DRAM records are keyed by a hash of the kernel sources' code: an
    edit of comments or layout keeps it, an edit of code changes it."""
    a = "int f(int x) {\n  // one\n  return x + 1; /* two\n lines */\n}\n"
    b = "int f(int x) {   return x + 1;\n\n}  // other words\n"
    c = "int f(int x) {\n  return x + 2;\n}\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    assert "asm(\"mov.b32 %0, %1;\")" in bench._code_only('asm("mov.b32 %0, %1;") // note')


def test_committed_traffic_records_match_their_profiles():
    """Each record of profiles/dram_traffic.json adds up, and the ncu summary it
    comes from names the same kernel-sources hash. Where the record is current
    for the forward, its DRAM bytes are within a factor 1.5 of the algorithmic
    O(N d) bytes (inputs once, outputs once), far below the N^2 traffic of
    materialised scores."""
    with open(bench.TRAFFIC_FILE) as f:
        rec = json.load(f)
    summaries = {
        "prefill8k_d128_h32": "dram_traffic_all_workloads.md",
        "n256_d64": "dram_traffic_all_workloads.md",
        "n1024_d64_b4h16": "dram_traffic_all_workloads.md",
        "n4096_d128_b2h16": "dram_traffic_all_workloads.md",
        "long32k_d128_h16_spiky": "dram_traffic_all_workloads.md",
        "prefill8k_d128_h32:bwd": "fa_bwd_kernels_prefill8k_d128.md",
        "decode32k_gqa8_b4": "fa_decode_kernel_decode32k_gqa8.md",
        "prefill8k_d128_h32:comparator": "dram_traffic_all_workloads.md",
    }
    assert set(rec) == set(summaries)
    for key, md in summaries.items():
        e = rec[key]
        assert e["dram_bytes_read"] + e["dram_bytes_write"] == e["dram_bytes_per_launch"], key
        with open(os.path.join(os.path.dirname(bench.TRAFFIC_FILE), md)) as f:
            assert e["kernel_source_hash"] in f.read(), (key, md)
    from exact_io_aware_34_gb300 import inputs
    for w in inputs.WORKLOADS:
        if w.name not in rec or bench.load_traffic(w.name) is None:
            continue
        reads = rec[w.name]["dram_bytes_read"]
        inputs_bytes = 3 * w.B * w.H * w.N * w.d * 2          # Q, K, V once
        assert inputs_bytes / 1.05 <= reads <= 1.05 * inputs_bytes + (1 << 20), w.name
        assert rec[w.name]["dram_bytes_per_launch"] <= 1.5 * w.B * w.H * w.N * (8 * w.d + 4) + (1 << 20), w.name


def test_head_shard_covers_every_head_once():
    for H in (1, 2, 5, 16, 32, 33):
        for world in (1, 2, 3, 4, 8):
            if H < world:
                with pytest.raises(ValueError):
                    bench.head_shard(H, world, 0)
                continue
            parts = [bench.head_shard(H, world, r) for r in range(world)]
            assert parts[0][0] == 0 and parts[-1][1] == H
            assert all(parts[r][1] == parts[r + 1][0] for r in range(world - 1))
            sizes = [b - a for a, b in parts]
            assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1


def _shard_rank(rank, world, port, out):
    """Two gloo ranks split the heads of the 8k prefill workload: each takes its
    range, the slowest rank's time is the job's, and the job's FLOPs are the
    workload's, whatever the split."""
    import torch.distributed as dist
    from exact_io_aware_34_gb300 import inputs
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = inputs.workload("prefill8k_d128_h32")
    h0, h1 = bench.head_shard(w.H, world, rank)
    my_flops = 4.0 * w.B * (h1 - h0) * w.N * w.N * w.d
    total = bench.reduce_max(0.0, world)          # barrier-like exchange
    t = bench.reduce_max(1.0 + rank, world)       # per-rank seconds; the job takes the slowest
    import torch
    flops = torch.tensor([my_flops], dtype=torch.float64)
    dist.all_reduce(flops)
    out[rank] = (h0, h1, t, float(flops.item()), total)
    dist.destroy_process_group()


def test_head_shard_two_gloo_ranks():
    from exact_io_aware_34_gb300 import inputs
    world = 2
    with mp.Manager() as man:
        out = man.dict()
        mp.spawn(_shard_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    w = inputs.workload("prefill8k_d128_h32")
    assert res[0][:2] == (0, 16) and res[1][:2] == (16, 32)
    assert res[0][2] == res[1][2] == 2.0
    assert res[0][3] == w.flops          # the ranks' shares add up to the whole workload


def test_gpus_flag_relaunches_under_torchrun(monkeypatch):
    calls = []
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(bench.subprocess, "call", lambda cmd: calls.append(cmd) or 0)
    assert bench.main(["--gpus", "4", "--steps", "3", "--warmup", "3", "--shard", "heads"]) == 0
    cmd = calls[0]
    assert cmd[1:4] == ["-m", "torch.distributed.run", "--nnodes=1"] and "--nproc-per-node=4" in cmd
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert cmd[cmd.index(os.path.abspath(bench.__file__)) + 1:] == ["--gpus", "4", "--steps", "3", "--warmup", "3", "--shard", "heads"]


def test_gpus_flag_must_match_world_size(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    with pytest.raises(SystemExit):
        bench.main(["--gpus", "4"])


def test_reference_arm_prints_its_line():
    """--impl reference times the float64 oracle on the host cores (no GPU) and
    prints one JSON line with the contract's keys, its own cpu_baseline and an
    e2e that moves no bytes between host and device."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3", "--ref-step-s", "0.2"], cwd=root, capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 3
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT and d["higher_is_better"] is True
    assert d["config"]["workload"] == "prefill8k_d128_h32"
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] == d["value"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
