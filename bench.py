"""Benchmark of the fused exact-attention forward pass.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference] [--workload NAME]

One step = one call of fa_fwd over the whole workload (every (b, h) and
query row). The default workload is the 8k-context prefill shape
(B=1, H=32, N=8192, d=128, bf16, seeded synthetic inputs). Metric: forward
TFLOP/s counted as 4*B*H*N^2*d / time. Rank 0 prints one JSON line.

Timing: W untimed warm-up steps; then K steps, each bracketed by CUDA events
on the launching stream, with the L2 cache flushed (a 512 MB write) before
every step, outside the events; barrier + synchronize around the timed
region; the max over ranks of the summed device time. For N > 1 (launched by
torchrun; ``--gpus N`` without a torchrun environment starts N ranks itself)
every rank runs its own copy of the workload (independent problems, no
collective on the data path): weak scaling. With ``--shard heads`` the ranks
split the heads of one workload instead (each rank its contiguous range of
heads, still no collective): strong scaling, value = the workload's FLOPs /
the slowest rank's time.

The same run also times the backward pass (fa_bwd, two launches) on the
same workload and reports it under "bwd" (skip with --no-bwd), and a decode
shape with shared K/V heads (fa_fwd_kv: B=4, 32 query heads on 8 K/V heads,
one query row against 32768 keys, d=128) under "decode" in K/V GB/s against
the HBM roofline (skip with --no-decode).

The other four workloads of the same family (N=256 d=64; B=4 H=16 N=1024
d=64; B=2 H=16 N=4096 d=128; the spiky N=32768 d=128 shape) are timed the same
way and reported under "per_config", each with its roofline fraction, clocks
and the CPU oracle on a row sample beside it (skip with --no-per-config).

--impl reference times the CPU oracle (float64, numpy) on the host cores, on a
bounded sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s (4·B·H·N²·d) and % of GB300 dense BF16 peak, 1 GPU"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "prefill8k_d128_h32"
# Sources that determine each kernel's machine code: a committed DRAM-traffic
# figure is used only while these are unchanged since its capture.
KERNEL_SOURCES = ["exact_io_aware_34_gb300/csrc/fa_fwd_kernel.cuh", "exact_io_aware_34_gb300/csrc/sm103a_ptx.cuh"]
BWD_KERNEL_SOURCES = ["exact_io_aware_34_gb300/csrc/fa_bwd_kernel.cuh", "exact_io_aware_34_gb300/csrc/fa_fwd_kernel.cuh",
                      "exact_io_aware_34_gb300/csrc/sm103a_ptx.cuh"]
DECODE_KERNEL_SOURCES = ["exact_io_aware_34_gb300/csrc/fa_decode_kernel.cuh", "exact_io_aware_34_gb300/csrc/fa_fwd_kernel.cuh",
                         "exact_io_aware_34_gb300/csrc/sm103a_ptx.cuh"]
NAIVE_KERNEL_SOURCES = ["exact_io_aware_34_gb300/csrc/naive_kernels.cuh", "exact_io_aware_34_gb300/csrc/sm103a_ptx.cuh"]
DECODE_WORKLOAD = "decode32k_gqa8_b4"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


# ----------------------------------------------------------------------------- helpers
def _code_only(text: str) -> str:
    """C++ source without its comments and with runs of whitespace collapsed,
    so that an edit of comments alone leaves the hash (and the machine code)
    unchanged. The kernels' string literals hold no comment markers."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(sources=None) -> str:
    h = hashlib.sha256()
    for rel in (KERNEL_SOURCES if sources is None else sources):
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in ("bf16_tflops", "bf16_tflops_sustained", "hbm_gbs")}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def load_traffic(workload: str, key_suffix: str = "", sources=None):
    """DRAM bytes per launch (per call for the backward) from a committed ncu
    summary, if it was taken on the current kernel sources; otherwise None."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    entry = t.get(workload + key_suffix)
    if not entry or entry.get("kernel_source_hash") != kernel_source_hash(sources):
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """SM clock, power and clock-event (throttle) reasons sampled every few ms
    while the timed region runs: NVML through ctypes in a background thread,
    or ``nvidia-smi -lms 200`` when NVML cannot be loaded."""
    # nvmlClocksEventReasons bits (nvml.h)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    SMI_FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
                  "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                  "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index: int, uuid: str | None = None, period_s: float = 0.005):
        self.gpu = gpu_index
        self.uuid = uuid
        self.period = period_s
        self.samples = []          # (sm_mhz, power_w, reason_bits)
        self.max_mhz = None
        self.out = ""
        self.proc = None
        self._thread = None
        self._stop = False
        self._nvml = None

    def _nvml_open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        ok = False
        if self.uuid:
            ok = lib.nvmlDeviceGetHandleByUUID(("GPU-" + self.uuid).encode(), ctypes.byref(h)) == 0
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.gpu), ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return lib, h, reasons_fn

    def _nvml_loop(self):
        import ctypes
        lib, h, reasons_fn = self._nvml
        clk, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop:
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                p = pw.value / 1000.0 if lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw)) == 0 else None
                r = rs.value if reasons_fn(h, ctypes.byref(rs)) == 0 else 0
                self.samples.append((float(clk.value), p, int(r)))
            time.sleep(self.period)

    def __enter__(self):
        try:
            self._nvml = self._nvml_open()
            import threading
            self._thread = threading.Thread(target=self._nvml_loop, daemon=True)
            self._thread.start()
        except (OSError, AttributeError):
            self._nvml = None
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--id={self.gpu}", "--query-gpu=" + ",".join(self.SMI_FIELDS),
                     "--format=csv,noheader,nounits", "-lms", "200"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self.proc = None
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop = True
            self._thread.join(timeout=2)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self):
        if self.samples:
            sm = [c for c, _, _ in self.samples]
            power = [p for _, p, _ in self.samples if p is not None]
            reasons = sorted({name for _, _, r in self.samples for bit, name in self.REASONS.items() if r & bit})
            return {"sm_mhz": statistics.median(sm), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                    "samples": len(sm), "sm_mhz_min": min(sm), "power_w_max": max(power) if power else None,
                    "source": "nvml"}
        rows = [r.split(", ") for r in (self.out or "").strip().splitlines() if r.strip()]
        rows = [r for r in rows if len(r) == len(self.SMI_FIELDS)]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "", 1).isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        power = [float(r[3]) for r in rows if r[3].replace(".", "", 1).isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None,
                "source": "nvidia-smi"}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def head_shard(H: int, world: int, rank: int):
    """[h0, h1): the contiguous range of heads ``rank`` takes when the H heads
    of one workload are split over ``world`` ranks, as even as possible."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank / world size")
    if H < world:
        raise ValueError(f"cannot split {H} heads over {world} ranks")
    per, extra = divmod(H, world)
    h0 = rank * per + min(rank, extra)
    return h0, h0 + per + (1 if rank < extra else 0)


def torchrun_command(n_gpus: int, argv, port: int):
    """The command that runs this script as ``n_gpus`` ranks on one node (one
    process per GPU), with the rendezvous on 127.0.0.1."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n_gpus}",
            "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *argv]


def _free_port() -> int:
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a float over all ranks (identity when world == 1)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ----------------------------------------------------------------------------- CPU oracle timing
def _oracle_rows_worker(args):
    """Pool task: oracle.attention_rows on the given (b, h, r) rows; returns seconds."""
    import numpy as np
    import oracle as _oracle
    name, rows = args
    Q, K, V, s = _cached_inputs(name)
    t0 = time.perf_counter()
    _oracle.attention_rows(Q, K, V, s, np.asarray(rows))
    return time.perf_counter() - t0


_INPUT_CACHE = {}


def _cached_inputs(name):
    """The workload's inputs as float32 numpy arrays, generated once per process.
    ``bwd:<name>`` adds the backward's dO; ``kv:<name>`` is a shared-K/V-head shape."""
    from exact_io_aware_34_gb300 import inputs as _inp
    if name not in _INPUT_CACHE:
        if name.startswith("kv:"):
            w = _inp.kv_workload(name[3:])
            q, k, v = _inp.make_kv(w.B, w.H, w.H_kv, w.N_q, w.N_kv, w.d, w.seed)
            _INPUT_CACHE[name] = (q.float().numpy(), k.float().numpy(), v.float().numpy(), w.scale)
        elif name.startswith("bwd:"):
            w = _inp.workload(name[4:])
            q, k, v, s = _inp.make_inputs(w)
            do = _inp.make_grad(w.B, w.H, w.N, w.d, w.seed)
            _INPUT_CACHE[name] = (q.float().numpy(), k.float().numpy(), v.float().numpy(), do.float().numpy(), s)
        else:
            q, k, v, s = _inp.make_inputs(_inp.workload(name))
            _INPUT_CACHE[name] = (q.float().numpy(), k.float().numpy(), v.float().numpy(), s)
    return _INPUT_CACHE[name]


def _oracle_bwd_worker(args):
    """Pool task: the backward oracle's work for query-row chunks (b, h, r0, r1):
    dQ of those rows and their contributions to dK and dV. Returns seconds."""
    import oracle as _oracle
    name, chunks = args
    Q, K, V, dO, s = _cached_inputs(name)
    t0 = time.perf_counter()
    for b, h, r0, r1 in chunks:
        _oracle.attention_bwd_heads(Q[:, :, r0:r1], K, V, dO[:, :, r0:r1], s, [(b, h)])
    return time.perf_counter() - t0


def _oracle_kv_worker(args):
    """Pool task: the shared-K/V-head oracle on the given (b, h) query heads. Returns seconds."""
    import oracle as _oracle
    name, heads = args
    Q, K, V, s = _cached_inputs(name)
    t0 = time.perf_counter()
    _oracle.attention_gqa_rows(Q, K, V, s, heads)
    return time.perf_counter() - t0


def _worker_init(name, ready):
    _cached_inputs(name)
    ready.wait()


def _noop(_):
    return 0


class OracleTimer:
    """Times the CPU oracle on row samples of a workload, in a pool of spawned
    single-threaded worker processes (one per host core). Every worker builds
    its copy of the inputs before the first timed task."""

    def __init__(self, name: str, cores: int | None = None, init_name: str | None = None):
        import multiprocessing as mp
        from exact_io_aware_34_gb300 import inputs as _inp
        self.name = name
        self.w = _inp.workload(name) if not name.startswith("kv:") else None
        self.cores = cores or len(os.sched_getaffinity(0))
        os.environ["OPENBLAS_NUM_THREADS"] = "1"
        os.environ["OMP_NUM_THREADS"] = "1"
        ctx = mp.get_context("spawn")
        ready = ctx.Barrier(self.cores)
        self.pool = ctx.Pool(self.cores, initializer=_worker_init, initargs=(init_name or name, ready))
        self.pool.map(_noop, range(4 * self.cores), chunksize=1)

    def run(self, n_rows: int, seed: int = 0):
        """Oracle rows (b, h, r) spread over the workload; returns (wall seconds, flops)."""
        import numpy as np
        w = self.w
        rng = np.random.default_rng(seed)
        flat = rng.choice(w.B * w.H * w.N, size=min(n_rows, w.B * w.H * w.N), replace=False)
        rows = np.stack([flat // (w.H * w.N), (flat // w.N) % w.H, flat % w.N], axis=1)
        # group rows by head so each task converts one head's K and V once
        order = np.lexsort((rows[:, 2], rows[:, 1], rows[:, 0]))
        rows = rows[order]
        chunks = [c.tolist() for c in np.array_split(rows, self.cores) if len(c)]
        t0 = time.perf_counter()
        self.pool.map(_oracle_rows_worker, [(self.name, c) for c in chunks])
        dt = time.perf_counter() - t0
        return dt, 4.0 * len(rows) * w.N * w.d

    def calibrate(self, target_s: float) -> int:
        """Rows per sample so that one sample takes about ``target_s`` seconds."""
        total = self.w.B * self.w.H * self.w.N
        n = 4 * self.cores
        while True:
            dt, _ = self.run(n, seed=99)
            if dt >= 0.2 * target_s or n >= total:
                break
            n = min(total, n * 4)
        rows = int(n * target_s / max(dt, 1e-4))
        return max(self.cores, min(rows, total))

    def close(self):
        self.pool.terminate()
        self.pool.join()


def cpu_baseline_bwd(name: str, target_s: float = 10.0):
    """The backward oracle (float64 numpy) on query-row chunks sampled from the
    workload, one single-threaded process per host core; TFLOP/s counting the
    five N x N x d products (10 * rows * N * d per chunk)."""
    import numpy as np
    from exact_io_aware_34_gb300 import inputs as _inp
    w = _inp.workload(name)
    t = OracleTimer(name, init_name="bwd:" + name)
    try:
        rng = np.random.default_rng(3)
        rows_per_chunk = 64
        n_chunks = t.cores
        while True:
            heads = rng.integers(0, w.B * w.H, size=n_chunks)
            starts = rng.integers(0, w.N - rows_per_chunk + 1, size=n_chunks)
            chunks = [(int(x // w.H), int(x % w.H), int(r0), int(r0) + rows_per_chunk) for x, r0 in zip(heads, starts)]
            parts = [c.tolist() for c in np.array_split(np.array(chunks), t.cores) if len(c)]
            t0 = time.perf_counter()
            t.pool.map(_oracle_bwd_worker, [("bwd:" + name, [tuple(x) for x in p]) for p in parts])
            dt = time.perf_counter() - t0
            if dt >= 0.5 * target_s or n_chunks >= 1024 * t.cores:
                break
            n_chunks = min(1024 * t.cores, max(n_chunks * 2, int(n_chunks * target_s / max(dt, 1e-3))))
    finally:
        t.close()
    flops = 10.0 * n_chunks * rows_per_chunk * w.N * w.d
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": t.cores, "kind": "oracle",
            "sample": f"{n_chunks} chunks of {rows_per_chunk} query rows of the {name} workload (dQ rows and their "
                      f"dK, dV contributions over all {w.N} keys), float64 numpy backward oracle, {t.cores} "
                      f"single-threaded worker processes, {dt:.1f} s"}


def cpu_baseline_decode(name: str):
    """The shared-K/V-head oracle over every query head of the decode workload,
    one single-threaded process per host core; GB/s of K/V processed."""
    import numpy as np
    from exact_io_aware_34_gb300 import inputs as _inp
    w = _inp.kv_workload(name)
    t = OracleTimer("kv:" + name)
    try:
        heads = [(b, h) for b in range(w.B) for h in range(w.H)]
        parts = [[tuple(int(v) for v in x) for x in c] for c in np.array_split(np.array(heads), t.cores) if len(c)]
        # the whole workload, repeated until about 3 s of wall time have passed
        reps = 0
        t0 = time.perf_counter()
        while True:
            t.pool.map(_oracle_kv_worker, [("kv:" + name, p) for p in parts])
            reps += 1
            dt = time.perf_counter() - t0
            if dt >= 3.0 or reps >= 1000:
                break
    finally:
        t.close()
    return {"value": reps * w.kv_bytes / dt / 1e9, "unit": "GB/s", "cores": t.cores, "kind": "oracle",
            "sample": f"the whole {name} workload ({len(heads)} query heads, {w.N_kv} keys each) {reps} times, "
                      f"float64 numpy oracle, {t.cores} single-threaded worker processes, {dt:.2f} s"}


def cpu_baseline(name: str, target_s: float = 15.0):
    t = OracleTimer(name)
    try:
        rows = t.calibrate(target_s)
        dt, flops = t.run(rows, seed=1)
    finally:
        t.close()
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": t.cores, "kind": "oracle",
            "sample": f"{rows} query rows drawn uniformly from the {name} workload (all {t.w.N} keys each), "
                      f"float64 numpy oracle, {t.cores} single-threaded worker processes, {dt:.1f} s"}


# The small configurations also timed on one host core (the whole workload, or
# as much of it as about `target_s` seconds allows).
SMALL_WORKLOADS = ("n256_d64", "n1024_d64_b4h16")


def cpu_baseline_single_core(name: str, target_s: float = 2.0):
    t = OracleTimer(name, cores=1)
    try:
        rows = t.calibrate(target_s)
        dt, flops = t.run(rows, seed=1)
    finally:
        t.close()
    total = t.w.B * t.w.H * t.w.N
    return {"workload": name, "value": flops / dt / 1e12, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{rows} of the {total} query rows of {name} (all {t.w.N} keys each), float64 numpy oracle, "
                      f"one single-threaded worker process, {dt:.2f} s"}


# ----------------------------------------------------------------------------- reference arm
def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    from exact_io_aware_34_gb300 import inputs
    w = inputs.workload(args.workload)
    t = OracleTimer(args.workload)
    try:
        rows = t.calibrate(args.ref_step_s)
        for i in range(args.warmup):
            t.run(rows, seed=1000 + i)
        times, flops = [], 0.0
        for i in range(args.steps):
            dt, f = t.run(rows, seed=i)
            times.append(dt)
            flops += f
    finally:
        t.close()
    total = sum(times)
    value = flops / total / 1e12
    sample = (f"each step: {rows} query rows drawn uniformly from the {w.name} workload (all {w.N} keys each), "
              f"float64 numpy oracle, {t.cores} single-threaded worker processes")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, bf16-rounded inputs)",
        "config": {**w.describe(), "workload": w.name, "sample_rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": t.cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- native arm
def launch_shape(fa, shape):
    """The forward's launch for a [B, H, N, d] problem on this device: CTAs,
    CTAs per cluster (1, or 2 when pairs share the last round's units) and
    the units of 256 query rows run whole."""
    g, c, wu = fa.fa_fwd_launch_shape(*shape)
    return {"grid": g, "cluster": c, "whole_units": wu}


def time_forward(fa, qd, kd, vd, o, lse, scale, flush, stream, steps, warmup, local, uuid):
    """``steps`` fa_fwd calls, each bracketed by CUDA events on ``stream`` with the
    L2 cache flushed before it (outside the events); returns (per-step ms, clocks)."""
    import torch
    for _ in range(warmup):
        fa.fa_fwd(qd, kd, vd, o, lse, scale)
    torch.cuda.synchronize(qd.device)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with ClockSampler(local, uuid) as clocks:
        for i in range(steps):
            flush.fill_(float(i))
            starts[i].record(stream)
            fa.fa_fwd(qd, kd, vd, o, lse, scale)
            ends[i].record(stream)
        torch.cuda.synchronize(qd.device)
    st, info = fa.fa_get_device_status()
    if st != fa.FA_OK:
        raise RuntimeError(f"device status after timed forward steps: {fa.fa_status_string(st)} {info}")
    return [a.elapsed_time(b) for a, b in zip(starts, ends)], clocks.summary()


def run_native(args):
    import torch
    world, rank, local = dist_setup()
    if args.shard == "heads":
        # the strong-scaling run times the forward alone
        args.no_bwd = args.no_comparator = args.no_decode = args.no_per_config = True
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)

    # The CPU baseline runs before the first GPU call (its worker pool is spawned).
    cpu = cpu_bwd = cpu_dec = None
    cpu_small = []
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.workload, target_s=args.cpu_seconds)
        cpu_small = [cpu_baseline_single_core(n) for n in SMALL_WORKLOADS]
        if not args.no_bwd:
            cpu_bwd = cpu_baseline_bwd(args.workload, target_s=min(10.0, args.cpu_seconds))
        if not args.no_decode:
            cpu_dec = cpu_baseline_decode(DECODE_WORKLOAD)
    cpu_cfg = {}
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.no_per_config:
        from exact_io_aware_34_gb300 import inputs as _inp
        for cw in _inp.WORKLOADS:
            if cw.name != args.workload:
                cpu_cfg[cw.name] = cpu_baseline(cw.name, target_s=args.cfg_cpu_seconds)

    from exact_io_aware_34_gb300 import build as fa_build
    from exact_io_aware_34_gb300 import fa, inputs
    fa_build.build()
    fa.load_library()
    w = inputs.workload(args.workload)
    q, k, v, scale = inputs.make_inputs(w)
    if args.shard == "heads":
        # this rank's contiguous range of the workload's heads
        h0, h1 = head_shard(w.H, world, rank)
        q, k, v = (x[:, h0:h1].contiguous() for x in (q, k, v))
    B, H, N, d = q.shape
    flops = 4.0 * B * H * N * N * d          # this rank's share (the whole workload unless sharded)
    qd, kd, vd = (x.to(device) for x in (q, k, v))
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    for _ in range(args.warmup):
        fa.fa_fwd(qd, kd, vd, o, lse, scale)
    torch.cuda.synchronize(device)
    st, info = fa.fa_get_device_status()
    if st != fa.FA_OK:
        raise RuntimeError(f"device status after warm-up: {fa.fa_status_string(st)} {info}")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world, device)
    torch.cuda.synchronize(device)
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        pass
    with ClockSampler(local, uuid) as clocks:
        for i in range(args.steps):
            flush.fill_(float(i))
            starts[i].record(stream)
            fa.fa_fwd(qd, kd, vd, o, lse, scale)
            ends[i].record(stream)
        torch.cuda.synchronize(device)
    barrier(world, device)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = reduce_max(sum(step_ms), world, device)
    st, info = fa.fa_get_device_status()
    if st != fa.FA_OK:
        raise RuntimeError(f"device status after timed steps: {fa.fa_status_string(st)} {info}")

    # The other workloads of the family, timed the same way (their own inputs,
    # flushed L2 before every step, clocks sampled during the timed steps).
    per_config = []
    if not args.no_per_config:
        peaks_pc, peak_src_pc = load_peaks()
        for cw in inputs.WORKLOADS:
            if cw.name == w.name:
                continue
            cq, ck, cv, cs = inputs.make_inputs(cw)
            cqd, ckd, cvd = (x.to(device) for x in (cq, ck, cv))
            co = torch.empty_like(cqd)
            cl = torch.empty(cqd.shape[:3], dtype=torch.float32, device=device)
            n_steps = max(3, min(args.steps, 20))
            c_ms, c_clk = time_forward(fa, cqd, ckd, cvd, co, cl, cs, flush, stream, n_steps, args.warmup, local,
                                       uuid)
            c_avg = sum(c_ms) / len(c_ms)
            c_val = cw.flops / (c_avg * 1e-3) / 1e12
            entry = {
                "workload": cw.name, "config": cw.describe(), "value": c_val, "unit": UNIT, "steps": n_steps,
                "ms_per_step": c_avg,
                "step_ms": {"min": min(c_ms), "median": statistics.median(c_ms), "max": max(c_ms)},
                "roofline": {"bound": "tensor", "achieved": c_val, "peak": peaks_pc["bf16_tflops"], "unit": UNIT,
                             "frac": c_val / peaks_pc["bf16_tflops"],
                             "frac_of_sustained": c_val / peaks_pc["bf16_tflops_sustained"],
                             "peak_source": f"{peak_src_pc} dense bf16 burst",
                             "traffic": load_traffic(cw.name),
                             "kernel": f"fa_fwd_kernel<{cw.d}>", "launch": launch_shape(fa, tuple(cqd.shape)),
                             "flops_per_launch": cw.flops,
                             "algorithmic_bytes_per_launch": cw.B * cw.H * cw.N * (8 * cw.d + 4)},
                "gpu_launches": n_steps,
                "l2": "flushed before every step (512 MB write, outside the events)",
                "clocks": c_clk,
            }
            if cw.name in cpu_cfg:
                entry["cpu_baseline"] = cpu_cfg[cw.name]
            per_config.append(entry)
            del cqd, ckd, cvd, co, cl
        torch.cuda.empty_cache()

    # The standard-attention comparator on the same inputs: S and P in HBM
    # ("01 · 注意力为什么是 IO 瓶颈" §3), same timing rules as the fused steps.
    comparator = None
    if not args.no_comparator:
        ws_bytes = fa.fa_naive_workspace_bytes(B, H, N)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
        o_n = torch.empty_like(qd)
        lse_n = torch.empty_like(lse)
        for _ in range(args.warmup):
            fa.fa_naive_fwd(qd, kd, vd, o_n, lse_n, scale, ws)
        torch.cuda.synchronize(device)
        n_steps = max(3, min(args.steps, 20))
        cs = [torch.cuda.Event(enable_timing=True) for _ in range(n_steps)]
        ce = [torch.cuda.Event(enable_timing=True) for _ in range(n_steps)]
        for i in range(n_steps):
            flush.fill_(float(i))
            cs[i].record(stream)
            fa.fa_naive_fwd(qd, kd, vd, o_n, lse_n, scale, ws)
            ce[i].record(stream)
        torch.cuda.synchronize(device)
        st, info = fa.fa_get_device_status()
        if st != fa.FA_OK:
            raise RuntimeError(f"device status after the comparator: {fa.fa_status_string(st)} {info}")
        naive_ms = sum(a.elapsed_time(b) for a, b in zip(cs, ce)) / n_steps
        fused_ms = sum(step_ms) / len(step_ms)
        # Its floor is HBM traffic: S written, read, written back as P and read
        # by the PV product (4 x 2 bytes per score), plus Q, K, V read, O and
        # LSE written.
        n_bytes = 4 * 2 * B * H * N * N + 4 * 2 * B * H * N * d + 4 * B * H * N
        peaks_c, peak_src_c = load_peaks()
        comparator = {
            "impl": "standard attention: S = QK^T, P = softmax(S) and O = PV as 3 launches, S/P in HBM (bf16)",
            "steps": n_steps, "ms_per_step": naive_ms, "value": flops / (naive_ms * 1e-3) / 1e12, "unit": UNIT,
            "speedup_of_fused": naive_ms / fused_ms,
            "workspace_bytes": ws_bytes, "fused_workspace_bytes": 0,
            "max_abs_diff_O_vs_fused": float((o_n.float() - o.float()).abs().max()),
            "roofline": {"bound": "hbm", "achieved": n_bytes / (naive_ms * 1e-3) / 1e9, "peak": peaks_c["hbm_gbs"],
                         "unit": "GB/s", "frac": n_bytes / (naive_ms * 1e-3) / 1e9 / peaks_c["hbm_gbs"],
                         "algorithmic_bytes_per_call": n_bytes, "peak_source": f"{peak_src_c} HBM copy bandwidth",
                         "traffic": load_traffic(w.name, ":comparator", NAIVE_KERNEL_SOURCES),
                         "kernels": "s_gemm_kernel (S, persistent), softmax_rows_kernel, gemm_bf16_kernel<d, 0> (PV)"},
        }
        del ws, o_n, lse_n
        torch.cuda.empty_cache()

    # The backward pass by recomputation on the same workload (O and LSE from the
    # forward above, dO seeded), same timing rules: flush before every step,
    # events on the launching stream, clocks sampled during the timed steps.
    bwd = None
    if not args.no_bwd:
        do = inputs.make_grad(B, H, N, d, w.seed).to(device)
        dq, dk, dv = (torch.empty_like(qd) for _ in range(3))
        ws_b = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N), dtype=torch.uint8, device=device)
        for _ in range(args.warmup):
            fa.fa_bwd(qd, kd, vd, o, do, lse, dq, dk, dv, scale, ws_b)
        torch.cuda.synchronize(device)
        st, info = fa.fa_get_device_status()
        if st != fa.FA_OK:
            raise RuntimeError(f"device status after backward warm-up: {fa.fa_status_string(st)} {info}")
        n_steps = max(3, min(args.steps, 20))
        bs = [torch.cuda.Event(enable_timing=True) for _ in range(n_steps)]
        be = [torch.cuda.Event(enable_timing=True) for _ in range(n_steps)]
        with ClockSampler(local, uuid) as bclocks:
            for i in range(n_steps):
                flush.fill_(float(i))
                bs[i].record(stream)
                fa.fa_bwd(qd, kd, vd, o, do, lse, dq, dk, dv, scale, ws_b)
                be[i].record(stream)
            torch.cuda.synchronize(device)
        st, info = fa.fa_get_device_status()
        if st != fa.FA_OK:
            raise RuntimeError(f"device status after backward steps: {fa.fa_status_string(st)} {info}")
        b_ms = [a.elapsed_time(b) for a, b in zip(bs, be)]
        bwd_ms = sum(b_ms) / n_steps
        bwd_flops = 2.5 * flops          # five N x N x d products per head: 10*B*H*N^2*d
        bwd = {
            "metric": "attention bwd TFLOP/s (10·B·H·N²·d: the five N×N×d products of the gradient)",
            "value": bwd_flops / (bwd_ms * 1e-3) / 1e12, "unit": UNIT, "steps": n_steps,
            "ms_per_step": bwd_ms,
            "step_ms": {"min": min(b_ms), "median": statistics.median(b_ms), "max": max(b_ms)},
            "executed_tflops": 3.5 * flops / (bwd_ms * 1e-3) / 1e12,   # S and dP formed in both CTA roles
            "gpu_launches": 2 * n_steps,
            "workspace_bytes": ws_b.numel(),
            "clocks": bclocks.summary(),
        }
        del do, dq, dk, dv, ws_b
        torch.cuda.empty_cache()

    # Decode with shared K/V heads (fa_fwd_kv, short-query kernel + merge):
    # bandwidth-bound, so it is measured in K/V bytes per second against the
    # HBM roofline. Same timing rules.
    decode = None
    if not args.no_decode:
        dw = inputs.kv_workload(DECODE_WORKLOAD)
        dq_, dk_, dv_ = (x.to(device) for x in inputs.make_kv(dw.B, dw.H, dw.H_kv, dw.N_q, dw.N_kv, dw.d, dw.seed))
        splits = fa.fa_fwd_kv_num_splits(dw.B, dw.H, dw.H_kv, dw.N_q, dw.N_kv, dw.d)
        dws_bytes = fa.fa_fwd_kv_workspace_bytes(dw.B, dw.H, dw.H_kv, dw.N_q, dw.N_kv, dw.d, 0)
        dws = torch.empty(max(dws_bytes, 128), dtype=torch.uint8, device=device)
        do_, dl_ = torch.empty_like(dq_), torch.empty(dq_.shape[:3], dtype=torch.float32, device=device)
        for _ in range(args.warmup):
            fa.fa_fwd_kv(dq_, dk_, dv_, do_, dl_, dw.scale, 0, dws)
        torch.cuda.synchronize(device)
        st, info = fa.fa_get_device_status()
        if st != fa.FA_OK:
            raise RuntimeError(f"device status after decode warm-up: {fa.fa_status_string(st)} {info}")
        n_steps = max(3, min(args.steps, 50))

        # K and V (537 MB) are four times the L2 and each byte is read once per
        # call, so calls run back to back ("inputs larger than L2"), as the copy
        # that gives the HBM peak does. Timed a second time with the 512 MB
        # write before each call: its dirty lines are written back while the
        # next call reads, which costs a bandwidth-bound kernel time of its own.
        def time_decode(write_flush: bool):
            es = [torch.cuda.Event(enable_timing=True) for _ in range(n_steps)]
            ee = [torch.cuda.Event(enable_timing=True) for _ in range(n_steps)]
            with ClockSampler(local, uuid) as clk:
                for i in range(n_steps):
                    if write_flush:
                        flush.fill_(float(i))
                    es[i].record(stream)
                    fa.fa_fwd_kv(dq_, dk_, dv_, do_, dl_, dw.scale, 0, dws)
                    ee[i].record(stream)
                torch.cuda.synchronize(device)
            st, info = fa.fa_get_device_status()
            if st != fa.FA_OK:
                raise RuntimeError(f"device status after decode steps: {fa.fa_status_string(st)} {info}")
            return [a.elapsed_time(b) for a, b in zip(es, ee)], clk.summary()

        d_ms, dclocks = time_decode(False)
        f_ms, _ = time_decode(True)
        dec_ms = sum(d_ms) / n_steps
        fl_ms = sum(f_ms) / n_steps
        decode = {
            "metric": "decode K/V read rate (GB/s: K and V bytes per call / time) with shared K/V heads",
            "value": dw.kv_bytes / (dec_ms * 1e-3) / 1e9, "unit": "GB/s", "steps": n_steps, "ms_per_step": dec_ms,
            "step_ms": {"min": min(d_ms), "median": statistics.median(d_ms), "max": max(d_ms)},
            "tflops": dw.flops / (dec_ms * 1e-3) / 1e12,
            "config": {**dw.describe(), "l2": "inputs larger than L2 (537 MB of K/V read once per call), calls back to back"},
            "with_l2_write_flush": {"ms_per_step": fl_ms, "value": dw.kv_bytes / (fl_ms * 1e-3) / 1e9, "unit": "GB/s",
                                    "l2": "512 MB written before every call, outside the events"},
            "num_splits": splits, "kv_bytes_per_call": dw.kv_bytes, "workspace_bytes": dws_bytes,
            "gpu_launches": n_steps * (2 if splits > 1 else 1), "clocks": dclocks,
        }
        del dq_, dk_, dv_, dws, do_, dl_
        torch.cuda.empty_cache()

    # End to end through the C ABI on host buffers (fa_fwd_host): every step
    # uploads the pinned host Q, K, V, runs the kernel and downloads O and LSE;
    # the library pipelines the copies with the kernel over head groups.
    qh, kh, vh = (x.pin_memory() for x in (q, k, v))
    oh = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    lh = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    hws = torch.empty(fa.fa_fwd_host_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=device)
    e2e_steps = max(3, min(args.steps, 10))
    for i in range(2):
        fa.fa_fwd_host(qh, kh, vh, oh, lh, scale, workspace=hws, device=device, stream=stream)
    torch.cuda.synchronize(device)
    barrier(world, device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(e2e_steps):
        fa.fa_fwd_host(qh, kh, vh, oh, lh, scale, workspace=hws, device=device, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize(device)
    e2e_ms = reduce_max(e0.elapsed_time(e1), world, device)
    del hws
    h2d = 3 * q.numel() * 2
    d2h = o.numel() * 2 + lse.numel() * 4

    if rank == 0:
        peaks, peak_src = load_peaks()
        avg_ms = sum(step_ms) / len(step_ms)
        achieved = flops / (avg_ms * 1e-3) / 1e12
        job_flops = w.flops if args.shard == "heads" else world * flops   # all ranks' work per step
        value = job_flops * args.steps / (total_ms * 1e-3) / 1e12
        traffic = load_traffic(w.name)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "strong" if args.shard == "heads" else "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; Q,K ~ N(0,1), V ~ U(-1,1), bf16)",
            "config": {**w.describe(), "l2": "flushed before every step (512 MB write, outside the events)",
                       "parallelism": (f"heads split over {world} ranks (no collective)" if args.shard == "heads"
                                       else f"replicas x{world} (independent problems per rank)")},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": UNIT,
                         "frac": achieved / peaks["bf16_tflops"], "traffic": traffic,
                         "peak_source": f"{peak_src} dense bf16 burst",
                         "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                         "kernel": f"fa_fwd_kernel<{d}>", "launch": launch_shape(fa, tuple(qd.shape)),
                         "flops_per_launch": flops,
                         "algorithmic_bytes_per_launch": B * H * N * (8 * d + 4)},
            "e2e": {"value": job_flops * e2e_steps / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / e2e_steps,
                    "api": "fa_fwd_host (C ABI, pinned host buffers; copies pipelined with the kernel)"},
            "gpu_launches": args.steps,
            "clocks": clocks.summary(),
            "step_ms": {"min": min(step_ms), "median": statistics.median(step_ms), "max": max(step_ms)},
        }
        if comparator is not None:
            line["comparator"] = comparator
        if bwd is not None:
            bwd["roofline"] = {"bound": "tensor", "achieved": bwd["value"], "peak": peaks["bf16_tflops"],
                               "unit": UNIT, "frac": bwd["value"] / peaks["bf16_tflops"],
                               "traffic": load_traffic(w.name, ":bwd", BWD_KERNEL_SOURCES),
                               "peak_source": f"{peak_src} dense bf16 burst",
                               "kernels": "bwd_prep_kernel, fa_bwd_kernel<%d> (dK/dV and dQ CTAs)" % d}
            if cpu_bwd is not None:
                bwd["cpu_baseline"] = cpu_bwd
            line["bwd"] = bwd
        if decode is not None:
            decode["roofline"] = {"bound": "hbm", "achieved": decode["value"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                  "frac": decode["value"] / peaks["hbm_gbs"],
                                  "traffic": load_traffic(DECODE_WORKLOAD, "", DECODE_KERNEL_SOURCES),
                                  "peak_source": f"{peak_src} HBM copy bandwidth",
                                  "kernels": "fa_decode_kernel<%d> + decode_merge_kernel<%d>" % (d, d)}
            if cpu_dec is not None:
                decode["cpu_baseline"] = cpu_dec
            line["decode"] = decode
        if per_config:
            line["per_config"] = per_config
        if cpu is not None:
            line["cpu_baseline"] = cpu
        if cpu_small:
            line["cpu_baseline_1core"] = cpu_small
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="CPU oracle sample size (seconds of work)")
    ap.add_argument("--ref-step-s", type=float, default=2.0, help="reference arm: seconds of oracle work per step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-comparator", action="store_true", help="skip timing standard attention (S/P in HBM)")
    ap.add_argument("--no-bwd", action="store_true", help="skip timing the backward pass")
    ap.add_argument("--no-decode", action="store_true", help="skip timing the shared-K/V-head decode shape")
    ap.add_argument("--no-per-config", action="store_true", help="skip timing the other four forward workloads")
    ap.add_argument("--shard", choices=["none", "heads"], default="none",
                    help="N > 1: 'none' = every rank runs the whole workload (weak scaling); 'heads' = the ranks "
                         "split its heads (strong scaling)")
    ap.add_argument("--cfg-cpu-seconds", type=float, default=4.0,
                    help="CPU oracle sample size for each of the other workloads (seconds of work)")
    raw_argv = list(sys.argv[1:] if argv is None else argv)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    env_world = os.environ.get("WORLD_SIZE")
    if env_world is None and args.gpus > 1:
        # no torchrun environment: start the N ranks (one per GPU) ourselves
        return subprocess.call(torchrun_command(args.gpus, raw_argv, _free_port()))
    if env_world is not None and int(env_world) != args.gpus:
        ap.error(f"--gpus {args.gpus} does not match WORLD_SIZE={env_world}")
    if args.impl == "reference":
        return run_reference(args)
    return run_native(args)


if __name__ == "__main__":
    sys.exit(main())
