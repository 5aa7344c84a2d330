"""bench.py end to end on the GPU (short runs): the JSON line carries every key
the measurement contract asks for (needs a GB300)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                         text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def test_bench_line_has_the_contract_keys():
    d = _run(["--steps", "3", "--warmup", "3", "--no-cpu-baseline", "--no-comparator", "--no-bwd", "--no-decode"])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks", "per_config"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["dtype"] == "bf16"
    assert d["config"]["workload"] == "prefill8k_d128_h32"
    assert d["value"] > 0 and d["gpu_launches"] == 3
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and 0 < r["frac"] == pytest.approx(r["achieved"] / r["peak"])
    assert r["launch"]["cluster"] in (1, 2) and 1 <= r["launch"]["grid"] <= 1024
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] == 3 * 32 * 8192 * 128 * 2
    assert e["d2h_bytes_per_step"] == 32 * 8192 * (128 * 2 + 4)
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    names = [c["workload"] for c in d["per_config"]]
    assert names == ["n256_d64", "n1024_d64_b4h16", "n4096_d128_b2h16", "long32k_d128_h16_spiky"]
    for c in d["per_config"]:
        assert c["value"] > 0 and c["roofline"]["frac"] > 0 and "clocks" in c


def test_bench_head_shard_on_one_rank():
    """--shard heads on a single rank is the whole workload (strong-scaling label)."""
    d = _run(["--steps", "3", "--warmup", "3", "--no-cpu-baseline", "--shard", "heads", "--workload",
              "n4096_d128_b2h16"])
    assert d["scaling"] == "strong" and "heads split" in d["config"]["parallelism"]
    assert d["value"] > 0 and "per_config" not in d and "bwd" not in d
