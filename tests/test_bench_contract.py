"""bench.py's output contract, on the CPU: the reference arm (the fp64 oracle timed on
this host) prints one JSON line with every key the contract asks for, and the DRAM
traffic figures committed under profiles/ are keyed to the current kernel sources and
to the workloads they were measured on (bench.py reports null for any other pairing).
"""
import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config",
                          "tiny_fp32", "--steps", "1", "--warmup", "0"], cwd=ROOT, capture_output=True, text=True,
                         timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1
    assert d["warmup"] >= 3  # the contract's minimum, enforced by bench.py
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["data"] == "synthetic" and d["dtype"] == "f64" and d["unit"] == "tokens/s"
    assert d["config"]["workload"] == "tiny_fp32" and d["value"] > 0 and d["ms_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_traffic_figures_are_keyed_to_source_and_workload():
    # Every committed figure names the kernel-source hash and the workload it was
    # measured on; a figure is reported only for exactly that pair (null after a
    # source change until it is captured again).
    lines = [ln.split() for ln in open(os.path.join(ROOT, "profiles", "traffic.txt"))
             if ln.strip() and not ln.startswith("#")]
    assert lines
    for f in lines:
        assert f[0] == "dram_bytes_per_launch" and len(f) == 4, f
        assert int(f[1]) > 1e8 and len(f[2]) == 16, f
        assert bench.read_traffic(f[2], f[3]) == float(f[1])
        # another workload or another source never borrows a figure
        assert bench.read_traffic(f[2], f[3] + "_other") is None
        assert bench.read_traffic("0" * 16, f[3]) is None


def test_reference_sample_is_sized_to_the_run(monkeypatch):
    # sized_reference times one group of units, then takes whole groups so that
    # warm-up + K steps fit REF_SECONDS (at least one group, at most every unit)
    import types
    clock = {"t": 0.0}
    monkeypatch.setattr(bench.time, "perf_counter", lambda: clock["t"])
    unit_s = 0.01  # simulated seconds per group of units

    def build(n):
        return n, 100.0 * n, f"{n} units"

    def run(n):
        clock["t"] += unit_s * -(-n // 4)  # groups of 4 run in parallel

    def sized(steps, warmup, n_units):
        args = types.SimpleNamespace(steps=steps, warmup=warmup)
        return bench.sized_reference(args, n_units, build, run, group=4)

    # K = 2500: 150 s / 2505 steps = 59.9 ms a step -> 5 groups of 4 units, 50 ms a step
    value, what = sized(2500, 5, 1000)
    assert what == "20 units"
    assert abs(value - 2000.0 / 0.05) < 1e-6 * value
    # few steps: the whole workload
    assert sized(3, 3, 1000)[1] == "1000 units"
    # a step budget below one group still takes one group
    assert sized(10 ** 6, 5, 1000)[1] == "4 units"
    # fewer units than a group
    assert sized(2500, 5, 3)[1] == "3 units"
