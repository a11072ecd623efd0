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


def test_traffic_figures_match_current_sources():
    rows = {"uniform_8x2048": bench.kernel_source_hash(),
            "conv_uniform_8x2048": bench.kernel_source_hash(bench.ROW_KERNEL_SOURCES["conv"]),
            "decode_spec_256x4": bench.kernel_source_hash(bench.ROW_KERNEL_SOURCES["decode"]),
            "gdn_uniform_8x2048": bench.kernel_source_hash(bench.ROW_KERNEL_SOURCES["gdn"])}
    for workload, khash in rows.items():
        t = bench.read_traffic(khash, workload)
        assert t is not None and t > 1e8, (workload, khash)
    # another workload or another source never borrows a figure
    assert bench.read_traffic(rows["uniform_8x2048"], "varlen_lognormal_32k") is None
    assert bench.read_traffic("0" * 16, "uniform_8x2048") is None
