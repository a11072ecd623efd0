"""Benchmark: Mamba2 SSD varlen prefill tokens/s per layer on one GB300.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config NAME] [--no-cpu-baseline]

A step is one pass of the whole hot path over one batch: the device metadata
builder (plan) and the SSD forward (every kernel of the path), with inputs
resident in HBM.  The workload is the uniform batch of 8 requests x 2048
tokens, H=80, P=64, N=128, G=1, chunk_size=256, bf16 in / fp32 state, D skip
and SiLU(z) gate (a ~2.7B Mamba2 layer).  Its inputs (~0.54 GB) exceed the
129 MB L2, so no flush is needed between steps.

The e2e figure goes through the public API with host buffers: every step copies its
inputs from pinned host memory to the device, plans, runs the forward and copies y
and the final states back; the reported value streams the steps (step k's copies in,
step k-1's forward and step k-2's results out overlap on three streams over two
device buffer sets), and e2e.serial_value runs them one after another.

Prints one JSON line (rank 0).  Under torchrun every rank runs its own copy
of the batch (independent problems: weak scaling, no data-path collective);
value = tokens of all ranks / max-over-ranks time.

--impl reference times the CPU fp64 oracle (the only reference there is: the
pages ship no code) on this host's cores, on the same workload and metric.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_CONFIG = "uniform_8x2048"
METRIC = "SSD varlen prefill tokens/s per layer (bf16, 1×GB300); % of roofline"
DECODE_METRIC = "SSD decode step tokens/s per layer (bf16, 1×GB300); % of roofline"
CONV_METRIC = "varlen causal conv1d tokens/s per layer (bf16, 1×GB300); % of roofline"
GDN_METRIC = "gated delta rule varlen prefill tokens/s per layer (bf16, 1×GB300); % of roofline"
# The files the forward's scan kernels (two heads per CTA for P = 64, one head per
# CTA otherwise, the segment-state passes) are compiled from; a DRAM-traffic figure
# in profiles/traffic.txt is valid only for this exact source.
KERNEL_SOURCES = ["mamba2_ssd_varlen_gb300/csrc/ssd_pair.cu", "mamba2_ssd_varlen_gb300/csrc/ssd_chunk_tc.cu",
                  "mamba2_ssd_varlen_gb300/csrc/tc_util.cuh", "mamba2_ssd_varlen_gb300/csrc/sm100.cuh",
                  "mamba2_ssd_varlen_gb300/csrc/ssd_internal.cuh", "mamba2_ssd_varlen_gb300/csrc/pdl.cuh",
                  # how a batch is cut into segments decides the scan's traffic too
                  "mamba2_ssd_varlen_gb300/csrc/ssd_api.cu", "mamba2_ssd_varlen_gb300/csrc/ssd_plan.cu"]


def env_rank():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def max_over_ranks(value, dist, device="cuda"):
    """The largest of every rank's value (the slowest rank's time), or the value
    itself on one rank."""
    if not dist:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def roofline_of(nbytes, flops, ms, peaks):
    """Roofline of one launch: the slower of the algorithmic bytes at the measured
    HBM bandwidth and the algorithmic flops at the measured bf16 tensor peak
    (burst: the kernel is timed launch by launch) decides the bound; achieved and
    peak are in that bound's unit, frac = roofline time / measured time."""
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    sec = ms / 1e3
    if t_tc > t_hbm:
        achieved = flops / sec / 1e12
        return {"bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(t_tc / sec, 4)}
    achieved = nbytes / sec / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(t_hbm / sec, 4)}


def replica_throughput(units_per_rank, world, ms):
    """Whole-job units per second when every rank processes units_per_rank in ms."""
    return units_per_rank * world / (ms / 1e3)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# The same for the kernels of the other rows (each bench line reports its own).
ROW_KERNEL_SOURCES = {
    "conv": ["mamba2_ssd_varlen_gb300/csrc/ssd_conv1d.cu", "mamba2_ssd_varlen_gb300/csrc/ssd_internal.cuh",
             "mamba2_ssd_varlen_gb300/csrc/pdl.cuh"],
    "decode": ["mamba2_ssd_varlen_gb300/csrc/ssd_decode.cu", "mamba2_ssd_varlen_gb300/csrc/ssd_internal.cuh",
               "mamba2_ssd_varlen_gb300/csrc/pdl.cuh"],
    "gdn": ["mamba2_ssd_varlen_gb300/csrc/ssd_gdn_tc.cu", "mamba2_ssd_varlen_gb300/csrc/ssd_gdn.cu",
            "mamba2_ssd_varlen_gb300/csrc/tc_util.cuh", "mamba2_ssd_varlen_gb300/csrc/sm100.cuh",
            "mamba2_ssd_varlen_gb300/csrc/ssd_internal.cuh", "mamba2_ssd_varlen_gb300/csrc/pdl.cuh"],
}


def kernel_source_hash(files=None):
    h = hashlib.sha256()
    for rel in (KERNEL_SOURCES if files is None else files):
        h.update(os.path.basename(rel).encode())
        h.update(open(os.path.join(ROOT, rel), "rb").read())
    return h.hexdigest()[:16]


def cost_model(prob, n_export_rows, n_block_writes):
    """Bytes and flops one step must move / do at minimum (no chunk-state traffic).

    bytes = x + y + z + B + C + dt in their dtype, + initial states read + final
    states, chunk exports and block checkpoints written (fp32).
    flops = T (4 P N H + Q P H + Q N G): the chunk-state and state-readout
    contractions plus the causal halves of the intra-chunk products.
    """
    T, H, P, N, G = prob["T"], prob["H"], prob["P"], prob["N"], prob["G"]
    Q = prob["chunk_size"]
    el = 4 if prob["dtype"] == "fp32" else 2
    tok_bytes = el * (T * H * P * (2 + (prob["z"] is not None)) + 2 * T * G * N + T * H)
    st = H * P * N * 4
    init_reads = 0
    if prob["init_slots"] is not None:
        init_reads = int((prob["init_slots"] >= 0).sum().item())
    finals = 0
    if prob.get("final_dense", True):
        finals += prob["R"]
    if prob["final_slots"] is not None:
        finals += int((prob["final_slots"] >= 0).sum().item())
    state_bytes = st * (init_reads + finals + n_export_rows + n_block_writes)
    flops = T * (4 * P * N * H + Q * P * H + Q * N * G)
    return {"bytes": tok_bytes + state_bytes, "flops": flops, "token_bytes": tok_bytes,
            "state_bytes": state_bytes}


def count_outputs(prob):
    """Export rows and block-checkpoint writes of the batch (index arithmetic only)."""
    cu = prob["cu_seqlens"].cpu().tolist()
    nc = prob["num_computed"]
    nc = [0] * prob["R"] if nc is None else nc.cpu().tolist()
    Q = prob["chunk_size"]
    rows = 0
    blocks = 0
    bt = prob["block_table"]
    btl = None if bt is None else bt.cpu().tolist()
    bs = prob["block_size"]
    for i in range(prob["R"]):
        L = cu[i + 1] - cu[i]
        s = nc[i]
        if L > 0:
            rows += (s + L - 1) // Q - s // Q + 1
        if btl is not None and bs > 0:
            kb = (s // bs + 1) * bs
            while kb <= s + L:
                if btl[i][kb // bs - 1] >= 0:
                    blocks += 1
                kb += bs
    return (rows if prob["export_chunks"] else 0), blocks


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]), "power": float(parts[3]),
                             "hw": parts[5], "hwt": parts[6], "swt": parts[7], "pcap": parts[8]})
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [r for r in rows if r["power"] > 200.0] or rows
        sms = sorted(r["sm"] for r in loaded)
        reasons = set()
        for r in loaded:
            if r["hw"].lower() == "active":
                reasons.add("hw_slowdown")
            if r["hwt"].lower() == "active":
                reasons.add("hw_thermal_slowdown")
            if r["swt"].lower() == "active":
                reasons.add("sw_thermal_slowdown")
            if r["pcap"].lower() == "active":
                reasons.add("sw_power_cap")
        return {"sm_mhz": sms[len(sms) // 2], "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(loaded)}


def time_steps(run, K, stream, dist, local_rank):
    """K steps timed with events only at their two ends, then K more with events
    around each step; the SM clocks are sampled over both passes.  An event
    recorded between two kernels keeps the next one from being scheduled before
    the previous ends (1.5-3.5 us a step), so throughput comes from the first
    pass and the per-launch average (the roofline's denominator) from the second.
    Returns (max-over-ranks ms per step of the first pass, per-step ms of the
    second, clocks)."""
    import torch
    sampler = ClockSampler(local_rank)
    sampler.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(K):
        run()
    t1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    total_ms = max_over_ranks(t0.elapsed_time(t1), dist)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in ev:
        a.record(stream)
        run()
        b.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    return total_ms / K, [a.elapsed_time(b) for a, b in ev], clocks


def read_traffic(kernel_hash, config=None):
    """DRAM bytes per launch of a kernel from the committed ncu summaries, or None
    when the figure is absent or the kernel source changed since.  Lines of the
    other rows carry the workload they were measured (or scaled) for."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    for line in open(p):
        parts = line.split()
        if len(parts) >= 3 and parts[0] == "dram_bytes_per_launch":
            if parts[2] == kernel_hash and (config is None or (len(parts) >= 4 and parts[3] == config)):
                return float(parts[1])
    return None


def cpu_baseline(prob, max_seconds=30.0):
    """Time the fp64 oracle, as it stands, on this host's cores."""
    import oracle
    import workloads
    ncores = os.cpu_count() or 1
    # Sample: whole requests, as many as fit the CPU budget (15.7 us per token-head-core
    # measured for P=64, N=128; scaled by P*N).
    per = 16e-6 * prob["P"] * prob["N"] / (64 * 128)
    lens = prob["lengths"]
    sel = []
    tok = 0
    for i, L in enumerate(lens):
        if sel and (tok + L) * prob["H"] * per / ncores > max_seconds:
            break
        sel.append(i)
        tok += L
    o = workloads.to_oracle(prob, requests=sel)
    t0 = time.perf_counter()
    oracle.forward(o, n_threads=ncores)
    dt = time.perf_counter() - t0
    # the same recurrence on one core, over the first request only
    o1 = workloads.to_oracle(prob, requests=sel[:1])
    t1 = time.perf_counter()
    oracle.forward(o1, n_threads=1)
    dt1 = time.perf_counter() - t1
    return {"value": tok / dt, "unit": "tokens/s", "cores": ncores, "kind": "oracle",
            "sample": f"{len(sel)} of {len(lens)} requests ({tok} tokens, all {prob['H']} heads), "
                      f"fp64 token-by-token recurrence, {dt:.2f} s",
            "value_one_core": lens[sel[0]] / dt1,
            "sample_one_core": f"request {sel[0]} ({lens[sel[0]]} tokens, all heads) on one core, {dt1:.2f} s"}


REF_SECONDS = 150.0  # the whole reference run (warm-up and timed steps) on the host cores


def sized_reference(args, n_units, build, run, group=1):
    """Times the oracle on a sample sized so that ``--warmup`` + ``--steps`` steps take
    about REF_SECONDS in all, whatever K is.  ``build(n)`` returns (sample, tokens it
    stands for, description) for the first n of ``n_units`` units of the workload;
    ``run(sample)`` runs the oracle on it.  Samples are whole multiples of ``group``
    units (the host's core count for an oracle that spreads units over threads, so
    that every core has work), timed once at one group to size them.  Returns
    (tokens/s: the median step, description)."""
    g = max(1, min(group, n_units))
    one, _, _ = build(g)
    t0 = time.perf_counter()
    run(one)
    t_group = max(time.perf_counter() - t0, 1e-5)
    per_step = REF_SECONDS / max(1, args.steps + args.warmup)
    n = min(n_units, g * max(1, int(per_step / t_group)))
    sample, tokens, what = build(n)
    for _ in range(args.warmup):
        run(sample)
    vals = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run(sample)
        vals.append(tokens / (time.perf_counter() - t0))
    return sorted(vals)[len(vals) // 2], what


def run_reference_decode(args, world):
    """The oracle on the machine's host cores for a decode step: a sample of whole
    requests (all heads) per timed step, sized by sized_reference."""
    import oracle
    import workloads
    prob = workloads.make_decode_problem(args.config, device="cpu")
    R, T, H = prob["R"], prob["T"], prob["H"]
    ncores = os.cpu_count() or 1

    def build(n):
        sel = list(range(n))
        tok = int(sum(prob["windows"][i] for i in sel))
        return (workloads.to_oracle_decode(prob, requests=sel), tok,
                f"{n} of {R} requests ({tok} tokens, all {H} heads), fp64 token-by-token recurrence")

    value, sample = sized_reference(args, R, build, lambda o: oracle.decode(o, n_threads=ncores), group=ncores)
    line = {"metric": DECODE_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": T / value * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": args.config, "T": T, "R": R, "H": H, "P": prob["P"], "N": prob["N"],
                       "G": prob["G"], "window": max(prob["windows"])},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": ncores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference_conv(args, world):
    """The conv1d oracle on the host cores: a channel sample per timed step, sized by
    sized_reference."""
    from oracle.conv1d import conv1d
    import workloads
    prob = workloads.make_conv_problem(args.config, device="cpu")
    T, D = prob["T"], prob["D"]

    def build(n):
        ch = list(range(0, D, max(1, D // n)))[:n]
        return (workloads.to_oracle_conv(prob, channels=ch), T * len(ch) / D,
                f"{len(ch)} of {D} channels, all {T} tokens, scaled to all channels")

    value, sample = sized_reference(args, D, build, conv1d)
    line = {"metric": CONV_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": T / value * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": args.config, "T": T, "R": prob["R"], "D": D, "W": prob["W"]},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def gdn_oracle_sample(prob, max_seconds):
    """The GDN oracle over whole requests of the workload, in order, until about
    ``max_seconds`` have passed; returns (tokens/s, what was sampled)."""
    from oracle.gdn import gdn_forward
    import workloads
    cu = prob["cu_seqlens"].cpu().numpy()
    done, t0 = [], time.perf_counter()
    for i in range(len(cu) - 1):
        gdn_forward(workloads.to_oracle_gdn(prob, requests=[i]))
        done.append(i)
        if time.perf_counter() - t0 > max_seconds:
            break
    dt = time.perf_counter() - t0
    toks = int(sum(cu[i + 1] - cu[i] for i in done))
    return toks / dt, f"{len(done)} of {len(cu) - 1} requests ({toks} tokens, all heads), numpy fp64"


def run_reference_gdn(args, world):
    """The GDN oracle on the host: units are (request, value head) in order, the
    heads of the first request before whole requests; the sample is sized by
    sized_reference and scaled to all heads."""
    from oracle.gdn import gdn_forward
    import workloads
    prob = workloads.make_gdn_problem(args.config, device="cpu")
    lens, Hv = prob["lengths"], int(prob["v"].shape[1])

    def build(n):
        if n <= Hv:
            return (workloads.to_oracle_gdn(prob, requests=[0], heads=list(range(n))), lens[0] * n / Hv,
                    f"request 0 ({lens[0]} tokens), {n} of {Hv} value heads, numpy fp64, scaled to all heads")
        k = min(len(lens), n // Hv)
        return (workloads.to_oracle_gdn(prob, requests=list(range(k))), sum(lens[:k]),
                f"{k} of {len(lens)} requests ({sum(lens[:k])} tokens, all heads), numpy fp64")

    value, sample = sized_reference(args, len(lens) * Hv, build, gdn_forward)
    T = prob["T"]
    line = {"metric": GDN_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": T / value * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": gdn_config(prob, args.config, world),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference(args, rank, world):
    import workloads
    if rank != 0:
        return
    if args.config in workloads.GDN_CONFIGS:
        return run_reference_gdn(args, world)
    if args.config in workloads.DECODE_CONFIGS:
        return run_reference_decode(args, world)
    if args.config in workloads.CONV_CONFIGS:
        return run_reference_conv(args, world)
    import oracle
    prob = workloads.make_problem(args.config, device="cpu")
    # Units are (request, head) in order, the heads of the first request before whole
    # requests; the sample is sized by sized_reference and scaled to all heads.
    lens, H = prob["lengths"], prob["H"]
    ncores = os.cpu_count() or 1

    def build(n):
        if n <= H:
            return (workloads.to_oracle(prob, requests=[0], heads=list(range(n))), lens[0] * n / H,
                    f"request 0 ({lens[0]} tokens), {n} of {H} heads, fp64 token-by-token recurrence, "
                    f"scaled to all heads")
        k = min(len(lens), n // H)
        return (workloads.to_oracle(prob, requests=list(range(k))), sum(lens[:k]),
                f"{k} of {len(lens)} requests ({sum(lens[:k])} tokens, all {H} heads), "
                f"fp64 token-by-token recurrence")

    value, sample = sized_reference(args, len(lens) * H, build, lambda o: oracle.forward(o, n_threads=ncores),
                                    group=ncores)
    T = prob["T"]
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": T / value * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": args.config, "T": T, "R": prob["R"], "H": prob["H"],
                       "P": prob["P"], "N": prob["N"], "G": prob["G"],
                       "chunk_size": prob["chunk_size"]},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": ncores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def decode_cost(prob):
    """Bytes one decode step must move: the read anchors' states, the states written
    to write anchors (fp32), and x, z, y, B, C, dt of the window tokens."""
    T, H, P, N, G = prob["T"], prob["H"], prob["P"], prob["N"], prob["G"]
    el = 4 if prob["dtype"] == "fp32" else 2
    tok_bytes = el * (T * H * P * (2 + (prob["z"] is not None)) + 2 * T * G * N + T * H)
    st = H * P * N * 4
    win = prob["windows"]
    reads = sum(1 for i, s in enumerate(prob["read_slots"].tolist()) if s >= 0 and win[i] > 0)
    writes = int((prob["write_slots"] >= 0).sum().item())
    return {"bytes": tok_bytes + st * (reads + writes), "token_bytes": tok_bytes,
            "state_bytes": st * (reads + writes), "flops": T * H * P * N * 4}


def run_decode_bench(args, rank, local_rank, world, dist):
    """The decode / speculative-decode step (ssd_varlen_decode), timed like the forward."""
    import torch
    import mamba2_ssd_varlen_gb300 as m
    import workloads
    peaks = load_peaks()
    prob = workloads.make_decode_problem(args.config, device="cuda")
    call = m.DecodeCall(prob)
    stream = torch.cuda.current_stream()
    cost = decode_cost(prob)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    assert call.status() == 0, "device error during warm-up"
    K = args.steps
    ms_per_step, k_ms, clocks = time_steps(call, K, stream, dist, local_rank)
    assert call.status() == 0, "device error during the timed region"
    k_avg = sum(k_ms) / K
    T = prob["T"]
    # End to end: the step's inputs (tokens, anchors) host -> device and y back;
    # the state pool stays resident in HBM (it is the cache the anchors index).
    host_in = {k: prob[k].cpu().pin_memory() for k in ("x", "dt", "B", "C", "z", "cu_seqlens", "read_slots",
                                                     "write_slots") if prob.get(k) is not None}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    y_host = torch.empty(call.y.shape, dtype=call.y.dtype, pin_memory=True)
    d2h = y_host.numel() * y_host.element_size()

    def e2e_step():
        for k_, t_ in host_in.items():
            prob[k_].copy_(t_, non_blocking=True)
        call()
        y_host.copy_(call.y, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = a.elapsed_time(b) / args.e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, dist)
    achieved = cost["bytes"] / (k_avg / 1e3) / 1e9
    line = {"metric": DECODE_METRIC, "value": T * world / (ms_per_step / 1e3), "unit": "tokens/s",
            "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if prob["dtype"] == "bf16" else "f32", "data": "synthetic",
            "config": {"workload": args.config, "T": T, "R": prob["R"], "H": prob["H"], "P": prob["P"],
                       "N": prob["N"], "G": prob["G"], "window": max(prob["windows"]),
                       "state_writes": int((prob["write_slots"] >= 0).sum().item()),
                       "parallelism": f"replicas{world}" if world > 1 else "single",
                       "l2": "state traffic larger than L2 (no flush)"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": read_traffic(kernel_source_hash(ROW_KERNEL_SOURCES["decode"]), args.config),
                         "peak_source": peaks["source"], "algorithmic_bytes": cost["bytes"],
                         "kernel": "ssd_varlen_decode", "kernel_ms_avg": round(k_avg, 5)},
            "gpu_launches": K, "clocks": clocks,
            "e2e": {"value": T * world / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h}}
    if rank == 0:
        print(json.dumps(line), flush=True)


def conv_cost(prob):
    """Bytes one conv1d must move: x and y, the weights and bias, the conv states
    read and written."""
    T, D, W = prob["T"], prob["D"], prob["W"]
    el = 4 if prob["dtype"] == "fp32" else 2
    states = int((prob["read_slots"] >= 0).sum().item()) + int((prob["write_slots"] >= 0).sum().item())
    return {"bytes": 2 * el * T * D + 4 * D * (W + 1) + el * D * (W - 1) * states, "flops": 2 * T * D * W}


def run_conv_bench(args, rank, local_rank, world, dist):
    """The varlen causal conv1d (ssd_varlen_conv1d), timed like the forward."""
    import torch
    import mamba2_ssd_varlen_gb300 as m
    import workloads
    peaks = load_peaks()
    prob = workloads.make_conv_problem(args.config, device="cuda")
    call = m.Conv1dCall(prob)
    stream = torch.cuda.current_stream()
    cost = conv_cost(prob)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    assert call.status() == 0, "device error during warm-up"
    K = args.steps
    ms_per_step, k_ms, clocks = time_steps(call, K, stream, dist, local_rank)
    assert call.status() == 0, "device error during the timed region"
    k_avg = max_over_ranks(sum(k_ms) / K, dist)
    T = prob["T"]
    host_x = prob["x"].cpu().pin_memory()
    y_host = torch.empty(call.y.shape, dtype=call.y.dtype, pin_memory=True)

    def e2e_step():
        prob["x"].copy_(host_x, non_blocking=True)
        call()
        y_host.copy_(call.y, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = a.elapsed_time(b) / args.e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, dist)
    achieved = cost["bytes"] / (k_avg / 1e3) / 1e9
    line = {"metric": CONV_METRIC, "value": T * world / (ms_per_step / 1e3), "unit": "tokens/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if prob["dtype"] == "bf16" else "f32",
            "data": "synthetic",
            "config": {"workload": args.config, "T": T, "R": prob["R"], "D": prob["D"], "W": prob["W"],
                       "parallelism": f"replicas{world}" if world > 1 else "single",
                       "l2": "x and y each larger than L2 (no flush)"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": read_traffic(kernel_source_hash(ROW_KERNEL_SOURCES["conv"]), args.config),
                         "peak_source": peaks["source"], "algorithmic_bytes": cost["bytes"],
                         "kernel": "ssd_varlen_conv1d", "kernel_ms_avg": round(k_avg, 5)},
            "gpu_launches": K, "clocks": clocks,
            "e2e": {"value": T * world / (e2e_ms / 1e3), "unit": "tokens/s",
                    "h2d_bytes_per_step": host_x.numel() * host_x.element_size(),
                    "d2h_bytes_per_step": y_host.numel() * y_host.element_size()}}
    if rank == 0:
        print(json.dumps(line), flush=True)


def gdn_config(prob, name, world):
    return {"workload": name, "T": prob["T"], "R": prob["R"], "Hk": prob["q"].shape[1], "Hv": prob["v"].shape[1],
            "K": prob["q"].shape[2], "V": prob["v"].shape[2], "chunk": 64, "l2norm": bool(prob["l2norm"]),
            "parallelism": f"replicas{world}" if world > 1 else "single",
            "l2": "q, k, v and o together larger than L2 (no flush)"}


def gdn_cost(prob):
    """Bytes one GDN prefill must move: q, k, v, o in their dtype, g and beta (fp32),
    the initial states read and every state written (fp32); and its algorithmic
    flops: per token and value head K*L (the two masked L x L products, half each)
    + 3*K*V (K S0, Q S0, K^T U) + L*V/2 (P U), times 2, with L = 64."""
    T, R = prob["T"], prob["R"]
    Hk, K = prob["q"].shape[1], prob["q"].shape[2]
    Hv, V = prob["v"].shape[1], prob["v"].shape[2]
    el = prob["q"].element_size()
    states = R if prob.get("final_dense", True) else 0
    if prob.get("init_slots") is not None:
        states += int((prob["init_slots"] >= 0).sum().item())
    if prob.get("final_slots") is not None:
        states += int((prob["final_slots"] >= 0).sum().item())
    if prob.get("block_table") is not None:
        states += int((prob["block_table"] >= 0).sum().item())
    byt = T * (2 * Hk * K + 2 * Hv * V) * el + T * Hv * 8 + states * Hv * K * V * 4
    flops = 2 * T * Hv * (K * 64 + 3 * K * V + 64 * V // 2)
    return {"bytes": byt, "flops": flops}


def run_gdn_bench(args, rank, local_rank, world, dist):
    """The gated-delta-rule prefill (ssd_varlen_gdn_forward), timed like the forward."""
    import torch
    import mamba2_ssd_varlen_gb300 as m
    import workloads
    peaks = load_peaks()
    prob = workloads.make_gdn_problem(args.config, device="cuda")
    call = m.GdnCall(prob)
    stream = torch.cuda.current_stream()
    cost = gdn_cost(prob)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    assert call.status() == 0, "device error during warm-up"
    K = args.steps
    ms_per_step, k_ms, clocks = time_steps(call, K, stream, dist, local_rank)
    assert call.status() == 0, "device error during the timed region"
    k_avg = max_over_ranks(sum(k_ms) / K, dist)
    T = prob["T"]
    hosts = {key: prob[key].cpu().pin_memory() for key in ("q", "k", "v", "g", "beta")}
    o_host = torch.empty(call.o.shape, dtype=call.o.dtype, pin_memory=True)

    def e2e_step():
        for key, t in hosts.items():
            prob[key].copy_(t, non_blocking=True)
        call()
        o_host.copy_(call.o, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = a.elapsed_time(b) / args.e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, dist)
    achieved = cost["bytes"] / (k_avg / 1e3) / 1e9
    line = {"metric": GDN_METRIC, "value": T * world / (ms_per_step / 1e3), "unit": "tokens/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": gdn_config(prob, args.config, world),
            "roofline": {**roofline_of(cost["bytes"], cost["flops"], k_avg, peaks),
                         "traffic": read_traffic(kernel_source_hash(ROW_KERNEL_SOURCES["gdn"]), args.config),
                         "peak_source": peaks["source"], "algorithmic_bytes": cost["bytes"],
                         "tensor_tflops": round(cost["flops"] / (k_avg / 1e3) / 1e12, 1),
                         "kernel": "ssd_varlen_gdn_forward", "kernel_ms_avg": round(k_avg, 5)},
            "gpu_launches": K, "clocks": clocks,
            "e2e": {"value": T * world / (e2e_ms / 1e3), "unit": "tokens/s",
                    "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in hosts.values()),
                    "d2h_bytes_per_step": o_host.numel() * o_host.element_size()}}
    if rank == 0 and not args.no_cpu_baseline:
        v, sample = gdn_oracle_sample(workloads.make_gdn_problem(args.config, device="cpu"), 10.0)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--heads-div", type=int, default=1,
                    help="profiling only: run the workload with H / d heads and G / d groups (at least 1), "
                         "the same tokens and kernels, so an ncu capture of many passes stays small")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    rank, local_rank, world = env_rank()
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    import mamba2_ssd_varlen_gb300 as m
    import workloads

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    m.load_library()
    if (args.config in workloads.DECODE_CONFIGS or args.config in workloads.CONV_CONFIGS
            or args.config in workloads.GDN_CONFIGS):
        bench_fn = (run_decode_bench if args.config in workloads.DECODE_CONFIGS else
                    run_conv_bench if args.config in workloads.CONV_CONFIGS else run_gdn_bench)
        bench_fn(args, rank, local_rank, world, dist)
        if dist:
            dist.destroy_process_group()
        return
    peaks = load_peaks()
    spec = workloads.CONFIGS[args.config]
    if args.heads_div > 1:
        import dataclasses
        spec = dataclasses.replace(spec, H=max(1, spec.H // args.heads_div), G=max(1, spec.G // args.heads_div))
    prob = workloads.make_problem(spec, device="cuda")
    call = m.Call(prob)
    stream = torch.cuda.current_stream()
    n_rows, n_blocks = count_outputs(prob)
    cost = cost_model(prob, n_rows, n_blocks)
    # The tensor-core path launches three kernels per forward (segment states,
    # their chain, the scan); the token-by-token path one.
    tc_path = prob["dtype"] == "bf16" and prob["P"] in (64, 128) and prob["N"] == 128
    kernels_per_forward = 3 if tc_path else 1

    def step():
        call.make_plan()
        call.forward()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert call.status() == 0, "device error during warm-up"

    # Two timed passes of K steps each, both inside the clock sampling: the first
    # with events only at its two ends (value, ms_per_step: an event recorded
    # between two kernels of a step costs that step 1.5-3.5 us, since it keeps the
    # next kernel from being scheduled before the previous one ends), the second
    # with events around each step's plan and forward (the forward's own average,
    # the roofline's denominator, and the plan's share).
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    sampler = ClockSampler(local_rank)
    sampler.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(K):
        call.make_plan()
        call.forward()
    t_end.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    total_ms = t_start.elapsed_time(t_end)
    for k in range(K):
        e0, e1, e2 = ev[k]
        e0.record(stream)
        call.make_plan()
        e1.record(stream)
        call.forward()
        e2.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    fwd_ms = sorted(e1.elapsed_time(e2) for _, e1, e2 in ev)
    plan_ms = sorted(e0.elapsed_time(e1) for e0, e1, _ in ev)
    fwd_avg = sum(fwd_ms) / K
    total_ms = max_over_ranks(total_ms, dist)
    assert call.status() == 0, "device error during the timed region"
    ms_per_step = total_ms / K
    T = prob["T"]
    value = T * world / (ms_per_step / 1e3)

    # End to end through the public API: pinned host inputs -> device, plan,
    # forward, result -> host, every step.
    host_in = {k: prob[k].cpu().pin_memory() for k in ("x", "dt", "B", "C", "z", "cu_seqlens")
               if prob[k] is not None}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    y_host = torch.empty(call.y.shape, dtype=call.y.dtype, pin_memory=True)
    fs_host = (torch.empty(call.final_states.shape, dtype=torch.float32, pin_memory=True)
               if call.final_states is not None else None)
    d2h = y_host.numel() * y_host.element_size() + (0 if fs_host is None else fs_host.numel() * 4)

    def e2e_step():
        for k_, t_ in host_in.items():
            prob[k_].copy_(t_, non_blocking=True)
        call.make_plan()
        call.forward()
        y_host.copy_(call.y, non_blocking=True)
        if fs_host is not None:
            fs_host.copy_(call.final_states, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    KE = args.e2e_steps
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(KE):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize()
    e2e_serial_ms = max_over_ranks(a.elapsed_time(b) / KE, dist)

    # The same steps streamed: two device buffer sets and three streams, so that
    # step k's host -> device copies, step k-1's forward and step k-2's results
    # going back overlap (a caller feeding batches through the API would do so).
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    sets = []
    for bi in range(2):
        pb = dict(prob)
        if bi:
            for k_ in host_in:
                pb[k_] = prob[k_].clone()
        sets.append({"prob": pb, "call": m.Call(pb, stream=s_comp),
                     "y": torch.empty(call.y.shape, dtype=call.y.dtype, pin_memory=True),
                     "fs": (torch.empty(call.final_states.shape, dtype=torch.float32, pin_memory=True)
                            if call.final_states is not None else None),
                     "ev_in": torch.cuda.Event(), "ev_comp": torch.cuda.Event(), "ev_out": torch.cuda.Event()})

    def pipe_step(k):
        st = sets[k % 2]
        with torch.cuda.stream(s_in):
            if k >= 2:
                s_in.wait_event(st["ev_comp"])   # the forward two steps back has read these inputs
            for k_, t_ in host_in.items():
                st["prob"][k_].copy_(t_, non_blocking=True)
            st["ev_in"].record(s_in)
        s_comp.wait_event(st["ev_in"])
        if k >= 2:
            s_comp.wait_event(st["ev_out"])      # its outputs of two steps back are home
        st["call"].make_plan()
        st["call"].forward()
        st["ev_comp"].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(st["ev_comp"])
            st["y"].copy_(st["call"].y, non_blocking=True)
            if st["fs"] is not None:
                st["fs"].copy_(st["call"].final_states, non_blocking=True)
            st["ev_out"].record(s_out)

    for k in range(4):
        pipe_step(k)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for k in range(KE):
        pipe_step(k)
    b.record(s_out)
    torch.cuda.synchronize()
    for st in sets:
        assert st["call"].status() == 0, "device error in the streamed end-to-end steps"
    e2e_ms = max_over_ranks(a.elapsed_time(b) / KE, dist)

    khash = kernel_source_hash()
    roofline = roofline_of(cost["bytes"], cost["flops"], fwd_avg, peaks)
    roofline.update({"traffic": read_traffic(khash, args.config + (f"/heads{args.heads_div}" if args.heads_div > 1 else "")), "peak_source": peaks["source"],
                     "algorithmic_bytes": cost["bytes"], "algorithmic_flops": cost["flops"],
                     "kernel": "ssd_varlen_forward", "kernel_ms_avg": round(fwd_avg, 5),
                     "tensor_frac_of_peak": round(cost["flops"] / (fwd_avg / 1e3) / 1e12 / peaks["bf16_tflops"], 4)})
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if prob["dtype"] == "bf16" else "f32",
            "data": "synthetic",
            "config": {"workload": args.config + (f"/heads{args.heads_div}" if args.heads_div > 1 else ""),
                       "T": T, "R": prob["R"], "H": prob["H"], "P": prob["P"], "N": prob["N"], "G": prob["G"],
                       "chunk_size": prob["chunk_size"], "global_batch": prob["R"], "seq_len": T // prob["R"],
                       "parallelism": f"replicas{world}" if world > 1 else "single",
                       "l2": "inputs larger than L2 (no flush)"},
            "roofline": roofline,
            "plan_ms_median": plan_ms[K // 2], "forward_ms_median": fwd_ms[K // 2],
            "gpu_launches": K * (1 + kernels_per_forward),
            "clocks": clocks,
            "e2e": {"value": T * world / (e2e_ms / 1e3), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "mode": "streamed: step k's copies in, step k-1's plan and forward and step k-2's "
                            "results out overlap (three streams, two device buffer sets)",
                    "serial_value": T * world / (e2e_serial_ms / 1e3)},
            "kernel_hash": khash}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(workloads.make_problem(args.config, device="cpu"))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
