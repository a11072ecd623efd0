"""Seeded synthetic inputs for the Mamba2 SSD varlen prefill.

Shared by the tests, the bench and the oracle's callers.  It holds none of the
method's arithmetic: only random draws, request lengths, slot assignments and
buffer shapes.  Every draw is seeded, so the same (config, seed, device) gives
the same tensors.

Value recipe (the same for every workload, following the workloads the SSD
varlen pages describe):
  x, B, C, z ~ N(0, 1); dt ~ N(0, 1) (softplus is applied by the method);
  dt_bias ~ U(-2, -1); A = -exp(U(0, ln 16)); D ~ N(0, 1);
  initial states in a pool of fp32 slots ~ N(0, 1) (tiny case) or N(0, 0.5^2).
Tensor layouts (row-major, last index fastest): x, z, y (T,H,P); B, C (T,G,N);
dt (T,H); dt_bias, A, D (H) fp32; states (..., H, P, N) fp32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass
class Spec:
    name: str
    H: int
    P: int
    N: int
    G: int
    chunk_size: int
    dtype: str                      # "bf16" or "fp32"
    lengths: list | None = None     # fixed lengths, else drawn by length_recipe
    length_recipe: str | None = None
    has_D: bool = True
    has_z: bool = False
    init: str = "none"              # "none", "tiny_req2", "half_even", "all"
    pool_slots: int = 0
    init_std: float = 0.5
    final_dense: bool = True        # write (R,H,P,N) final states
    final_slots: bool = False       # write finals into distinct pool slots
    export_chunks: bool = False
    block_size: int = 0             # block-checkpoint scatter granularity (0 = off)
    extra: dict = field(default_factory=dict)


# The five workloads: a tiny fp32 correctness case and four bf16 layer shapes.
CONFIGS: dict[str, Spec] = {
    "tiny_fp32": Spec("tiny_fp32", H=4, P=16, N=16, G=1, chunk_size=16, dtype="fp32",
                      lengths=[5, 17, 42], has_D=True, has_z=False, init="tiny_req2",
                      pool_slots=3, init_std=1.0),
    "uniform_8x2048": Spec("uniform_8x2048", H=80, P=64, N=128, G=1, chunk_size=256,
                           dtype="bf16", lengths=[2048] * 8, has_D=True, has_z=True),
    "varlen_lognormal_32k": Spec("varlen_lognormal_32k", H=128, P=64, N=128, G=8,
                                 chunk_size=256, dtype="bf16", length_recipe="lognormal64",
                                 has_D=True, has_z=False, init="half_even", pool_slots=256),
    "long_131072": Spec("long_131072", H=64, P=64, N=128, G=1, chunk_size=128,
                        dtype="bf16", lengths=[131072], has_D=True, has_z=False,
                        export_chunks=True),
    "block_ckpt_varlen": Spec("block_ckpt_varlen", H=64, P=128, N=128, G=8, chunk_size=128,
                              dtype="bf16", length_recipe="uniform128", has_D=True,
                              has_z=False, init="all", pool_slots=4096, final_dense=False,
                              final_slots=True, block_size=1024),
}
CONFIG_ORDER = ["tiny_fp32", "uniform_8x2048", "varlen_lognormal_32k", "long_131072",
                "block_ckpt_varlen"]
CONFIG_SEED = {name: i for i, name in enumerate(CONFIG_ORDER)}


def draw_lengths(spec: Spec, seed: int) -> list[int]:
    if spec.lengths is not None:
        return list(spec.lengths)
    rng = np.random.default_rng(seed)
    if spec.length_recipe == "lognormal64":
        # 64 lognormal(mu = ln 400, sigma = 1) draws clipped to [1, 4096], then
        # rescaled so the batch holds exactly 32768 tokens (shape kept).
        raw = np.clip(rng.lognormal(mean=math.log(400.0), sigma=1.0, size=64), 1, 4096)
        lens = np.clip(np.rint(raw * (32768.0 / raw.sum())), 1, 4096).astype(np.int64)
        diff = 32768 - int(lens.sum())
        i = 0
        while diff != 0:
            j = i % 64
            step = 1 if diff > 0 else -1
            if 1 <= lens[j] + step <= 4096:
                lens[j] += step
                diff -= step
            i += 1
        return [int(v) for v in lens]
    if spec.length_recipe == "uniform128":
        return [int(v) for v in rng.integers(1, 8193, size=128)]
    raise ValueError(spec.length_recipe)


def _randn(shape, gen, device, dtype, std=1.0):
    t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def make_problem(spec: Spec | str, seed: int | None = None, device="cpu", lengths=None,
                 num_computed=None, chunk_size=None, canary: float | None = None):
    """Draw one batch.  Returns a dict of tensors plus integer settings.

    lengths / num_computed / chunk_size override the spec (tests use this for
    ragged and resumed cases).  canary: value written into every pool slot that
    no request reads, so tests can check that untouched slots stay intact.
    """
    if isinstance(spec, str):
        spec = CONFIGS[spec]
    if seed is None:
        seed = CONFIG_SEED.get(spec.name, 0)
    lens = list(lengths) if lengths is not None else draw_lengths(spec, seed)
    R = len(lens)
    T = int(sum(lens))
    H, P, N, G = spec.H, spec.P, spec.N, spec.G
    dt_ = torch.float32 if spec.dtype == "fp32" else torch.bfloat16
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    rng = np.random.default_rng(seed + 1000)

    cu = torch.zeros(R + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    prob = {
        "spec": spec.name,
        "lengths": lens,
        "T": T, "R": R, "H": H, "P": P, "N": N, "G": G,
        "chunk_size": int(chunk_size or spec.chunk_size),
        "block_size": spec.block_size,
        "export_chunks": spec.export_chunks,
        "final_dense": spec.final_dense,
        "dtype": spec.dtype,
        "cu_seqlens": cu.to(dev),
        "num_computed": None,
    }
    prob["x"] = _randn((T, H, P), gen, dev, dt_)
    prob["dt"] = _randn((T, H), gen, dev, dt_)
    prob["dt_bias"] = (torch.rand((H,), generator=gen, device=dev) * -1.0 - 1.0)
    prob["A"] = -torch.exp(torch.rand((H,), generator=gen, device=dev) * math.log(16.0))
    prob["B"] = _randn((T, G, N), gen, dev, dt_)
    prob["C"] = _randn((T, G, N), gen, dev, dt_)
    prob["D"] = _randn((H,), gen, dev, torch.float32) if spec.has_D else None
    prob["z"] = _randn((T, H, P), gen, dev, dt_) if spec.has_z else None

    if num_computed is not None:
        prob["num_computed"] = torch.tensor(list(num_computed), dtype=torch.int32, device=dev)
    ncomp = list(num_computed) if num_computed is not None else [0] * R

    S = spec.pool_slots
    init_slots = final_slots = block_table = None
    pool = None
    if spec.init == "tiny_req2":
        init_slots = [-1] * R
        init_slots[min(2, R - 1)] = 1
    elif spec.init == "half_even":
        perm = rng.permutation(S)
        init_slots = [int(perm[i // 2]) if i % 2 == 0 else -1 for i in range(R)]
    elif spec.init == "all":
        perm = rng.permutation(S)
        init_slots = [int(v) for v in perm[:R]]
        used = R
        if spec.final_slots:
            final_slots = [int(v) for v in perm[used:used + R]]
            used += R
        if spec.block_size > 0:
            bs = spec.block_size
            W = max(1, max((ncomp[i] + lens[i]) // bs for i in range(R)))
            block_table = np.full((R, W), -1, dtype=np.int32)
            for i in range(R):
                for j in range(ncomp[i] // bs, (ncomp[i] + lens[i]) // bs):
                    block_table[i, j] = int(perm[used])
                    used += 1
            if used > S:
                raise ValueError("pool too small for the block table")
    if S > 0:
        pool = torch.zeros((S, H, P, N), dtype=torch.float32, device=dev)
        if canary is not None:
            pool.fill_(canary)
        if init_slots is not None:
            for s in sorted({v for v in init_slots if v >= 0}):
                pool[s] = _randn((H, P, N), gen, dev, torch.float32, spec.init_std)
    prob["state_pool"] = pool
    prob["init_slots"] = (torch.tensor(init_slots, dtype=torch.int32, device=dev)
                          if init_slots is not None else None)
    prob["final_slots"] = (torch.tensor(final_slots, dtype=torch.int32, device=dev)
                           if final_slots is not None else None)
    prob["block_table"] = (torch.from_numpy(block_table).to(dev)
                           if block_table is not None else None)
    return prob


def to_oracle(prob: dict, requests=None, heads=None) -> dict:
    """Host float64/int64 copies of a problem, in the form oracle.forward takes.

    Values are upcast exactly (bf16 and fp32 are both subsets of fp64).  With
    ``requests`` only those requests' tokens are copied (repacked in order); the
    original indices are kept under "requests".  With ``heads`` only those
    heads are copied; each selected head then gets its own group (its B and C
    columns are copied alongside), which leaves every head's inputs unchanged.
    """
    def f64(t):
        return None if t is None else t.detach().to("cpu").to(torch.float64).numpy()

    def i64(t):
        return None if t is None else t.detach().to("cpu").to(torch.int64).numpy()

    H = prob["H"]
    G = prob["G"]
    hsel = list(range(H)) if heads is None else [int(h) for h in heads]
    gsel = [h // (H // G) for h in hsel] if heads is not None else list(range(G))
    cu = i64(prob["cu_seqlens"])
    sel = list(range(len(cu) - 1)) if requests is None else [int(i) for i in requests]
    out = {"chunk_size": prob["chunk_size"], "block_size": prob["block_size"],
           "export_chunks": prob["export_chunks"], "requests": sel, "heads": hsel}
    out["dt_bias"] = f64(prob["dt_bias"])[hsel]
    out["A"] = f64(prob["A"])[hsel]
    out["D"] = None if prob["D"] is None else f64(prob["D"])[hsel]
    hidx = torch.tensor(hsel, dtype=torch.long)
    gidx = torch.tensor(gsel, dtype=torch.long)
    pieces = {k: [] for k in ("x", "dt", "B", "C", "z")}
    new_cu = [0]
    for i in sel:
        a, b = int(cu[i]), int(cu[i + 1])
        for k in pieces:
            t = prob[k]
            if t is None:
                continue
            t = t[a:b].detach().to("cpu")
            t = t.index_select(1, gidx if k in ("B", "C") else hidx)
            pieces[k].append(t.to(torch.float64))
        new_cu.append(new_cu[-1] + (b - a))
    for k in pieces:
        out[k] = torch.cat(pieces[k]).numpy() if prob[k] is not None else None
    out["cu_seqlens"] = np.asarray(new_cu, dtype=np.int64)
    nc = prob["num_computed"]
    out["num_computed"] = None if nc is None else i64(nc)[sel]
    for k in ("init_slots", "final_slots"):
        out[k] = None if prob[k] is None else i64(prob[k])[sel]
    bt = prob["block_table"]
    out["block_table"] = None if bt is None else i64(bt)[sel]
    pool = prob["state_pool"]
    if pool is None:
        out["state_pool"] = None
    elif requests is None and heads is None:
        out["state_pool"] = f64(pool)
    else:
        used = set()
        for k in ("init_slots", "final_slots"):
            if out[k] is not None:
                used.update(int(v) for v in out[k] if v >= 0)
        if out["block_table"] is not None:
            used.update(int(v) for v in out["block_table"].ravel() if v >= 0)
        out["state_pool"] = _SparsePool(pool, used, hidx)
    return out


class _SparsePool:
    """Host view of the few pool slots a sampled check touches (avoids copying 17 GB)."""

    def __init__(self, pool, slots, hidx):
        self.shape = (pool.shape[0], len(hidx)) + tuple(pool.shape[2:])
        self.slots = {s: pool[s].detach().to("cpu").index_select(0, hidx).to(torch.float64).numpy()
                      for s in slots}

    def __getitem__(self, s):
        return self.slots[int(s)]

    def __setitem__(self, s, v):
        self.slots[int(s)] = np.asarray(v, dtype=np.float64)

    def copy(self):
        c = _SparsePool.__new__(_SparsePool)
        c.shape = self.shape
        c.slots = {k: v.copy() for k, v in self.slots.items()}
        return c


# ---- decode / speculative-decode steps --------------------------------------
@dataclass
class DecodeSpec:
    """A decode step: R requests, each with a window of new tokens (1 for a plain
    decode step, 1 + drafts for a speculative step), a read anchor per request and
    a write anchor per token in one fp32 state pool."""
    name: str
    H: int
    P: int
    N: int
    G: int
    dtype: str
    windows: list
    has_D: bool = True
    has_z: bool = True
    read_zero_every: int = 0   # every k-th request starts from zeros (read slot -1); 0 = none
    write_every: int = 1       # every k-th token of a window writes its state (the last always does)
    init_std: float = 0.5


DECODE_CONFIGS: dict[str, DecodeSpec] = {
    "decode_tiny_fp32": DecodeSpec("decode_tiny_fp32", H=4, P=16, N=16, G=1, dtype="fp32",
                                   windows=[1, 3, 0, 2], has_z=False, read_zero_every=3, write_every=2),
    # the uniform prefill workload's layer shape, 256 requests with speculative
    # windows of 1 verified + 3 draft tokens, every position keeping its state
    "decode_spec_256x4": DecodeSpec("decode_spec_256x4", H=80, P=64, N=128, G=1, dtype="bf16",
                                    windows=[4] * 256),
}
# a quarter of it, for profiler captures that replay the kernel many times
DECODE_CONFIGS["decode_spec_64x4"] = DecodeSpec("decode_spec_64x4", H=80, P=64, N=128, G=1, dtype="bf16",
                                                windows=[4] * 64)
DECODE_SEED = {"decode_tiny_fp32": 100, "decode_spec_256x4": 101, "decode_spec_64x4": 102}


def make_decode_problem(spec: DecodeSpec | str, seed: int | None = None, device="cpu", windows=None,
                        canary: float | None = None):
    """Draw one decode step.  Read slots are distinct, write slots distinct and
    disjoint from them; the pool holds R + T slots (unused slots hold ``canary``)."""
    if isinstance(spec, str):
        spec = DECODE_CONFIGS[spec]
    if seed is None:
        seed = DECODE_SEED.get(spec.name, 0)
    win = list(windows) if windows is not None else list(spec.windows)
    R, T = len(win), int(sum(win))
    H, P, N, G = spec.H, spec.P, spec.N, spec.G
    dt_ = torch.float32 if spec.dtype == "fp32" else torch.bfloat16
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    rng = np.random.default_rng(seed + 1000)
    cu = torch.zeros(R + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(win, dtype=torch.int64), 0).to(torch.int32)
    prob = {"spec": spec.name, "windows": win, "T": T, "R": R, "H": H, "P": P, "N": N, "G": G,
            "dtype": spec.dtype, "cu_seqlens": cu.to(dev)}
    prob["x"] = _randn((T, H, P), gen, dev, dt_)
    prob["dt"] = _randn((T, H), gen, dev, dt_)
    prob["dt_bias"] = (torch.rand((H,), generator=gen, device=dev) * -1.0 - 1.0)
    prob["A"] = -torch.exp(torch.rand((H,), generator=gen, device=dev) * math.log(16.0))
    prob["B"] = _randn((T, G, N), gen, dev, dt_)
    prob["C"] = _randn((T, G, N), gen, dev, dt_)
    prob["D"] = _randn((H,), gen, dev, torch.float32) if spec.has_D else None
    prob["z"] = _randn((T, H, P), gen, dev, dt_) if spec.has_z else None
    S = R + T
    perm = rng.permutation(S)
    read = [int(v) for v in perm[:R]]
    if spec.read_zero_every:
        read = [-1 if i % spec.read_zero_every == spec.read_zero_every - 1 else s for i, s in enumerate(read)]
    write = [-1] * T
    k = R
    for i in range(R):
        a, L = int(cu[i]), win[i]
        for j in range(L):
            if j == L - 1 or j % spec.write_every == spec.write_every - 1:
                write[a + j] = int(perm[k])
                k += 1
    pool = torch.full((S, H, P, N), 0.0 if canary is None else canary, dtype=torch.float32, device=dev)
    for s in read:
        if s >= 0:
            pool[s] = _randn((H, P, N), gen, dev, torch.float32, spec.init_std)
    prob["state_pool"] = pool
    prob["read_slots"] = torch.tensor(read, dtype=torch.int32, device=dev)
    prob["write_slots"] = torch.tensor(write, dtype=torch.int32, device=dev)
    return prob


def to_oracle_decode(prob: dict, requests=None, heads=None) -> dict:
    """Host float64 copies of a decode step, in the form oracle.decode takes.  With
    ``requests`` / ``heads`` only those are copied (requests repacked in order, each
    selected head its own group); the pool is then a view of the read slots only."""
    def f64(t):
        return None if t is None else t.detach().to("cpu").to(torch.float64).numpy()

    H, G = prob["H"], prob["G"]
    hsel = list(range(H)) if heads is None else [int(h) for h in heads]
    cu = prob["cu_seqlens"].detach().to("cpu").to(torch.int64).numpy()
    sel = list(range(len(cu) - 1)) if requests is None else [int(i) for i in requests]
    hidx = torch.tensor(hsel, dtype=torch.long)
    gidx = torch.tensor([h // (H // G) for h in hsel] if heads is not None else list(range(G)),
                        dtype=torch.long)
    toks = torch.tensor([t for i in sel for t in range(int(cu[i]), int(cu[i + 1]))], dtype=torch.long)
    new_cu = np.zeros(len(sel) + 1, dtype=np.int64)
    new_cu[1:] = np.cumsum([int(cu[i + 1] - cu[i]) for i in sel])

    def take(t, gdim=False):
        if t is None:
            return None
        t = t.detach().to("cpu")[toks]
        return f64(t.index_select(1, gidx if gdim else hidx))

    read = prob["read_slots"].detach().to("cpu").numpy()
    write = prob["write_slots"].detach().to("cpu").numpy() if prob.get("write_slots") is not None else None
    out = {"cu_seqlens": new_cu, "x": take(prob["x"]), "dt": take(prob["dt"]),
           "B": take(prob["B"], True), "C": take(prob["C"], True), "z": take(prob.get("z")),
           "dt_bias": f64(prob["dt_bias"])[hsel], "A": f64(prob["A"])[hsel],
           "D": None if prob.get("D") is None else f64(prob["D"])[hsel],
           "read_slots": read[sel], "write_slots": None if write is None else write[toks.numpy()],
           "requests": sel, "heads": hsel, "tokens": toks.numpy()}
    pool = prob["state_pool"]
    if requests is None and heads is None:
        out["state_pool"] = f64(pool)
    else:
        out["state_pool"] = _SparsePool(pool, [int(s) for s in read[sel] if 0 <= s < pool.shape[0]], hidx)
    return out


# ---- varlen causal conv1d ----------------------------------------------------
@dataclass
class ConvSpec:
    """A varlen causal depthwise conv1d over D channels with a W-wide kernel; every
    request reads its conv state from one slot and writes it to another."""
    name: str
    D: int
    W: int
    dtype: str
    lengths: list
    silu: bool = True
    has_bias: bool = True
    read_zero_every: int = 0   # every k-th request starts from zeros (read slot -1)


CONV_CONFIGS: dict[str, ConvSpec] = {
    "conv_tiny_fp32": ConvSpec("conv_tiny_fp32", D=16, W=4, dtype="fp32", lengths=[5, 17, 0, 2, 42],
                               read_zero_every=2),
    # the conv of the uniform prefill workload's layer: x, B and C channels
    # (H P + 2 G N = 80 * 64 + 2 * 128) of 8 requests x 2048 tokens
    "conv_uniform_8x2048": ConvSpec("conv_uniform_8x2048", D=5376, W=4, dtype="bf16", lengths=[2048] * 8),
}
CONV_SEED = {"conv_tiny_fp32": 200, "conv_uniform_8x2048": 201}


def make_conv_problem(spec: ConvSpec | str, seed: int | None = None, device="cpu", lengths=None,
                      canary: float | None = None):
    if isinstance(spec, str):
        spec = CONV_CONFIGS[spec]
    if seed is None:
        seed = CONV_SEED.get(spec.name, 0)
    lens = list(lengths) if lengths is not None else list(spec.lengths)
    R, T = len(lens), int(sum(lens))
    D, W = spec.D, spec.W
    dt_ = torch.float32 if spec.dtype == "fp32" else torch.bfloat16
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    rng = np.random.default_rng(seed + 1000)
    cu = torch.zeros(R + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    prob = {"spec": spec.name, "lengths": lens, "T": T, "R": R, "D": D, "W": W, "dtype": spec.dtype,
            "cu_seqlens": cu.to(dev), "silu": spec.silu}
    prob["x"] = _randn((T, D), gen, dev, dt_)
    prob["weight"] = _randn((D, W), gen, dev, torch.float32, 0.5)
    prob["bias"] = _randn((D,), gen, dev, torch.float32, 0.5) if spec.has_bias else None
    S = 2 * R
    perm = rng.permutation(S)
    read = [int(v) for v in perm[:R]]
    if spec.read_zero_every:
        read = [-1 if i % spec.read_zero_every == spec.read_zero_every - 1 else s for i, s in enumerate(read)]
    write = [int(v) for v in perm[R:]]
    pool = torch.full((S, D, W - 1), 0.0 if canary is None else canary, dtype=dt_, device=dev)
    for s in read:
        if s >= 0:
            pool[s] = _randn((D, W - 1), gen, dev, dt_)
    prob["conv_pool"] = pool
    prob["read_slots"] = torch.tensor(read, dtype=torch.int32, device=dev)
    prob["write_slots"] = torch.tensor(write, dtype=torch.int32, device=dev)
    return prob


def to_oracle_conv(prob: dict, channels=None) -> dict:
    """Host float64 copies of a conv1d problem for oracle.conv1d (optionally a channel subset)."""
    def f64(t):
        return None if t is None else t.detach().to("cpu").to(torch.float64).numpy()

    cidx = None if channels is None else torch.tensor(list(channels), dtype=torch.long)

    def cols(t, dim):
        if t is None or cidx is None:
            return f64(t)
        return f64(t.detach().to("cpu").index_select(dim, cidx))

    return {"x": cols(prob["x"], 1), "weight": cols(prob["weight"], 0), "bias": cols(prob.get("bias"), 0),
            "cu_seqlens": prob["cu_seqlens"].detach().to("cpu").numpy().astype(np.int64),
            "conv_pool": cols(prob["conv_pool"], 1),
            "read_slots": prob["read_slots"].detach().to("cpu").numpy(),
            "write_slots": prob["write_slots"].detach().to("cpu").numpy(), "silu": prob["silu"]}


# ---- gated delta rule (GDN) prefill ------------------------------------------
# Value recipe: q, k, v ~ N(0, 1) (q and k are l2-normalised inside the method
# when l2norm is set); per value head a decay rate a_h = exp(U(0, ln 16)) and
# g = -a_h * softplus(N(0, 1) - 4) (log decays of about -0.005 to -1); beta =
# sigmoid(N(0, 1)); initial states N(0, 0.5^2).  Layouts: q, k (T,Hk,K); v, o
# (T,Hv,V); g, beta (T,Hv) fp32; states (..., Hv, K, V) fp32.

@dataclass
class GdnSpec:
    name: str
    Hk: int
    Hv: int
    K: int
    V: int
    lengths: list
    dtype: str = "bf16"
    l2norm: bool = True
    init: str = "none"          # "none" or "all" (every request reads a slot)
    final_slots: bool = False
    export_chunks: bool = False
    block_size: int = 0
    final_dense: bool = True


GDN_CONFIGS: dict[str, GdnSpec] = {
    "gdn_small": GdnSpec("gdn_small", Hk=2, Hv=4, K=128, V=64, lengths=[37, 64, 1, 130, 0, 200],
                         init="all", final_slots=True, export_chunks=True, block_size=128),
    # the uniform 8 x 2048 token layout in a GDN layer shape: 16 key heads, 32 value
    # heads, 128 x 128 state per value head
    "gdn_uniform_8x2048": GdnSpec("gdn_uniform_8x2048", Hk=16, Hv=32, K=128, V=128, lengths=[2048] * 8),
}
GDN_SEED = {"gdn_small": 300, "gdn_uniform_8x2048": 301}


def make_gdn_problem(spec: GdnSpec | str, seed: int | None = None, device="cpu", lengths=None,
                     num_computed=None, canary: float | None = None):
    """Draw one GDN prefill.  With init "all" every request reads a distinct slot;
    final slots and block-table slots are distinct from them and from each other
    (unused pool slots hold ``canary``)."""
    if isinstance(spec, str):
        spec = GDN_CONFIGS[spec]
    if seed is None:
        seed = GDN_SEED.get(spec.name, 0)
    lens = list(lengths) if lengths is not None else list(spec.lengths)
    R, T = len(lens), int(sum(lens))
    Hk, Hv, K, V = spec.Hk, spec.Hv, spec.K, spec.V
    dt_ = torch.float32 if spec.dtype == "fp32" else torch.bfloat16
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    rng = np.random.default_rng(seed + 1000)
    cu = torch.zeros(R + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    prob = {"spec": spec.name, "lengths": lens, "T": T, "R": R, "cu_seqlens": cu.to(dev),
            "block_size": spec.block_size, "export_chunks": spec.export_chunks, "l2norm": spec.l2norm,
            "final_dense": spec.final_dense, "scale": None}
    prob["q"] = _randn((T, Hk, K), gen, dev, dt_)
    prob["k"] = _randn((T, Hk, K), gen, dev, dt_)
    prob["v"] = _randn((T, Hv, V), gen, dev, dt_)
    rate = torch.exp(torch.rand((Hv,), generator=gen, device=dev) * math.log(16.0))
    prob["g"] = -rate * torch.nn.functional.softplus(_randn((T, Hv), gen, dev, torch.float32) - 4.0)
    prob["beta"] = torch.sigmoid(_randn((T, Hv), gen, dev, torch.float32))
    ncomp = list(num_computed) if num_computed is not None else [0] * R
    prob["num_computed"] = (torch.tensor(ncomp, dtype=torch.int32, device=dev)
                            if num_computed is not None else None)
    init_slots = final_slots = block_table = pool = None
    if spec.init == "all" or spec.final_slots or spec.block_size:
        bs = spec.block_size
        W = max(1, max((ncomp[i] + lens[i]) // bs for i in range(R))) if bs else 0
        S = 2 * R + (R * W if bs else 0) + 4
        perm = rng.permutation(S)
        used = 0
        if spec.init == "all":
            init_slots = [int(v) for v in perm[:R]]
            used = R
        if spec.final_slots:
            final_slots = [int(v) for v in perm[used:used + R]]
            used += R
        if bs:
            block_table = np.full((R, W), -1, dtype=np.int32)
            for i in range(R):
                for j in range(ncomp[i] // bs, (ncomp[i] + lens[i]) // bs):
                    block_table[i, j] = int(perm[used])
                    used += 1
        pool = torch.full((S, Hv, K, V), 0.0 if canary is None else canary, dtype=torch.float32, device=dev)
        for s in (init_slots or []):
            pool[s] = _randn((Hv, K, V), gen, dev, torch.float32, 0.5)
    prob["state_pool"] = pool
    prob["init_slots"] = None if init_slots is None else torch.tensor(init_slots, dtype=torch.int32, device=dev)
    prob["final_slots"] = None if final_slots is None else torch.tensor(final_slots, dtype=torch.int32, device=dev)
    prob["block_table"] = None if block_table is None else torch.from_numpy(block_table).to(dev)
    return prob


def to_oracle_gdn(prob: dict, requests=None, heads=None) -> dict:
    """Host float64 copies of a GDN problem, in the form oracle.gdn.gdn_forward takes.
    With ``requests`` / ``heads`` only those are copied (requests repacked in order;
    each selected value head gets its own copy of its key head's q and k; slots,
    num_computed and the block table follow the selected requests)."""
    def f64(t):
        return None if t is None else t.detach().to("cpu").to(torch.float64).numpy()

    Hk, Hv = prob["q"].shape[1], prob["v"].shape[1]
    cu = prob["cu_seqlens"].detach().to("cpu").to(torch.int64).numpy()
    sel = list(range(len(cu) - 1)) if requests is None else [int(i) for i in requests]
    toks = torch.tensor([t for i in sel for t in range(int(cu[i]), int(cu[i + 1]))], dtype=torch.long)
    new_cu = np.zeros(len(sel) + 1, dtype=np.int64)
    new_cu[1:] = np.cumsum([int(cu[i + 1] - cu[i]) for i in sel])
    hsel = list(range(Hv)) if heads is None else [int(h) for h in heads]
    kidx = torch.tensor([h // (Hv // Hk) for h in hsel] if heads is not None else list(range(Hk)), dtype=torch.long)
    hidx = torch.tensor(hsel, dtype=torch.long)

    def take(t, key=False):
        return f64(t.detach().to("cpu")[toks].index_select(1, kidx if key else hidx))

    def pick(t):
        return None if t is None else t.detach().to("cpu").numpy()[sel]

    pool = prob.get("state_pool")
    out = {"q": take(prob["q"], True), "k": take(prob["k"], True), "v": take(prob["v"]),
           "g": take(prob["g"]), "beta": take(prob["beta"]), "cu_seqlens": new_cu,
           "num_computed": pick(prob.get("num_computed")), "chunk_size": 64,
           "block_size": prob.get("block_size") or 0, "block_table": pick(prob.get("block_table")),
           "state_pool": None if pool is None else f64(pool.detach().to("cpu").index_select(1, hidx)),
           "init_slots": pick(prob.get("init_slots")), "final_slots": pick(prob.get("final_slots")),
           "export_chunks": bool(prob.get("export_chunks")), "scale": prob.get("scale"),
           "l2norm": bool(prob.get("l2norm")), "requests": sel, "heads": hsel, "tokens": toks.numpy()}
    return out
