"""CPU fp64 oracle for the Mamba2 SSD varlen prefill -- TEST INFRASTRUCTURE ONLY.

Only tests/, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline leg may
import this package.  The product library never loads it, and it never loads
the product library: the two share no code.  The only module both sides use is
the seeded input generator (``workloads``), which holds none of the method's
arithmetic.

Layers:
* ``ssd_oracle.c`` -- the token-by-token fp64 recurrence (see its header).
* ``checkpoints``  -- which token counts feed the chunk-state export, the
  block-checkpoint scatter and the final state (index arithmetic only).
* ``forward``      -- applies the library's call semantics on top: initial
  states gathered from the pool by slot (-1 = zeros), outputs scattered back
  by slot, so a test can compare every buffer the library writes.

Every function here is pinned by tests/test_oracle_pins.py (brute-force
quadratic SSD form, closed forms for A = 0, B = 0 and T = 1, packing and
split-state invariance, hand-worked golden values).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from . import checkpoints

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libssd_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ssd_oracle.c with the host compiler (plain -O2, no fast-math)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        f = lib.ssd_oracle_varlen
        P = ctypes.c_void_p
        f.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                      ctypes.c_int32, ctypes.c_int32,
                      P, P, P, P, P, P, P, P, P, P, P, P,
                      ctypes.c_int64, P, P, P, P, ctypes.c_int]
        f.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def recurrence(cu_seqlens, x, dt, dt_bias, A, B, C, D=None, z=None, h0=None,
               rec_k=None, tasks=None, n_threads: int = 0):
    """Run the fp64 recurrence over a packed batch.

    cu_seqlens (R+1) ints; x (T,H,P); dt (T,H); dt_bias, A, D (H); B, C (T,G,N);
    z (T,H,P) or None; h0 (R,H,P,N) or None.  rec_k: optional list of R
    ascending lists of token counts (0..L_i) after which the state is recorded.
    tasks: optional (n,2) array of (request, head) pairs to compute (others are
    left at zero).  Returns (y, h_final, rec_states) as float64 arrays.
    """
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    x, dt, dt_bias, A, B, C = map(_f64, (x, dt, dt_bias, A, B, C))
    D, z, h0 = _f64(D), _f64(z), _f64(h0)
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    R = cu.shape[0] - 1
    y = np.zeros((T, H, P), dtype=np.float64)
    h_final = np.zeros((R, H, P, N), dtype=np.float64)
    rec_off = rec_arr = rec_states = None
    if rec_k is not None:
        counts = [len(v) for v in rec_k]
        rec_off = np.zeros(R + 1, dtype=np.int64)
        rec_off[1:] = np.cumsum(counts)
        rec_arr = np.ascontiguousarray(
            np.concatenate([np.asarray(v, dtype=np.int64) for v in rec_k])
            if rec_off[-1] > 0 else np.zeros(1, dtype=np.int64))
        rec_states = np.zeros((max(int(rec_off[-1]), 1), H, P, N), dtype=np.float64)
    tk = None
    n_tasks = 0
    if tasks is not None:
        tk = np.ascontiguousarray(np.asarray(tasks, dtype=np.int32).reshape(-1, 2))
        n_tasks = tk.shape[0]
    rc = _load().ssd_oracle_varlen(
        T, R, H, P, N, G, _ptr(cu), _ptr(x), _ptr(dt), _ptr(dt_bias), _ptr(A), _ptr(B),
        _ptr(C), _ptr(D), _ptr(z), _ptr(h0), _ptr(rec_off), _ptr(rec_arr), n_tasks,
        _ptr(tk), _ptr(y), _ptr(h_final), _ptr(rec_states), int(n_threads))
    if rc != 0:
        raise ValueError(f"ssd_oracle_varlen failed with code {rc}")
    if rec_states is not None:
        rec_states = rec_states[: int(rec_off[-1])]
    return y, h_final, rec_states


def forward(prob: dict, n_threads: int = 0, requests=None, heads=None):
    """The library's call semantics, computed by the oracle.

    ``prob`` holds numpy arrays (any float dtype; upcast exactly to fp64):
      x, dt, dt_bias, A, B, C, D|None, z|None, cu_seqlens, num_computed|None,
      chunk_size, block_size, state_pool|None (S,H,P,N), init_slots|None,
      final_slots|None, block_table|None (R,W), export_chunks (bool).
    ``requests``/``heads`` restrict the work to a sample; outputs of the other
    (request, head) pairs are left at zero and only the sampled ones may be
    compared.

    Returns a dict with y (T,H,P), final_states (R,H,P,N), chunk_states
    (n_chunks,H,P,N) or None, and state_pool (the pool after this call's
    writes; untouched slots keep their input values) or None.
    """
    cu = np.asarray(prob["cu_seqlens"], dtype=np.int64)
    R = cu.shape[0] - 1
    lengths = np.diff(cu)
    ncomp = prob.get("num_computed")
    x = prob["x"]
    T, H, P = x.shape
    N = prob["B"].shape[2]
    pool = prob.get("state_pool")
    init_slots = prob.get("init_slots")
    h0 = None
    if init_slots is not None:
        h0 = np.zeros((R, H, P, N), dtype=np.float64)
        for i in range(R):
            s = int(init_slots[i])
            if s >= 0:
                h0[i] = pool[s]
    recs, first_chunk = checkpoints.checkpoint_records(
        lengths, ncomp, int(prob["chunk_size"]), int(prob.get("block_size") or 0),
        prob.get("block_table"), bool(prob.get("export_chunks", False)))
    rec_k = [[] for _ in range(R)]
    for r in recs:
        if not rec_k[r.request] or rec_k[r.request][-1] != r.k:
            rec_k[r.request].append(r.k)
    tasks = None
    if requests is not None or heads is not None:
        req_list = range(R) if requests is None else requests
        head_list = range(H) if heads is None else heads
        tasks = [(int(i), int(h)) for i in req_list for h in head_list]
    y, hf, rec = recurrence(cu, x, prob["dt"], prob["dt_bias"], prob["A"], prob["B"],
                            prob["C"], prob.get("D"), prob.get("z"), h0, rec_k, tasks,
                            n_threads)
    # position of (request, k) inside rec
    row_of = {}
    row = 0
    for i in range(R):
        for k in rec_k[i]:
            row_of[(i, k)] = row
            row += 1
    out = {"y": y, "final_states": hf, "chunk_states": None, "state_pool": None}
    if prob.get("export_chunks"):
        cs = np.zeros((first_chunk[R], H, P, N), dtype=np.float64)
        for r in recs:
            if r.kind == "chunk":
                cs[r.dest] = rec[row_of[(r.request, r.k)]]
        out["chunk_states"] = cs
    if pool is not None:
        new_pool = (np.array(pool, dtype=np.float64, copy=True)
                    if isinstance(pool, np.ndarray) else pool.copy())
        for r in recs:
            if r.kind == "block":
                new_pool[r.dest] = rec[row_of[(r.request, r.k)]]
        fs = prob.get("final_slots")
        if fs is not None:
            for i in range(R):
                if int(fs[i]) >= 0:
                    new_pool[int(fs[i])] = hf[i]
        out["state_pool"] = new_pool
    out["first_chunk"] = np.asarray(first_chunk, dtype=np.int64)
    return out


def decode(prob: dict, n_threads: int = 0):
    """The decode step's call semantics (ssd_varlen_decode), computed by the oracle.

    "Automatic prefix caching for GDN hybrid models (mamba_cache_mode=all) with MTP
    speculative decoding", Purpose (Kernels/layers): decode kernels with dual
    read/write state anchors.  Each request's window of new tokens is a short
    varlen sequence of the recurrence above: its state starts from
    state_pool[read_slots[i]] (zeros when the slot is < 0) and the state after
    token t is written to state_pool[write_slots[t]] when that slot is >= 0.

    ``prob`` holds numpy arrays (upcast exactly to fp64): x, dt, dt_bias, A, B, C,
    D|None, z|None, cu_seqlens (window boundaries), state_pool (indexable by slot,
    (H,P,N) per slot), read_slots (R), write_slots (T) or None.

    Returns {"y": (T,H,P), "writes": {slot: (H,P,N) state written there}}.
    """
    cu = np.asarray(prob["cu_seqlens"], dtype=np.int64)
    R = cu.shape[0] - 1
    x = prob["x"]
    T, H, P = x.shape
    N = prob["B"].shape[2]
    pool = prob["state_pool"]
    S = pool.shape[0]
    read = np.asarray(prob["read_slots"], dtype=np.int64)
    write = prob.get("write_slots")
    write = np.full(T, -1, dtype=np.int64) if write is None else np.asarray(write, dtype=np.int64)
    h0 = np.zeros((R, H, P, N), dtype=np.float64)
    for i in range(R):
        if 0 <= read[i] < S:
            h0[i] = pool[int(read[i])]
    rec_k = [[t - int(cu[i]) + 1 for t in range(int(cu[i]), int(cu[i + 1])) if 0 <= write[t] < S]
             for i in range(R)]
    y, _, rec = recurrence(cu, x, prob["dt"], prob["dt_bias"], prob["A"], prob["B"], prob["C"],
                           prob.get("D"), prob.get("z"), h0, rec_k, None, n_threads)
    writes = {}
    row = 0
    for i in range(R):
        for t in range(int(cu[i]), int(cu[i + 1])):
            if 0 <= write[t] < S:
                writes[int(write[t])] = rec[row]
                row += 1
    return {"y": y, "writes": writes}
