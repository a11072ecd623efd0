"""CPU fp64 oracle of the gated delta rule (GDN) varlen prefill -- TEST INFRASTRUCTURE ONLY.

Only tests/, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline leg may use
this module; the product library never loads it and it never loads the product.

"Automatic prefix caching for GDN hybrid models (mamba_cache_mode=all) with MTP
speculative decoding" (Purpose, Kernels/layers) runs the gated-delta-rule layers
of GDN hybrid models through a chunk kernel that exports per-chunk intermediate
states, and checkpoints them with the same block-aligned scatter as the Mamba2
path.  The pages print no formula for the rule; this oracle takes the published
gated delta rule (Yang, Kautz and Hatamizadeh, "Gated Delta Networks: Improving
Mamba2 with Delta Rule", 2024), with the state S a K x V matrix per value head,
token by token for every request i and value head h (key head h // (Hv/Hk)):

    q~, k~ = q_t, k_t, or q_t / sqrt(|q_t|^2 + 1e-6), k_t / sqrt(|k_t|^2 + 1e-6)
    S      <- exp(g_t) S                          (the gate: a scalar decay)
    u      =  beta_t (v_t - S^T k~)               (the delta: what k~ should read)
    S      <- S + k~ u^T                          (the rank-one write)
    o_t    =  scale * S^T q~                      (after the write)

S starts from state_pool[init_slots[i]] (zeros when absent or < 0).  State
outputs follow the same index rules as the SSD path (``checkpoints``): chunks
cut at absolute multiples of chunk_size, export row first_chunk[i] + j = the
state after chunk j, block checkpoints through block_table, final states.
Everything in fp64 from the exact inputs.
"""
from __future__ import annotations

import numpy as np

from . import checkpoints

L2_EPS = 1e-6


def _l2n(a: np.ndarray) -> np.ndarray:
    return a / np.sqrt(np.sum(a * a, axis=-1, keepdims=True) + L2_EPS)


def gdn_forward(prob: dict, requests=None) -> dict:
    """prob: q (T,Hk,K), k (T,Hk,K), v (T,Hv,V), g (T,Hv), beta (T,Hv), cu_seqlens (R+1),
    num_computed|None (R), chunk_size, block_size, block_table|None (R,W),
    state_pool|None (S,Hv,K,V), init_slots|None, final_slots|None, export_chunks (bool),
    scale|None (K^-1/2), l2norm (bool).  ``requests`` restricts the work to a sample.

    Returns {"o": (T,Hv,V), "final_states": (R,Hv,K,V), "chunk_states": (n,Hv,K,V)|None,
             "state_pool": pool after the writes|None, "first_chunk": (R+1)}."""
    q = np.asarray(prob["q"], dtype=np.float64)
    k = np.asarray(prob["k"], dtype=np.float64)
    v = np.asarray(prob["v"], dtype=np.float64)
    g = np.asarray(prob["g"], dtype=np.float64)
    beta = np.asarray(prob["beta"], dtype=np.float64)
    T, Hk, K = q.shape
    Hv, V = v.shape[1], v.shape[2]
    ratio = Hv // Hk
    scale = prob.get("scale")
    scale = K ** -0.5 if scale is None else float(scale)
    if prob.get("l2norm"):
        q, k = _l2n(q), _l2n(k)
    cu = np.asarray(prob["cu_seqlens"], dtype=np.int64)
    R = cu.shape[0] - 1
    ncomp = prob.get("num_computed")
    pool = prob.get("state_pool")
    init = prob.get("init_slots")
    recs, first_chunk = checkpoints.checkpoint_records(
        np.diff(cu), ncomp, int(prob["chunk_size"]), int(prob.get("block_size") or 0),
        prob.get("block_table"), bool(prob.get("export_chunks", False)))
    want = {}
    for r in recs:
        want.setdefault((r.request, r.k), []).append(r)

    o = np.zeros((T, Hv, V))
    final = np.zeros((R, Hv, K, V))
    chunk_states = np.zeros((first_chunk[R], Hv, K, V)) if prob.get("export_chunks") else None
    new_pool = None if pool is None else np.array(pool, dtype=np.float64, copy=True)
    heads_k = np.arange(Hv) // ratio
    for i in (range(R) if requests is None else requests):
        S = np.zeros((Hv, K, V))
        if init is not None and int(init[i]) >= 0:
            S = np.array(pool[int(init[i])], dtype=np.float64, copy=True)
        a, b = int(cu[i]), int(cu[i + 1])
        for j, t in enumerate(range(a, b)):
            kt = k[t, heads_k]                                   # (Hv, K)
            qt = q[t, heads_k]
            S *= np.exp(g[t])[:, None, None]
            u = beta[t][:, None] * (v[t] - np.einsum("hk,hkv->hv", kt, S))
            S += kt[:, :, None] * u[:, None, :]
            o[t] = scale * np.einsum("hk,hkv->hv", qt, S)
            for r in want.get((i, j + 1), []):
                if r.kind == "chunk":
                    chunk_states[r.dest] = S
                else:
                    new_pool[r.dest] = S
        final[i] = S
    fs = prob.get("final_slots")
    if new_pool is not None and fs is not None:
        for i in (range(R) if requests is None else requests):
            if int(fs[i]) >= 0:
                new_pool[int(fs[i])] = final[i]
    return {"o": o, "final_states": final, "chunk_states": chunk_states, "state_pool": new_pool,
            "first_chunk": np.asarray(first_chunk, dtype=np.int64)}
