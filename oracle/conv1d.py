"""CPU fp64 oracle of the varlen causal depthwise conv1d -- TEST INFRASTRUCTURE ONLY.

Only tests/, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline leg may use
this module; the product library never loads it and it never loads the product.

What it computes ("[Model] Mamba2 varlen and metadata refactor", Purpose items
1-2: varlen inputs packed by cu_seqlens, metadata from the batch; "Automatic
prefix caching for GDN hybrid models (mamba_cache_mode=all) with MTP
speculative decoding", Purpose, Kernels/layers: the causal_conv1d decode kernel
with dual read/write state anchors), per request i over its packed tokens
[cu[i], cu[i+1]) and per channel c:

    xin      = [conv_state_in (W-1 values, oldest first), x[cu[i]:cu[i+1], c]]
    y[t, c]  = act(bias[c] + sum_{k=0}^{W-1} weight[c, k] * xin[j + k])   (j = t - cu[i])
    conv_state_out = the last W-1 values of xin

conv_state_in is conv_pool[read_slots[i]] (zeros when the slot is < 0);
conv_state_out goes to conv_pool[write_slots[i]] when that slot is >= 0.
act is the identity or SiLU.  Everything in fp64 from the exact inputs.
"""
from __future__ import annotations

import numpy as np


def conv1d(prob: dict) -> dict:
    """prob: x (T,D), weight (D,W), bias (D)|None, cu_seqlens (R+1), conv_pool (S,D,W-1),
    read_slots (R)|None, write_slots (R)|None, silu (bool).

    Returns {"y": (T,D), "writes": {slot: (D,W-1) state written there},
             "final": (R,D,W-1) the conv state after each request}."""
    x = np.asarray(prob["x"], dtype=np.float64)
    w = np.asarray(prob["weight"], dtype=np.float64)
    D, W = w.shape
    bias = np.zeros(D) if prob.get("bias") is None else np.asarray(prob["bias"], dtype=np.float64)
    cu = np.asarray(prob["cu_seqlens"], dtype=np.int64)
    R = cu.shape[0] - 1
    pool = prob["conv_pool"]
    S = pool.shape[0]
    read = prob.get("read_slots")
    write = prob.get("write_slots")
    y = np.zeros_like(x)
    final = np.zeros((R, D, W - 1))
    writes = {}
    for i in range(R):
        a, b = int(cu[i]), int(cu[i + 1])
        init = np.zeros((D, W - 1))
        if read is not None and 0 <= int(read[i]) < S:
            init = np.asarray(pool[int(read[i])], dtype=np.float64)
        xin = np.concatenate([init, x[a:b].T], axis=1)           # (D, W-1+L)
        for j in range(b - a):
            acc = bias + (w * xin[:, j:j + W]).sum(axis=1)
            y[a + j] = acc / (1.0 + np.exp(-acc)) if prob.get("silu") else acc
        final[i] = xin[:, xin.shape[1] - (W - 1):]
        if write is not None and 0 <= int(write[i]) < S:
            writes[int(write[i])] = final[i]
    return {"y": y, "writes": writes, "final": final}
