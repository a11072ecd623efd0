"""Pins of the gated-delta-rule oracle (oracle.gdn) -- CPU.

Fixed against: a scalar case worked by hand; the closed form of a pure decay
(beta = 0); the delta rule's exact retrieval and overwrite with orthonormal keys
(its defining property); an independent chunked formulation (the WY form: a
unit-lower-triangular solve per chunk, written here with numpy.linalg.solve);
split-and-resume, packing, the l2-norm flag and the key-head sharing (GQA).
"""
import math

import numpy as np
import pytest

from oracle.gdn import gdn_forward


def _prob(rng, lengths, Hk=2, Hv=4, K=8, V=6, init=True, l2norm=False, Q=4, scale=None):
    T = int(sum(lengths))
    R = len(lengths)
    S = 3 * R + 4
    p = {"q": rng.normal(size=(T, Hk, K)), "k": rng.normal(size=(T, Hk, K)), "v": rng.normal(size=(T, Hv, V)),
         "g": -rng.uniform(0.0, 0.7, size=(T, Hv)), "beta": rng.uniform(0.0, 1.0, size=(T, Hv)),
         "cu_seqlens": np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64), "num_computed": None,
         "chunk_size": Q, "block_size": 0, "block_table": None,
         "state_pool": rng.normal(size=(S, Hv, K, V)) * 0.5,
         "init_slots": np.arange(R) if init else None, "final_slots": np.arange(R, 2 * R),
         "export_chunks": True, "scale": scale, "l2norm": l2norm}
    if not l2norm:  # keep the un-normalised keys small enough for a stable delta rule
        p["q"] /= math.sqrt(K)
        p["k"] /= math.sqrt(K)
    return p


def test_scalar_worked_by_hand():
    # K = V = 1, one head, scale 1.  S0 = 2; token 1: g = ln 0.5, beta 0.5, k 1, v 3, q 1
    #   S = 0.5*2 = 1, u = 0.5*(3 - 1*1) = 1, S = 1 + 1*1 = 2, o = 2
    # token 2: g = 0, beta 1, k 2, v 1, q 1
    #   S = 2, u = 1*(1 - 2*2) = -3, S = 2 + 2*(-3) = -4, o = -4
    p = {"q": np.array([[[1.0]], [[1.0]]]), "k": np.array([[[1.0]], [[2.0]]]), "v": np.array([[[3.0]], [[1.0]]]),
         "g": np.array([[math.log(0.5)], [0.0]]), "beta": np.array([[0.5], [1.0]]),
         "cu_seqlens": np.array([0, 2]), "chunk_size": 16, "state_pool": np.array([[[[2.0]]]]),
         "init_slots": np.array([0]), "scale": 1.0}
    out = gdn_forward(p)
    np.testing.assert_allclose(out["o"][:, 0, 0], [2.0, -4.0], rtol=0, atol=1e-14)
    np.testing.assert_allclose(out["final_states"][0, 0], [[-4.0]], rtol=0, atol=1e-14)


def test_beta_zero_is_pure_decay():
    rng = np.random.default_rng(1)
    p = _prob(rng, [9, 5])
    p["beta"][:] = 0.0
    out = gdn_forward(p)
    cu = p["cu_seqlens"]
    for i in range(2):
        S0 = p["state_pool"][p["init_slots"][i]]
        G = np.cumsum(p["g"][cu[i]:cu[i + 1]], axis=0)          # (L, Hv)
        for j, t in enumerate(range(cu[i], cu[i + 1])):
            for h in range(4):
                ref = 8 ** -0.5 * math.exp(G[j, h]) * (S0[h].T @ p["q"][t, h // 2])
                np.testing.assert_allclose(out["o"][t, h], ref, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(out["final_states"][i], np.exp(G[-1])[:, None, None] * S0, rtol=1e-12)


def test_delta_rule_exact_retrieval_and_overwrite():
    # Orthonormal keys, no decay, beta = 1, zero initial state: a write makes the
    # state return exactly the written value for that key, and a second write to
    # the same key replaces it.  Queries (beta = 0) read what is stored.
    K = V = 8
    e = np.eye(K)
    vals = np.arange(1, 4 * V + 1, dtype=np.float64).reshape(4, V) / 7.0
    keys = [e[0], e[3], e[0], e[5]]                 # key 0 written twice
    qs = keys + [e[3], e[0], e[5], e[1]]
    T = 8
    p = {"q": np.array(qs)[:, None, :], "k": np.array(keys + [e[2]] * 4)[:, None, :],
         "v": np.concatenate([vals, np.zeros((4, V))])[:, None, :],
         "g": np.zeros((T, 1)), "beta": np.array([1.0] * 4 + [0.0] * 4)[:, None],
         "cu_seqlens": np.array([0, T]), "chunk_size": 4, "scale": 1.0}
    o = gdn_forward(p)["o"][:, 0]
    for t in range(4):
        np.testing.assert_allclose(o[t], vals[t], rtol=0, atol=1e-14)   # reads back the write
    np.testing.assert_allclose(o[4], vals[1], rtol=0, atol=1e-14)      # key 3 untouched
    np.testing.assert_allclose(o[5], vals[2], rtol=0, atol=1e-14)      # key 0 overwritten
    np.testing.assert_allclose(o[6], vals[3], rtol=0, atol=1e-14)
    np.testing.assert_allclose(o[7], np.zeros(V), rtol=0, atol=1e-14)  # never written


def _chunked_wy(q, k, v, g, beta, S0, scale, Q, s):
    """One request, one head, by chunks cut at absolute multiples of Q: per chunk
    with in-chunk log-gate prefix sums G, gamma = exp(G):
      (I + A) U = diag(beta) (V - diag(gamma) K S0),  A[a,r] = beta_a e^{G_a-G_r} k_a.k_r (r < a)
      O = scale (diag(gamma) Q S0 + tril(e^{G_t-G_s} Q K^T) U)
      S = gamma_last S0 + (diag(e^{G_last-G}) K)^T U."""
    L = len(q)
    S = S0.copy()
    o = np.zeros((L, v.shape[1]))
    pos = 0
    while pos < L:
        end = min(((s + pos) // Q + 1) * Q - s, L)
        Kc, Qc, Vc, bc = k[pos:end], q[pos:end], v[pos:end], beta[pos:end]
        G = np.cumsum(g[pos:end])
        gam = np.exp(G)
        n = end - pos
        A = np.tril(bc[:, None] * np.exp(G[:, None] - G[None, :]) * (Kc @ Kc.T), -1)
        U = np.linalg.solve(np.eye(n) + A, bc[:, None] * (Vc - gam[:, None] * (Kc @ S)))
        P = np.tril(np.exp(G[:, None] - G[None, :]) * (Qc @ Kc.T))
        o[pos:end] = scale * (gam[:, None] * (Qc @ S) + P @ U)
        S = gam[-1] * S + (Kc * np.exp(G[-1] - G)[:, None]).T @ U
        pos = end
    return o, S


@pytest.mark.parametrize("Q,l2norm", [(4, False), (8, True), (16, True)])
def test_matches_chunked_wy_form(Q, l2norm):
    rng = np.random.default_rng(Q)
    lengths = [23, 1, 9, 40]
    p = _prob(rng, lengths, Q=Q, l2norm=l2norm)
    p["num_computed"] = np.array([3, 0, 16, 5])
    out = gdn_forward(p)
    cu = p["cu_seqlens"]
    q, k = p["q"], p["k"]
    if l2norm:
        q = q / np.sqrt((q * q).sum(-1, keepdims=True) + 1e-6)
        k = k / np.sqrt((k * k).sum(-1, keepdims=True) + 1e-6)
    for i in range(len(lengths)):
        a, b = cu[i], cu[i + 1]
        for h in range(4):
            o, S = _chunked_wy(q[a:b, h // 2], k[a:b, h // 2], p["v"][a:b, h], p["g"][a:b, h], p["beta"][a:b, h],
                               p["state_pool"][p["init_slots"][i], h], 8 ** -0.5, Q, int(p["num_computed"][i]))
            np.testing.assert_allclose(out["o"][a:b, h], o, rtol=1e-10, atol=1e-11)
            np.testing.assert_allclose(out["final_states"][i, h], S, rtol=1e-10, atol=1e-11)


def test_chunk_export_is_the_state_after_each_chunk():
    rng = np.random.default_rng(7)
    p = _prob(rng, [11, 6], Q=4)
    p["num_computed"] = np.array([2, 0])
    out = gdn_forward(p)
    # request 0 covers absolute [2, 13): chunk ends after 2, 6, 10, 11 tokens
    for j, n in enumerate([2, 6, 10, 11]):
        cut = dict(p, q=p["q"][:n], k=p["k"][:n], v=p["v"][:n], g=p["g"][:n], beta=p["beta"][:n],
                   cu_seqlens=np.array([0, n]), num_computed=np.array([2]), init_slots=p["init_slots"][:1],
                   final_slots=None, export_chunks=False)
        np.testing.assert_allclose(out["chunk_states"][out["first_chunk"][0] + j],
                                   gdn_forward(cut)["final_states"][0], rtol=0, atol=1e-13)
    assert out["first_chunk"].tolist() == [0, 4, 6]


@pytest.mark.parametrize("cut", [1, 5, 8, 13])
def test_split_resume_equals_unsplit(cut):
    rng = np.random.default_rng(20 + cut)
    p = _prob(rng, [17])
    whole = gdn_forward(p)
    sl = lambda a, b: {key: p[key][a:b] for key in ("q", "k", "v", "g", "beta")}
    first = gdn_forward(dict(p, **sl(0, cut), cu_seqlens=np.array([0, cut])))
    pool = p["state_pool"].copy()
    pool[5] = first["final_states"][0]
    second = gdn_forward(dict(p, **sl(cut, 17), cu_seqlens=np.array([0, 17 - cut]),
                              num_computed=np.array([cut]), state_pool=pool, init_slots=np.array([5])))
    np.testing.assert_allclose(np.concatenate([first["o"], second["o"]]), whole["o"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(second["final_states"], whole["final_states"], rtol=1e-12, atol=1e-13)


def test_packing_equals_separate_runs():
    rng = np.random.default_rng(3)
    lengths = [4, 0, 9, 2]
    p = _prob(rng, lengths)
    out = gdn_forward(p)
    cu = p["cu_seqlens"]
    for i in range(4):
        one = gdn_forward(dict(p, **{key: p[key][cu[i]:cu[i + 1]] for key in ("q", "k", "v", "g", "beta")},
                               cu_seqlens=np.array([0, lengths[i]]), init_slots=p["init_slots"][i:i + 1],
                               final_slots=p["final_slots"][i:i + 1]))
        np.testing.assert_array_equal(out["o"][cu[i]:cu[i + 1]], one["o"])
        np.testing.assert_array_equal(out["final_states"][i], one["final_states"][0])
    # an empty request's final state is its initial state
    np.testing.assert_array_equal(out["final_states"][1], p["state_pool"][p["init_slots"][1]])


def test_l2norm_flag_equals_prenormalised_inputs():
    rng = np.random.default_rng(5)
    p = _prob(rng, [12, 7], l2norm=True)
    n = lambda a: a / np.sqrt((a * a).sum(-1, keepdims=True) + 1e-6)
    pre = dict(p, q=n(p["q"]), k=n(p["k"]), l2norm=False)
    a, b = gdn_forward(p), gdn_forward(pre)
    np.testing.assert_allclose(a["o"], b["o"], rtol=1e-13, atol=1e-14)


def test_shared_key_heads_equal_duplicated_keys():
    rng = np.random.default_rng(6)
    p = _prob(rng, [10, 3], Hk=2, Hv=4)
    dup = dict(p, q=np.repeat(p["q"], 2, axis=1), k=np.repeat(p["k"], 2, axis=1))
    a, b = gdn_forward(p), gdn_forward(dup)
    np.testing.assert_array_equal(a["o"], b["o"])
    np.testing.assert_array_equal(a["final_states"], b["final_states"])
