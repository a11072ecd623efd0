"""Pins the CPU oracle to facts other than itself (CPU only, no GPU).

Each test names what fixes the expected value: the materialised quadratic SSD
form (tests/brute_force.py, independent code), closed forms (A = 0 is a plain
cumulative sum, B = 0 is pure decay of the initial state, one token worked by
hand), and the invariances the SSD varlen pages rely on (packing requests
with cu_seqlens equals running them apart; resuming from a final state equals
the unsplit run).  A plausible slip in the oracle -- a dropped term, a sign,
an index, a transposed outer product, a missing reset between requests --
fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import checkpoints
from brute_force import quadratic_one, softplus

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_problem(rng, lengths, H=4, P=5, N=7, G=2, with_D=True, with_z=True, with_h0=True,
                  A_zero=False, B_zero=False):
    T = int(sum(lengths))
    R = len(lengths)
    cu = np.zeros(R + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lengths)
    p = {
        "cu": cu,
        "x": rng.standard_normal((T, H, P)),
        "dt": rng.standard_normal((T, H)),
        "dt_bias": rng.uniform(-2, -1, H),
        "A": np.zeros(H) if A_zero else -np.exp(rng.uniform(0, math.log(16), H)),
        "B": np.zeros((T, G, N)) if B_zero else rng.standard_normal((T, G, N)),
        "C": rng.standard_normal((T, G, N)),
        "D": rng.standard_normal(H) if with_D else None,
        "z": rng.standard_normal((T, H, P)) if with_z else None,
        "h0": rng.standard_normal((R, H, P, N)) if with_h0 else None,
    }
    return p


def _run(p, rec_k=None):
    return oracle.recurrence(p["cu"], p["x"], p["dt"], p["dt_bias"], p["A"], p["B"], p["C"],
                             p["D"], p["z"], p["h0"], rec_k=rec_k, n_threads=2)


def _one(p, i, h):
    """Slice (request i, head h) for the brute-force forms."""
    a, b = int(p["cu"][i]), int(p["cu"][i + 1])
    H = p["x"].shape[1]
    G = p["B"].shape[1]
    g = h // (H // G)
    return dict(x=p["x"][a:b, h], dt=p["dt"][a:b, h], dt_bias=p["dt_bias"][h], A=p["A"][h],
                B=p["B"][a:b, g], C=p["C"][a:b, g],
                D=None if p["D"] is None else p["D"][h],
                z=None if p["z"] is None else p["z"][a:b, h],
                h0=None if p["h0"] is None else p["h0"][i, h])


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_brute_force_quadratic_form(seed):
    rng = np.random.default_rng(seed)
    p = _rand_problem(rng, [5, 17, 42, 1, 0, 9])
    y, hf, _ = _run(p)
    R, H = len(p["cu"]) - 1, p["x"].shape[1]
    for i in range(R):
        a, b = int(p["cu"][i]), int(p["cu"][i + 1])
        for h in range(H):
            yq, hq = quadratic_one(**_one(p, i, h))
            np.testing.assert_allclose(y[a:b, h], yq, rtol=1e-11, atol=1e-11)
            np.testing.assert_allclose(hf[i, h], hq, rtol=1e-11, atol=1e-11)


def test_A_zero_is_a_plain_cumulative_sum():
    rng = np.random.default_rng(3)
    p = _rand_problem(rng, [11, 6], A_zero=True, with_z=False)
    y, hf, _ = _run(p)
    H, P, N = p["x"].shape[1], p["x"].shape[2], p["B"].shape[2]
    G = p["B"].shape[1]
    for i in range(2):
        a, b = int(p["cu"][i]), int(p["cu"][i + 1])
        for h in range(H):
            g = h // (H // G)
            dtp = softplus(p["dt"][a:b, h] + p["dt_bias"][h])
            terms = np.stack([dtp[t] * np.outer(p["x"][a + t, h], p["B"][a + t, g])
                              for t in range(b - a)])
            states = p["h0"][i, h][None] + np.cumsum(terms, axis=0)
            y_ref = np.einsum("tpn,tn->tp", states, p["C"][a:b, g]) + p["D"][h] * p["x"][a:b, h]
            np.testing.assert_allclose(y[a:b, h], y_ref, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(hf[i, h], states[-1], rtol=1e-12, atol=1e-12)


def test_B_zero_is_pure_decay_of_the_initial_state():
    rng = np.random.default_rng(4)
    p = _rand_problem(rng, [13, 4], B_zero=True)
    y, hf, _ = _run(p)
    H, G = p["x"].shape[1], p["B"].shape[1]
    for i in range(2):
        a, b = int(p["cu"][i]), int(p["cu"][i + 1])
        for h in range(H):
            g = h // (H // G)
            cs = np.cumsum(softplus(p["dt"][a:b, h] + p["dt_bias"][h]) * p["A"][h])
            inter = np.exp(cs)[:, None] * (p["C"][a:b, g] @ p["h0"][i, h].T)
            gate = p["z"][a:b, h] / (1 + np.exp(-p["z"][a:b, h]))
            y_ref = (inter + p["D"][h] * p["x"][a:b, h]) * gate
            np.testing.assert_allclose(y[a:b, h], y_ref, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(hf[i, h], math.exp(cs[-1]) * p["h0"][i, h], rtol=1e-12)


def test_one_token_worked_by_hand():
    # dt + dt_bias = 0 gives dt' = ln 2; A = -1 then gives decay exp(-ln 2) = 1/2.
    # P = 2, N = 3, one head, one group.
    x = np.array([[[1.0, -2.0]]])
    dt = np.array([[0.5]])
    dt_bias = np.array([-0.5])
    A = np.array([-1.0])
    B = np.array([[[2.0, 0.0, -1.0]]])
    C = np.array([[[3.0, 1.0, 4.0]]])
    D = np.array([0.25])
    h0 = np.array([[[[1.0, 2.0, 3.0], [0.0, -1.0, 0.5]]]])
    y, hf, _ = oracle.recurrence([0, 1], x, dt, dt_bias, A, B, C, D, None, h0)
    ln2 = math.log(2.0)
    # state = h0/2 + ln2 * x (outer) B
    s = [[0.5 + 2 * ln2, 1.0, 1.5 - ln2], [0.0 - 4 * ln2, -0.5, 0.25 + 2 * ln2]]
    np.testing.assert_allclose(hf[0, 0], s, rtol=1e-15, atol=1e-15)
    y0 = 3 * s[0][0] + 1 * s[0][1] + 4 * s[0][2] + 0.25 * 1.0
    y1 = 3 * s[1][0] + 1 * s[1][1] + 4 * s[1][2] + 0.25 * -2.0
    np.testing.assert_allclose(y[0, 0], [y0, y1], rtol=1e-14)
    # by hand: y0 = 1.5 + 6 ln2 + 1 + 6 - 4 ln2 + 0.25 = 8.75 + 2 ln2
    assert abs(y[0, 0, 0] - (8.75 + 2 * ln2)) < 1e-13
    # y1 = -12 ln2 - 0.5 + 1 + 8 ln2 - 0.5 = -4 ln2
    assert abs(y[0, 0, 1] - (-4 * ln2)) < 1e-13


def test_two_tokens_worked_by_hand_with_gate():
    # P = N = 1.  dt' = ln 2 both steps, A = -1 so each step halves the state.
    # t1: h = ln2 * x1 * B1 = ln2 * 1 * 2 = 2 ln2;       y1 = h * C1 = 6 ln2
    # t2: h = 2 ln2 / 2 + ln2 * x2 * B2 = ln2 + ln2 * 3 * (-1) = -2 ln2
    #     y2 = (h * C2 + D x2) * silu(z2) = (-2 ln2 * 5 + 0.5 * 3) * silu(z2)
    x = np.array([[[1.0]], [[3.0]]])
    dt = np.zeros((2, 1))
    B = np.array([[[2.0]], [[-1.0]]])
    C = np.array([[[3.0]], [[5.0]]])
    z = np.array([[[0.0]], [[1.5]]])
    y, hf, _ = oracle.recurrence([0, 2], x, dt, np.array([0.0]), np.array([-1.0]), B, C,
                                 np.array([0.5]), z, None)
    ln2 = math.log(2.0)
    silu = lambda v: v / (1 + math.exp(-v))
    assert abs(y[0, 0, 0] - 6 * ln2 * silu(0.0)) < 1e-14      # silu(0) = 0
    assert abs(y[1, 0, 0] - (-10 * ln2 + 1.5) * silu(1.5)) < 1e-13
    assert abs(hf[0, 0, 0, 0] - (-2 * ln2)) < 1e-14


def test_softplus_threshold_reading():
    # Above 20 the reading takes softplus(v) = v; at 19 it is log1p(exp(19)).
    for v, expect in ((25.0, 25.0), (19.0, math.log1p(math.exp(19.0))), (-30.0, math.log1p(math.exp(-30.0)))):
        x = np.ones((1, 1, 1))
        B = np.ones((1, 1, 1))
        _, hf, _ = oracle.recurrence([0, 1], x, np.array([[v]]), np.array([0.0]), np.array([0.0]),
                                     B, B, None, None, None)
        assert hf[0, 0, 0, 0] == pytest.approx(expect, rel=1e-15, abs=0)


def test_packing_equals_separate_runs():
    rng = np.random.default_rng(5)
    lengths = [7, 0, 19, 3]
    p = _rand_problem(rng, lengths)
    y, hf, _ = _run(p)
    for i, L in enumerate(lengths):
        a, b = int(p["cu"][i]), int(p["cu"][i + 1])
        q = dict(p)
        q["cu"] = np.array([0, L])
        for k in ("x", "dt", "B", "C", "z"):
            q[k] = p[k][a:b]
        q["h0"] = p["h0"][i:i + 1]
        ys, hs, _ = _run(q)
        np.testing.assert_array_equal(ys, y[a:b])
        np.testing.assert_array_equal(hs[0], hf[i])


@pytest.mark.parametrize("k", [1, 5, 16, 17, 40])
def test_split_state_resume_equals_unsplit(k):
    rng = np.random.default_rng(6)
    L = 41
    p = _rand_problem(rng, [L])
    y, hf, rec = _run(p, rec_k=[[k]])
    pre = dict(p)
    pre["cu"] = np.array([0, k])
    for key in ("x", "dt", "B", "C", "z"):
        pre[key] = p[key][:k]
    y1, h1, _ = _run(pre)
    post = dict(p)
    post["cu"] = np.array([0, L - k])
    for key in ("x", "dt", "B", "C", "z"):
        post[key] = p[key][k:]
    post["h0"] = h1
    y2, h2, _ = _run(post)
    np.testing.assert_allclose(np.concatenate([y1, y2]), y, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(h2, hf, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(rec[0], h1[0], rtol=0, atol=0)


def test_group_map_is_contiguous():
    # With G = 2 and H = 4, heads 0-1 read group 0 and heads 2-3 read group 1:
    # zeroing group 1's B and C must leave heads 0-1 unchanged and make heads
    # 2-3 carry only D x (no initial state).
    rng = np.random.default_rng(7)
    p = _rand_problem(rng, [9], with_h0=False, with_z=False)
    y, _, _ = _run(p)
    q = dict(p)
    q["B"] = p["B"].copy()
    q["C"] = p["C"].copy()
    q["B"][:, 1] = 0.0
    q["C"][:, 1] = 0.0
    y2, _, _ = _run(q)
    np.testing.assert_array_equal(y2[:, :2], y[:, :2])
    np.testing.assert_allclose(y2[:, 2:], p["D"][2:, None] * p["x"][:, 2:], rtol=1e-15)


def test_chunk_ends_golden():
    g = json.load(open(os.path.join(GOLDEN, "checkpoint_map.json")))
    for c in g["chunk_cases"]:
        assert checkpoints.request_chunk_ends(c["L"], c["s"], c["Q"]) == c["chunk_ends"], c["why"]
    for c in g["block_cases"]:
        got = checkpoints.request_block_boundaries(c["L"], c["s"], c["bs"])
        assert [list(v) for v in got] == c["blocks"], c["why"]


def test_checkpoint_records_golden():
    g = json.load(open(os.path.join(GOLDEN, "checkpoint_map.json")))
    for c in g["record_cases"]:
        recs, first = checkpoints.checkpoint_records(
            c["lengths"], c["num_computed"], c["Q"], c["block_size"], c["block_table"],
            c["export_chunks"])
        assert first == c["first_chunk"], c["why"]
        got = sorted((r.request, r.k, r.kind, r.dest) for r in recs)
        assert got == sorted(tuple(v) for v in c["records"]), c["why"]


def test_forward_pool_semantics_against_truncated_runs():
    """Every pool write and export row equals the state of a run truncated at
    that token, which pins the record positions independently of the record
    bookkeeping; untouched slots keep their canary value."""
    rng = np.random.default_rng(8)
    lengths = [10, 0, 6]
    ncomp = [3, 5, 0]
    H, P, N, G = 2, 3, 4, 1
    p = _rand_problem(rng, lengths, H=H, P=P, N=N, G=G, with_h0=False)
    S = 32
    pool = np.full((S, H, P, N), 7.0)
    pool[1] = rng.standard_normal((H, P, N))
    pool[2] = rng.standard_normal((H, P, N))
    prob = {"x": p["x"], "dt": p["dt"], "dt_bias": p["dt_bias"], "A": p["A"], "B": p["B"],
            "C": p["C"], "D": p["D"], "z": p["z"], "cu_seqlens": p["cu"], "num_computed": ncomp,
            "chunk_size": 4, "block_size": 4, "state_pool": pool,
            "init_slots": [1, 2, -1], "final_slots": [30, 29, 28],
            "block_table": [[-1, 11, 12, -1], [-1, -1, -1, -1], [21, 22, -1, -1]],
            "export_chunks": True}
    out = oracle.forward(prob, n_threads=2)

    def truncated(i, k):
        a = int(p["cu"][i])
        h0 = np.zeros((1, H, P, N)) if prob["init_slots"][i] < 0 else pool[prob["init_slots"][i]][None]
        _, hf, _ = oracle.recurrence([0, k], p["x"][a:a + k], p["dt"][a:a + k], p["dt_bias"],
                                     p["A"], p["B"][a:a + k], p["C"][a:a + k], p["D"],
                                     p["z"][a:a + k], h0)
        return hf[0]

    newp = out["state_pool"]
    np.testing.assert_allclose(newp[11], truncated(0, 5), rtol=1e-14)
    np.testing.assert_allclose(newp[12], truncated(0, 9), rtol=1e-14)
    np.testing.assert_allclose(newp[21], truncated(2, 4), rtol=1e-14)
    np.testing.assert_allclose(newp[30], truncated(0, 10), rtol=1e-14)
    np.testing.assert_allclose(newp[29], pool[2], rtol=0)        # empty request: final = initial
    np.testing.assert_allclose(newp[28], truncated(2, 6), rtol=1e-14)
    for j, (i, k) in enumerate([(0, 1), (0, 5), (0, 9), (0, 10), (2, 4), (2, 6)]):
        np.testing.assert_allclose(out["chunk_states"][j], truncated(i, k), rtol=1e-14)
    touched = {1, 2, 11, 12, 21, 28, 29, 30}
    for s in range(S):
        if s not in touched:
            assert np.all(newp[s] == 7.0)
    np.testing.assert_array_equal(newp[1], pool[1])


def test_tiny_config_matches_brute_force():
    """The tiny fp32 workload end to end through the forward wrapper."""
    import workloads
    prob = workloads.make_problem("tiny_fp32")
    o = workloads.to_oracle(prob)
    out = oracle.forward(o, n_threads=2)
    cu = o["cu_seqlens"]
    H = o["x"].shape[1]
    for i in range(3):
        a, b = int(cu[i]), int(cu[i + 1])
        s = int(o["init_slots"][i])
        for h in range(H):
            h0 = o["state_pool"][s][h] if s >= 0 else None
            yq, hq = quadratic_one(o["x"][a:b, h], o["dt"][a:b, h], o["dt_bias"][h], o["A"][h],
                                   o["B"][a:b, 0], o["C"][a:b, 0], o["D"][h], None, h0)
            np.testing.assert_allclose(out["y"][a:b, h], yq, rtol=1e-10, atol=1e-10)
            np.testing.assert_allclose(out["final_states"][i, h], hq, rtol=1e-10, atol=1e-10)
