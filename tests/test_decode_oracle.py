"""Pins of the decode-step oracle (oracle.decode) -- CPU.

The decode step ("Automatic prefix caching for GDN hybrid models
(mamba_cache_mode=all) with MTP speculative decoding", Purpose, Kernels/layers:
dual read/write state anchors in the decode kernels) is the recurrence over a
short window per request, starting from a read-anchor slot and writing the state
after chosen tokens to write-anchor slots.  The recurrence itself is pinned in
test_oracle_pins.py; these pins fix the anchor bookkeeping: worked by hand, and
against independent runs of the recurrence on truncated windows.
"""
import math

import numpy as np
import pytest

import oracle

silu = lambda v: v / (1 + math.exp(-v))  # noqa: E731
LN2 = math.log(2.0)


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def test_decode_window_worked_by_hand():
    # P = N = 1, dt' = ln 2 (dt + dt_bias = 0) so exp(dt' A) = 1/2 with A = -1.
    # Request 0: window of 2 tokens from read slot 1 (h = 4), writing slots 2, 3.
    #   t0: h = 4/2 + ln2 * 1 * 2 = 2 + 2 ln2;   y0 = (3 h + 0.5 * 1) * silu(0) = 0
    #   t1: h = (2 + 2 ln2)/2 + ln2 * 3 * (-1) = 1 - 2 ln2
    #       y1 = (5 h + 0.5 * 3) * silu(1.5)
    # Request 1: one token from zeros (read slot -1), no write:
    #   h = ln2 * 2 * 1 = 2 ln2;  y = (1 * h + 0.5 * 2) * silu(2)
    prob = {
        "cu_seqlens": np.array([0, 2, 3]),
        "x": np.array([[[1.0]], [[3.0]], [[2.0]]]),
        "dt": np.zeros((3, 1)),
        "dt_bias": np.array([0.0]),
        "A": np.array([-1.0]),
        "B": np.array([[[2.0]], [[-1.0]], [[1.0]]]),
        "C": np.array([[[3.0]], [[5.0]], [[1.0]]]),
        "D": np.array([0.5]),
        "z": np.array([[[0.0]], [[1.5]], [[2.0]]]),
        "state_pool": np.array([[[[7.0]]], [[[4.0]]], [[[0.0]]], [[[0.0]]]]),
        "read_slots": np.array([1, -1]),
        "write_slots": np.array([2, 3, -1]),
    }
    out = oracle.decode(prob)
    y = out["y"][:, 0, 0]
    assert abs(y[0]) < 1e-15
    assert abs(y[1] - (5 * (1 - 2 * LN2) + 1.5) * silu(1.5)) < 1e-13
    assert abs(y[2] - (2 * LN2 + 1.0) * silu(2.0)) < 1e-13
    assert sorted(out["writes"]) == [2, 3]
    assert abs(out["writes"][2][0, 0, 0] - (2 + 2 * LN2)) < 1e-14
    assert abs(out["writes"][3][0, 0, 0] - (1 - 2 * LN2)) < 1e-14


def _random_step(rng, windows, H=3, P=4, N=5, G=1):
    T = int(sum(windows))
    cu = np.concatenate([[0], np.cumsum(windows)]).astype(np.int64)
    R = len(windows)
    S = R + T
    pool = rng.normal(size=(S, H, P, N))
    perm = rng.permutation(S)
    read = perm[:R].copy()
    read[1] = -1
    write = np.full(T, -1)
    k = R
    for t in range(T):
        if rng.random() < 0.7:
            write[t] = perm[k]
            k += 1
    return {"cu_seqlens": cu, "x": rng.normal(size=(T, H, P)), "dt": rng.normal(size=(T, H)),
            "dt_bias": rng.uniform(-2, -1, size=H), "A": -np.exp(rng.uniform(0, np.log(16), size=H)),
            "B": rng.normal(size=(T, G, N)), "C": rng.normal(size=(T, G, N)), "D": rng.normal(size=H),
            "z": rng.normal(size=(T, H, P)), "state_pool": pool, "read_slots": read, "write_slots": write}


@pytest.mark.parametrize("seed", [0, 1])
def test_decode_equals_truncated_runs(seed):
    # Every written state equals the final state of a separate run of the window
    # truncated after that token, from the read anchor; y equals the full run.
    rng = np.random.default_rng(seed)
    windows = [1, 4, 3, 0, 2]
    prob = _random_step(rng, windows)
    out = oracle.decode(prob)
    cu = prob["cu_seqlens"]
    pool = prob["state_pool"]
    n_written = 0
    for i in range(len(windows)):
        a, b = int(cu[i]), int(cu[i + 1])
        s = int(prob["read_slots"][i])
        h0 = (pool[s] if s >= 0 else np.zeros_like(pool[0]))[None]
        for t in range(a, b):
            sl = slice(a, t + 1)
            y_t, hf, _ = oracle.recurrence([0, t + 1 - a], prob["x"][sl], prob["dt"][sl], prob["dt_bias"],
                                           prob["A"], prob["B"][sl], prob["C"][sl], prob["D"], prob["z"][sl], h0)
            np.testing.assert_allclose(out["y"][t], y_t[-1], rtol=0, atol=1e-12)
            w = int(prob["write_slots"][t])
            if w >= 0:
                np.testing.assert_allclose(out["writes"][w], hf[0], rtol=0, atol=1e-12)
                n_written += 1
    assert n_written == len(out["writes"]) == int((prob["write_slots"] >= 0).sum())


def test_empty_window_and_zero_anchor():
    rng = np.random.default_rng(3)
    prob = _random_step(rng, [0, 1, 0])
    prob["read_slots"] = np.array([0, -1, 1])
    prob["write_slots"] = np.array([3])
    out = oracle.decode(prob)
    assert list(out["writes"]) == [3]
    # the only token starts from zeros: its state is dt' x (outer) B
    dtp = np.log1p(np.exp(prob["dt"][0] + prob["dt_bias"]))
    h = dtp[:, None, None] * prob["x"][0][:, :, None] * prob["B"][0, 0][None, None, :]
    for w, v in out["writes"].items():
        np.testing.assert_allclose(v, h, rtol=1e-14, atol=1e-14)
