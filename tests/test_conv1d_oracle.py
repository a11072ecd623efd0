"""Pins of the varlen causal conv1d oracle (oracle.conv1d) -- CPU.

Fixed against: numpy's own 1-D convolution per channel (an independent
formulation), a case worked by hand (including a request shorter than the conv
state), split-and-resume through the conv state, and packing invariance.
"""
import math

import numpy as np
import pytest

from oracle.conv1d import conv1d


def _prob(rng, lengths, D=6, W=4, silu=False, read=None, write=None):
    T = int(sum(lengths))
    R = len(lengths)
    S = 2 * R
    return {"x": rng.normal(size=(T, D)), "weight": rng.normal(size=(D, W)), "bias": rng.normal(size=D),
            "cu_seqlens": np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64),
            "conv_pool": rng.normal(size=(S, D, W - 1)),
            "read_slots": np.arange(R) if read is None else np.asarray(read),
            "write_slots": np.arange(R, 2 * R) if write is None else np.asarray(write), "silu": silu}


@pytest.mark.parametrize("W", [2, 3, 4])
def test_matches_numpy_convolve(W):
    rng = np.random.default_rng(W)
    p = _prob(rng, [7, 1, 3, 12], W=W)
    out = conv1d(p)
    cu = p["cu_seqlens"]
    for i in range(len(cu) - 1):
        a, b = cu[i], cu[i + 1]
        for c in range(p["x"].shape[1]):
            xin = np.concatenate([p["conv_pool"][p["read_slots"][i], c], p["x"][a:b, c]])
            ref = np.convolve(xin, p["weight"][c][::-1], mode="valid") + p["bias"][c]
            np.testing.assert_allclose(out["y"][a:b, c], ref, rtol=1e-13, atol=1e-13)


def test_worked_by_hand():
    # D = 1, W = 3, weight [1, 2, 3], bias 0.5.
    # Request 0 from state [10, 20], inputs [1, 2]:
    #   y0 = 10 + 40 + 3 + 0.5 = 53.5, y1 = 20 + 2 + 6 + 0.5 = 28.5, state out [1, 2]
    # Request 1 from zeros (read slot -1), one input [5] (shorter than the state):
    #   y = 3 * 5 + 0.5 = 15.5, state out [0, 5]; with SiLU y = 15.5 sigma(15.5)
    p = {"x": np.array([[1.0], [2.0], [5.0]]), "weight": np.array([[1.0, 2.0, 3.0]]), "bias": np.array([0.5]),
         "cu_seqlens": np.array([0, 2, 3]), "conv_pool": np.array([[[10.0, 20.0]], [[0.0, 0.0]], [[0.0, 0.0]]]),
         "read_slots": np.array([0, -1]), "write_slots": np.array([1, 2]), "silu": False}
    out = conv1d(p)
    np.testing.assert_array_equal(out["y"][:, 0], [53.5, 28.5, 15.5])
    np.testing.assert_array_equal(out["writes"][1], [[1.0, 2.0]])
    np.testing.assert_array_equal(out["writes"][2], [[0.0, 5.0]])
    p["silu"] = True
    y = conv1d(p)["y"][:, 0]
    assert abs(y[2] - 15.5 / (1 + math.exp(-15.5))) < 1e-13


@pytest.mark.parametrize("k", [1, 2, 5, 9])
def test_split_resume_equals_unsplit(k):
    rng = np.random.default_rng(10 + k)
    full = _prob(rng, [10], read=[0], write=[1])
    out = conv1d(full)
    first = dict(full, x=full["x"][:k], cu_seqlens=np.array([0, k]))
    o1 = conv1d(first)
    pool2 = full["conv_pool"].copy()
    pool2[0] = o1["final"][0]
    second = dict(full, x=full["x"][k:], cu_seqlens=np.array([0, 10 - k]), conv_pool=pool2)
    o2 = conv1d(second)
    np.testing.assert_allclose(np.concatenate([o1["y"], o2["y"]]), out["y"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(o2["final"][0], out["final"][0], rtol=0, atol=0)


def test_packing_equals_separate_runs():
    rng = np.random.default_rng(3)
    p = _prob(rng, [4, 0, 6, 2], silu=True)
    out = conv1d(p)
    cu = p["cu_seqlens"]
    for i in range(4):
        one = dict(p, x=p["x"][cu[i]:cu[i + 1]], cu_seqlens=np.array([0, cu[i + 1] - cu[i]]),
                   read_slots=p["read_slots"][i:i + 1], write_slots=p["write_slots"][i:i + 1])
        o = conv1d(one)
        np.testing.assert_allclose(out["y"][cu[i]:cu[i + 1]], o["y"], rtol=0, atol=0)
        np.testing.assert_array_equal(out["final"][i], o["final"][0])
    # an empty request passes its state through
    np.testing.assert_array_equal(out["final"][1], p["conv_pool"][p["read_slots"][1]])
