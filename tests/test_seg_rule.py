"""The work-segment rules the plan applies (restated in seg_rule.py): hand-worked
cases and the properties the kernels rely on -- every inner cut a multiple of
256 (so pieces and chunks of up to 256 tokens never straddle a segment
boundary), every segment 1-2048 tokens (the segment-state pre-pass's limit),
and the workspace bound on segments that are not the last of their request."""
import numpy as np
import pytest

import seg_rule


def lengths(c):
    return [b - a for a, b in zip(c[:-1], c[1:])]


def test_hand_worked_tail_shortened_cases():
    # a 2048-token request: head 1280, then 512, then the last 256
    assert seg_rule.cuts(0, 2048, 2048, True) == [0, 1280, 1792, 2048]
    # resumed at 5: the last cut stays at least 129 tokens before the end
    assert seg_rule.cuts(5, 2048, 2048, True) == [5, 1280, 1792, 2053]
    # 1100 tokens: a head of 256 would be too short to cut off, one tail cut only
    assert seg_rule.cuts(0, 1100, 2048, True) == [0, 768, 1100]
    # short requests stay whole
    assert seg_rule.cuts(0, 300, 2048, True) == [0, 300]
    assert seg_rule.cuts(77, 1, 2048, True) == [77, 78]
    # a long head is cut backwards into equal 256-multiples of at most 2048
    assert seg_rule.cuts(0, 5000, 2048, True) == [0, 1280, 2816, 4352, 4864, 5000]


def test_multiples_rule_cases():
    assert seg_rule.cuts(0, 2048, 1024, False) == [0, 1024, 2048]
    assert seg_rule.cuts(1000, 100, 1024, False) == [1000, 1024, 1100]
    assert seg_rule.cuts(3, 4096, 2048, False) == [3, 2048, 4096, 4099]


def test_rule_follows_the_average_request_length():
    assert seg_rule.rule_of(8 * 1024, 8) == (2048, False)
    assert seg_rule.rule_of(8 * 1024 + 1, 8) == (2048, True)
    assert seg_rule.rule_of(8 * 2048, 8) == (2048, True)
    assert seg_rule.rule_of(8 * 2048 + 1, 8) == (2048, False)
    # the one-head path (P = 128, or an odd number of heads per group) has no
    # 2048-token pre-pass limit
    assert seg_rule.rule_of(8 * 4000, 8, P=128) == (8192, False)
    assert seg_rule.rule_of(8 * 4000, 8, P=64, H=6, G=2) == (8192, False)
    assert seg_rule.rule_of(8 * 1500, 8, P=128) == (2048, True)


@pytest.mark.parametrize("tail", [True, False])
def test_properties_over_random_requests(tail):
    rng = np.random.default_rng(7 if tail else 8)
    length = 2048
    for _ in range(20000):
        s = int(rng.integers(0, 6000))
        L = int(rng.integers(1, 20000)) if rng.random() < 0.5 else int(rng.integers(1, 3000))
        c = seg_rule.cuts(s, L, length, tail)
        assert c[0] == s and c[-1] == s + L
        lens = lengths(c)
        assert all(1 <= x <= 2048 for x in lens), (s, L, c)
        assert all(x % 256 == 0 for x in c[1:-1]), (s, L, c)
        if tail:
            assert len(c) - 1 <= -(-L // 2048) + 2, (s, L, c)
            if len(c) > 2:
                assert 129 <= lens[-1] <= 384, (s, L, c)
        else:
            assert all(x % length == 0 for x in c[1:-1])


@pytest.mark.parametrize("tail", [True, False])
def test_workspace_bound_on_non_final_segments(tail):
    # ssd_api.cu sizes the chained states for at most floor((T + 4095 R) / 2048)
    # non-final segments (tail-shortened) or floor((T + R (len - 2)) / len).
    rng = np.random.default_rng(11 if tail else 12)
    for _ in range(3000):
        R = int(rng.integers(1, 40))
        L = rng.integers(1, 5000, R)
        s = rng.integers(0, 3000, R)
        T = int(L.sum())
        length = 2048
        nonfinal = sum(len(seg_rule.cuts(int(a), int(b), length, tail)) - 2 for a, b in zip(s, L))
        bound = (T + 4095 * R) // 2048 if tail else (T + R * (length - 2)) // length
        assert nonfinal <= min(bound, T - 1)
