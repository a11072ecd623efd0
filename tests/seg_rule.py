"""The plan's work-segment rules, restated for the tests (host-side, plain Python).

A request at absolute positions [s, s + L) is cut into work segments, given as
their boundaries [s, c1, ..., e]:
  * multiples of `len` (batches averaging at most 1024 or more than 2048 tokens
    a request: len 2048 when the segment-state pre-pass is the two-head kernel --
    P = 64, N = 128, an even number of heads per group -- else 8192): cuts at the
    multiples of len strictly inside;
  * tail-shortened (batches averaging 1024-2048 tokens): the last segment starts
    at t1, the last multiple of 256 at least 129 tokens before the end, if
    t1 - s >= 256; the one before at t2 = t1 - 512, if t2 - s >= 512; the head
    before them is cut from its end backwards into n = ceil(length / 2048)
    segments of one stride (the smallest multiple of 256 not below length / n),
    the first taking the rest.
"""

PLAN_TAIL_SEGS = 1  # ssd_plan.flags bit


def cuts(s, L, length, tail):
    e = s + L
    if L <= 0:
        return [s, s]
    if not tail:
        n = (e - 1) // length - s // length + 1
        return [s] + [(s // length + k) * length for k in range(1, n)] + [e]
    head_end, tail_cuts = e, []
    if L >= 385:
        t1 = (e - 129) // 256 * 256
        if t1 - s >= 256:
            if t1 - 512 - s >= 512:
                tail_cuts, head_end = [t1 - 512, t1], t1 - 512
            else:
                tail_cuts, head_end = [t1], t1
    hlen = head_end - s
    n = -(-hlen // 2048)
    stride = (-(-hlen // n) + 255) // 256 * 256 if n > 1 else hlen
    return [s] + [head_end - stride * (n - k) for k in range(1, n)] + tail_cuts + [e]


def rule_of(T, R, P=64, N=128, H=2, G=1):
    """(len, tail) the plan picks for a batch of T tokens in R requests."""
    if 1024 * R < T <= 2048 * R:
        return 2048, True
    two_head_prepass = P == 64 and N == 128 and (H // G) % 2 == 0
    return (2048 if two_head_prepass else 8192), False
