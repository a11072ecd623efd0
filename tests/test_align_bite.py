"""Block-aligned prefill bites (ssd_varlen_align_bite) -- host only, CPU.

The rules of "Automatic prefix caching for GDN hybrid models
(mamba_cache_mode=all) with MTP speculative decoding" (engine core:
kernel-chunk-aligned prefill clipping and block-aligned split; review note:
re-align a misaligned start even in the final bite), as cases and as
properties of a scheduler loop driven by random budgets.
"""
import numpy as np
import pytest

import mamba2_ssd_varlen_gb300 as m


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mamba2_ssd_varlen_gb300 import build
    build.build()
    m.load_library()


@pytest.mark.parametrize("start,end,total,align,expect", [
    (0, 3000, 10000, 1024, 2048),       # aligned start: end clipped down to a boundary
    (0, 1024, 10000, 1024, 1024),       # already on a boundary
    (0, 500, 10000, 1024, 0),           # budget below one block: nothing this step
    (2048, 3000, 10000, 1024, 2048),    # ... from any aligned start
    (1000, 5000, 10000, 1024, 1024),    # misaligned start: re-aligned at the next boundary
    (1000, 1010, 10000, 1024, 1010),    # ... or earlier when the budget ends first
    (1000, 10000, 10000, 1024, 1024),   # the final bite from a misaligned start is re-aligned too
    (9300, 10000, 10000, 1024, 10000),  # no boundary left before the end: the tail as proposed
    (8192, 9999, 10000, 1024, 9999),    # aligned start, end past the last boundary: ends anywhere
    (2048, 9500, 10000, 1024, 9500),    # ... also when the bite crosses several boundaries
    (0, 7, 7, 16, 7),                   # a prompt shorter than one block: one bite
])
def test_cases(start, end, total, align, expect):
    assert m.ssd_varlen_align_bite(start, end, total, align) == expect


@pytest.mark.parametrize("args", [(0, 0, 10, 4), (5, 4, 10, 4), (0, 11, 10, 4), (-1, 3, 10, 4), (0, 3, 10, 0)])
def test_rejects_bad_arguments(args):
    with pytest.raises(m.SsdError):
        m.ssd_varlen_align_bite(*args)


@pytest.mark.parametrize("seed", range(6))
def test_scheduler_loop_properties(seed):
    # A scheduler loop under random budgets, from a random (possibly
    # misaligned) start: bites tile the rest of the prompt; a bite that ends
    # off the grid before the last boundary is a misaligned start's whole
    # budget short of the next boundary; once a bite ends on the grid every
    # later bite up to the last boundary starts on it.
    rng = np.random.default_rng(seed)
    for _ in range(200):
        align = int(rng.choice([16, 256, 1024]))
        total = int(rng.integers(1, 20 * align))
        start = int(rng.integers(0, total))
        last_aligned = total // align * align
        pos, bites, steps = start, [], 0
        while pos < total:
            steps += 1
            assert steps < 10000
            budget = int(rng.integers(1, 4 * align))
            proposed = min(total, pos + budget)
            end = m.ssd_varlen_align_bite(pos, proposed, total, align)
            assert pos <= end <= proposed
            if end == pos:   # below one block from an aligned start: wait
                assert pos % align == 0 and proposed < last_aligned and budget < align
                continue
            bites.append((pos, end, proposed))
            pos = end
        seen_aligned = False
        for a, b, proposed in bites:
            if seen_aligned and a <= last_aligned:
                assert a % align == 0
            if b % align:
                assert b > last_aligned or (a % align and b == proposed and b < (a // align + 1) * align)
            seen_aligned = seen_aligned or b % align == 0
