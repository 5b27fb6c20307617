"""The unit path's stop rule against the one-pass rule (host-side model of the
decomposition; no GPU, no oracle).

The stability test of a block is the same on both paths: before the one-pass
stop, every block sees the same probe states. What the unit path changes is the
bookkeeping. Each unit of ck consecutive list positions names its first stop
position from its own stable bits, starting from the patience count entering
it. That count is taken from the previous unit's trailing run of stable blocks,
saturated at the patience. The item's stop is the smallest position named.
This module checks, by brute force over random stable-bit sequences, block-0
positions, unit lengths and patiences, that this equals the one-pass stop
(explainer sec. 2.3: `patience` consecutive stable blocks; sec. 2.4: never
before block 0). It also checks that the decomposition needs patience <= ck,
the condition the library requires.
"""
import math

import numpy as np
import pytest


def one_pass_stop(stable, patience, p0):
    """First list position where `patience` consecutive blocks were stable and
    block 0 (at list position p0, or absent when p0 < 0) has been processed;
    the last position otherwise."""
    n = len(stable)
    count = 0
    for i in range(n):
        count = count + 1 if stable[i] else 0
        seen0 = p0 < 0 or i >= p0
        if i == n - 1 or (stable[i] and count >= patience and seen0):
            return i
    raise AssertionError("unreachable")


def unit_stop(stable, patience, p0, ck):
    """The unit path's rule: per unit, the count entering it from the previous
    unit's trailing stable run (saturated at patience); the first position the
    unit names; the smallest over units."""
    n = len(stable)
    named = []
    for k in range(math.ceil(n / ck)):
        lo, hi = k * ck, min(n, (k + 1) * ck)
        count = 0
        if k > 0:
            run = 0
            for i in range(lo - 1, lo - ck - 1, -1):
                if not stable[i]:
                    break
                run += 1
            count = min(run, patience)
        for i in range(lo, hi):
            count = min(count + 1, patience) if stable[i] else 0
            seen0 = p0 < 0 or i >= p0
            if i == n - 1 or (stable[i] and count >= patience and seen0):
                named.append(i)
                break
    return min(named)


def _cases(seed, count):
    rng = np.random.default_rng(seed)
    for _ in range(count):
        n = int(rng.integers(1, 200))
        ck = int(rng.integers(8, 17))
        p_stable = float(rng.choice([0.3, 0.6, 0.85, 0.95]))
        stable = rng.random(n) < p_stable
        stable[0] = False  # the first block has no previous probe
        p0 = -1 if rng.random() < 0.3 else int(rng.integers(0, n))
        yield stable, ck, p0


@pytest.mark.parametrize("seed", range(6))
def test_unit_rule_equals_one_pass_rule(seed):
    for stable, ck, p0 in _cases(seed, 400):
        for patience in range(1, ck + 1):
            assert unit_stop(stable, patience, p0, ck) == one_pass_stop(stable, patience, p0), (ck, patience, p0)


def test_decomposition_needs_patience_at_most_the_unit_length():
    # every block from list position 1 on is stable; with patience 20 and units of 8
    # blocks the one-pass rule stops at position 20, inside the third unit. The count
    # entering that unit comes from the second unit alone (8, saturated at the
    # patience), not from the run that began in the first unit (15), so the unit rule
    # misses it and runs on to the list's end
    ck, patience = 8, 20
    stable = np.ones(40, bool)
    stable[0] = False
    assert one_pass_stop(stable, patience, -1) == 20
    assert unit_stop(stable, patience, -1, ck) == 39
    # with patience <= ck the same list decomposes correctly
    for p in range(1, ck + 1):
        assert unit_stop(stable, p, -1, ck) == one_pass_stop(stable, p, -1) == p
