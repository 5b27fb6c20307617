"""Pins of the block-selection oracle (oracle/select.py), CPU only.

The oracle is checked against an independent statement of the same recipe
(the input-list construction of the long-context workload in workloads.py),
against scores derived by hand on a tiny paged cache, and against the list
rules (ties to the lower block index, block 0 and the last blocks always
kept, the order) on hand-made score vectors.
"""
import numpy as np
import pytest

import workloads as W
from oracle import select as S


def _bf16(x):
    return W.f32_to_bf16_bits(np.asarray(x, np.float32))


def test_matches_the_long_context_workload_recipe():
    w = W.config(5, small=True)
    res = S.select_blocks(w, 0.25, 8)
    for it, (lst, _) in res.items():
        b, g = divmod(it, w.num_kv_heads)
        row = w.visit_order[b, g]
        assert lst == [int(x) for x in row[row >= 0]], it


def test_hand_scores_on_a_tiny_paged_cache():
    # d = 4, two query heads per KV head, block_size 4, page_size 2, 5 blocks (19 tokens)
    B, Hq, Hkv, d, Ps, bs = 1, 2, 1, 4, 2, 4
    q = np.zeros((B, Hq, d), np.float32)
    q[0, 0] = [2, 0, 0, 0]
    q[0, 1] = [0, 4, 0, 0]          # qbar = [1, 2, 0, 0]
    N = 19
    npages = (N + Ps - 1) // Ps
    perm = np.array([7, 3, 9, 0, 5, 1, 8, 2, 6, 4])   # logical page -> physical page
    k = np.zeros((10, Hkv, Ps, d), np.float32)
    want = []
    for c in range(5):
        toks = range(4 * c, min(4 * c + 4, N))
        vals = []
        for j, t in enumerate(toks):
            row = np.array([c + j, -0.5 * c, 3.0, float(t % 3)], np.float32)  # exact in bf16
            k[perm[t // Ps], 0, t % Ps] = row
            vals.append(row)
        kbar = np.mean(vals, axis=0)
        want.append(float(kbar[0] * 1 + kbar[1] * 2))
    table = np.zeros((B, npages), np.int32)
    table[0] = perm[:npages]
    got = S.block_scores(_bf16(q), _bf16(k), table, N, 0, 0, num_q_heads=Hq, num_kv_heads=Hkv, page_size=Ps,
                         block_size=bs, dtype="bf16")
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
    # the last block has 3 tokens: its mean is over those three only
    assert abs(want[4] - (((4 + 5 + 6) / 3) - 2.0 * 2)) < 1e-12


@pytest.mark.parametrize("scores,frac,last,expect", [
    ([5, 1, 9, 9, 2, 7], 0.5, 0, [0, 5, 3, 2]),      # top 3 = {2, 3, 5} (9, 9, 7), plus block 0
    ([1, 1, 1, 1], 0.5, 0, [0, 1]),                 # all equal: lower indices first -> {0, 1}
    ([0, 3, 2, 1, 4], 0.0, 2, [0, 4, 3]),           # nothing by score: block 0 and the last two
    ([0, 3, 2, 1, 4], 1.0, 0, [0, 4, 3, 2, 1]),     # everything, most recent first
    ([-1, -2, -3], 0.34, 0, [0, 1]),                # ceil(0.34 * 3) = 2: blocks 0 and 1
    ([], 0.25, 8, []),
])
def test_list_rules(scores, frac, last, expect):
    assert S.kept_list(np.asarray(scores, np.float64), frac, last) == expect


@pytest.mark.parametrize("scores,frac,last,expect", [
    ([5, 1, 9, 9, 2, 7], 0.5, 0, [0, 2, 3, 5]),      # by score 9, 9 (lower index first), 7
    ([0, 3, 2, 1, 4], 0.0, 2, [0, 4, 3]),            # block 0 and the last two, by score 4 > 1
    ([0, 3, 2, 1, 4], 1.0, 0, [0, 4, 1, 2, 3]),      # everything by score
    ([7, 1, 1, 5], 0.25, 1, [0, 3]),                 # top block is 0 itself; last block 3
])
def test_importance_order(scores, frac, last, expect):
    assert S.kept_list(np.asarray(scores, np.float64), frac, last, order="importance") == expect
    # the same kept set as the recency order
    rec = S.kept_list(np.asarray(scores, np.float64), frac, last)
    assert sorted(rec) == sorted(expect)
