"""Pins for the top-k oracle (no GPU): the full-sort definition against a textbook repeated
selection on tiny rows full of ties, the padding rules, the page-table emit against its
inverse, and the row checker against planted mistakes."""

import numpy as np
import pytest

from oracle import topk as otk


def _select_by_repeated_max(vals, k):
    """k rounds of 'take the largest remaining' (first position among equals)."""
    left = list(range(len(vals)))
    out = []
    for _ in range(min(k, len(vals))):
        best = max(left, key=lambda i: (vals[i], -i))
        out.append(best)
        left.remove(best)
    return out


@pytest.mark.parametrize("seed", range(6))
def test_full_sort_equals_repeated_selection(seed):
    rng = np.random.default_rng(seed)
    for _ in range(200):
        n = int(rng.integers(0, 14))
        vals = rng.choice([-2.0, -0.5, 0.0, 0.5, 1.0, 3.0], size=n)  # many ties
        k = int(rng.integers(1, 10))
        sel, thr = otk.topk_positions(vals, n, k)
        want = _select_by_repeated_max(list(vals), k)
        assert list(sel) == want
        if want:
            assert thr == vals[want[-1]]


def test_padding_and_prefix():
    table = np.array([[5, 2, 9, 0]])
    scores = np.arange(256, dtype=np.float64)[None, :]
    ids, thr = otk.topk_page_table(scores, [3], table, 1, 8)  # fewer valid than k
    assert list(ids[0, 3:]) == [-1] * 5 and thr[0] == 0.0
    assert sorted(ids[0, :3]) == [5 * 64 + 0, 5 * 64 + 1, 5 * 64 + 2]
    ids, thr = otk.topk_page_table(scores, [0], table, 1, 4)  # no valid token
    assert np.all(ids == -1) and thr == [None]
    ids, _ = otk.topk_page_table(scores, [200], table, 1, 4)  # the largest of the prefix only
    assert list(ids[0]) == [0 * 64 + 7, 0 * 64 + 6, 0 * 64 + 5, 0 * 64 + 4]  # page index 3


def test_emit_matches_inverse_table():
    rng = np.random.default_rng(3)
    table = rng.permutation(40)[:10]
    pos = rng.integers(0, 640, 300)
    ids = otk.emit_ids(pos, table)
    inv = {int(p): j for j, p in enumerate(table)}
    back = np.array([inv[int(i) // 64] * 64 + int(i) % 64 for i in ids])
    assert np.array_equal(back, pos)


def test_checker_rejects_planted_mistakes():
    rng = np.random.default_rng(4)
    n, k = 300, 32
    scores = np.round(rng.standard_normal(n) * 4) / 4  # ties
    table = rng.permutation(20)[:5]
    ids, _ = otk.topk_page_table(scores[None, :], [n], table[None, :], 1, k)
    good = ids[0].copy()
    otk.check_row(good, scores, n, k, table)
    rng.shuffle(good)  # any order of the selected ids is fine
    otk.check_row(good, scores, n, k, table)
    sel, thr = otk.topk_positions(scores, n, k)
    low = [u for u in range(n) if scores[u] < thr][0]
    bad_cases = []
    b = ids[0].copy(); b[0] = otk.emit_ids([low], table)[0]; bad_cases.append(b)   # a low score
    b = ids[0].copy(); b[1] = b[0]; bad_cases.append(b)                               # duplicate
    b = ids[0].copy(); b[2] = -1; bad_cases.append(b)                                 # hole
    short = ids[0].copy(); bad_cases.append(short[: k - 1])                           # wrong size
    for bad in bad_cases:
        with pytest.raises(AssertionError):
            otk.check_row(bad, scores, n, k, table)
    # a position beyond the valid prefix
    ids2, _ = otk.topk_page_table(scores[None, :], [100], table[None, :], 1, k)
    b = ids2[0].copy(); b[0] = otk.emit_ids([250], table)[0]
    with pytest.raises(AssertionError):
        otk.check_row(b, scores, 100, k, table)


def test_check_row_within_accepts_near_ties_and_rejects_planted_mistakes():
    rng = np.random.default_rng(11)
    n, k = 300, 40
    table = rng.permutation(20)[:5]
    vals = rng.standard_normal(n)
    order = np.argsort(-vals)
    thr = vals[order[k - 1]]
    tol = 1e-3
    vals[order[k]] = thr - tol / 2  # the (k+1)-th largest within tol of the k-th
    good = otk.emit_ids(order[:k], table)
    otk.check_row_within(np.asarray(good), vals, n, k, table, tol)
    # swapping the k-th for the near-tie is also a correct answer within tol
    swapped = otk.emit_ids(np.r_[order[: k - 1], order[k]], table)
    otk.check_row_within(np.asarray(swapped), vals, n, k, table, tol)
    with pytest.raises(AssertionError):  # ... but not at tol = 0
        otk.check_row_within(np.asarray(swapped), vals, n, k, table, 0.0)
    # a clearly lower score instead of a selected one
    low = otk.emit_ids(np.r_[order[: k - 1], order[-1]], table)
    with pytest.raises(AssertionError):
        otk.check_row_within(np.asarray(low), vals, n, k, table, tol)
    # a duplicate, a hole (-1 inside), a position past the prefix
    dup = np.asarray(good).copy(); dup[1] = dup[0]
    hole = np.asarray(good).copy(); hole[3] = -1
    with pytest.raises(AssertionError):
        otk.check_row_within(dup, vals, n, k, table, tol)
    with pytest.raises(AssertionError):
        otk.check_row_within(hole, vals, n, k, table, tol)
    with pytest.raises(AssertionError):
        otk.check_row_within(np.asarray(good), vals, 100, k, table, tol)
