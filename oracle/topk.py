"""Exact top-k of index scores with the page-table emit, in fp64 (the step before sparse
attention: it produces the attention's index list).

TEST INFRASTRUCTURE ONLY (the oracle): the product path never imports this module.

Source: "FlashMLA 与 DSA：内核、流水线和正确性边界", section 5.5 (a query token's top-k over
its scores, emitted as physical cache ids ``page_table[u / 64] * 64 + u % 64``) and section
5.1's note that the output order is not part of the contract (set membership only); and
"sparse-attention co-design", section 5, step five (top-k over the causally visible
positions only; a row with fewer valid tokens than k is padded with an invalid id such as -1,
never with a repeated token).

This is the plain definition: a full sort of the valid prefix.  Ties at the threshold may be
broken any way (any k largest form a correct answer); ``check_row`` compares what is unique
(every score above the k-th largest value is selected) and checks the rest for validity.
"""

from __future__ import annotations

import numpy as np


def topk_positions(scores_row: np.ndarray, valid_len: int, k: int):
    """(positions of the k largest scores among the first valid_len, in descending order of
    score, threshold value or None).  Fewer than k valid positions: all of them."""
    n = max(0, min(int(valid_len), scores_row.shape[0]))
    vals = np.asarray(scores_row[:n], dtype=np.float64)
    order = np.argsort(-vals, kind="stable")  # a full sort; stable keeps ties in position order
    sel = order[: min(k, n)]
    thr = float(vals[sel[-1]]) if sel.size else None
    return sel, thr


def emit_ids(positions: np.ndarray, table_row: np.ndarray, page: int = 64) -> np.ndarray:
    """Physical cache ids of logical positions through one sequence's page table."""
    positions = np.asarray(positions, dtype=np.int64)
    return (np.asarray(table_row, dtype=np.int64)[positions // page] * page + positions % page)


def topk_page_table(scores: np.ndarray, valid_len, block_table: np.ndarray, s_q: int, k: int):
    """scores [n_tok, ld] (fp64 values), valid_len [n_tok], block_table [b, max_pages];
    token t belongs to request t // s_q.  Returns (ids int32 [n_tok, k] with the selected ids
    first and -1 after them, thresholds list (None for an empty row))."""
    n_tok = scores.shape[0]
    out = np.full((n_tok, k), -1, dtype=np.int32)
    thr = []
    for t in range(n_tok):
        sel, th = topk_positions(scores[t], int(valid_len[t]), k)
        out[t, : sel.size] = emit_ids(sel, block_table[t // s_q])
        thr.append(th)
    return out, thr


def check_row(got: np.ndarray, scores_row: np.ndarray, valid_len: int, k: int,
              table_row: np.ndarray, page: int = 64) -> None:
    """Assert that one output row is a correct top-k: the selected ids first, then -1; no
    duplicate; every position scoring above the k-th largest value is selected; every
    selected position is valid and scores at least that value."""
    n = max(0, min(int(valid_len), scores_row.shape[0]))
    m = min(k, n)
    got = np.asarray(got, dtype=np.int64)
    assert got.shape == (k,)
    assert np.all(got[m:] == -1), "entries after the selected ones must be -1"
    ids = got[:m]
    assert np.all(ids >= 0), "a selected entry is -1"
    assert np.unique(ids).size == m, "duplicate ids"
    # back from physical ids to logical positions through the inverse of the page table
    inv = {int(pg): j for j, pg in enumerate(np.asarray(table_row, dtype=np.int64))}
    pos = np.array([inv[int(i) // page] * page + int(i) % page for i in ids], dtype=np.int64)
    assert np.all(pos < n), "a selected position is outside the valid prefix"
    _, thr = topk_positions(scores_row, n, k)
    if m == 0:
        return
    vals = np.asarray(scores_row[:n], dtype=np.float64)
    assert np.all(vals[pos] >= thr), "a selected score is below the k-th largest value"
    above = np.nonzero(vals > thr)[0]
    assert np.isin(above, pos).all(), "a score above the k-th largest value was left out"


def check_row_within(got: np.ndarray, scores_row: np.ndarray, valid_len: int, k: int,
                     table_row: np.ndarray, tol: float, page: int = 64) -> None:
    """``check_row`` for scores known only to within ``tol`` (the selection was made on scores
    computed in lower precision): the selected ids first, then -1; no duplicate; every
    selected position valid and scoring at least the k-th largest value minus tol; every
    position scoring above the k-th largest value plus tol selected.  With tol = 0 this is
    ``check_row``."""
    n = max(0, min(int(valid_len), scores_row.shape[0]))
    m = min(k, n)
    got = np.asarray(got, dtype=np.int64)
    assert got.shape == (k,)
    assert np.all(got[m:] == -1), "entries after the selected ones must be -1"
    ids = got[:m]
    assert np.all(ids >= 0), "a selected entry is -1"
    assert np.unique(ids).size == m, "duplicate ids"
    inv = {int(pg): j for j, pg in enumerate(np.asarray(table_row, dtype=np.int64))}
    pos = np.array([inv[int(i) // page] * page + int(i) % page for i in ids], dtype=np.int64)
    assert np.all(pos < n), "a selected position is outside the valid prefix"
    if m == 0:
        return
    _, thr = topk_positions(scores_row, n, k)
    vals = np.asarray(scores_row[:n], dtype=np.float64)
    assert np.all(vals[pos] >= thr - tol), "a selected score is below the k-th largest value"
    above = np.nonzero(vals > thr + tol)[0]
    assert np.isin(above, pos).all(), "a score above the k-th largest value was left out"

