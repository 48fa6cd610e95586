"""Base-2 online softmax state, step by step, in fp64.

TEST INFRASTRUCTURE ONLY (the oracle): the product path never imports this module.

Source: "FlashMLA Sparse Decode 完整计算过程详解", step 9 (mask, row max, running max,
rescale factor, exponentials, running sum), step 11 (the second block's update), step
12 (final L and M) and step 14.2 (final lse = ln(L) + M / log2(e), or +inf when L = 0;
a split keeps log2(L) + M, or -inf when L = 0).  Scores arrive unscaled and are
multiplied by ``sm_scale * log2(e)`` inside the exponent (step 2.3 and step 9.4).

This restates the recurrence the decode kernel runs; ``tests/test_oracle.py`` pins it with
the page's printed numbers and checks that running it block by block reaches the
two-pass definition in ``sparse_mla_oracle.c``.
"""

from __future__ import annotations

import math

import numpy as np

LOG2E = 1.0 / math.log(2.0)


class State:
    """Running (M, L) of one query head in the base-2 domain; M starts at -inf."""

    def __init__(self) -> None:
        self.m = -math.inf
        self.l = 0.0

    def update(self, scores: np.ndarray, scale_log2: float, valid: np.ndarray | None = None):
        """Fold one block of raw scores; returns (p, scale_for_old).

        p[i] = 2^(score_i * scale_log2 - M_new) (0 for masked slots), and the caller
        rescales its running output by scale_for_old = 2^(M_old - M_new).
        """
        t = np.asarray(scores, dtype=np.float64) * scale_log2
        if valid is not None:
            t = np.where(valid, t, -math.inf)
        cur = float(np.max(t)) if t.size else -math.inf
        new = max(self.m, cur)
        if new == -math.inf:  # nothing valid yet: no contribution, nothing to rescale
            return np.zeros_like(t), 1.0
        scale_for_old = math.pow(2.0, self.m - new) if self.m != -math.inf else 0.0
        p = np.exp2(t - new)
        self.l = self.l * scale_for_old + float(np.sum(p))
        self.m = new
        return p, scale_for_old

    def lse(self) -> float:
        """Natural-log lse of an unsplit row: ln(L) + M / log2(e); +inf when L = 0."""
        return math.inf if self.l == 0.0 else math.log(self.l) + self.m / LOG2E

    def lse2(self) -> float:
        """Base-2 lse kept by a split: log2(L) + M; -inf when L = 0."""
        return -math.inf if self.l == 0.0 else math.log2(self.l) + self.m


def run(scores: np.ndarray, v: np.ndarray, scale_log2: float, block: int = 64,
        valid: np.ndarray | None = None):
    """Whole-row online softmax over blocks of ``block`` slots; returns (O, lse)."""
    st = State()
    acc = np.zeros(v.shape[1], dtype=np.float64)
    n = scores.shape[0]
    for lo in range(0, n, block):
        hi = min(n, lo + block)
        p, a = st.update(scores[lo:hi], scale_log2, None if valid is None else valid[lo:hi])
        acc = acc * a + p @ v[lo:hi]
    if st.l == 0.0:
        return np.zeros_like(acc), math.inf
    return acc / st.l, st.lse()
