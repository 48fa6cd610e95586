"""LSE-weighted merge of split-KV partial results, in fp64.

TEST INFRASTRUCTURE ONLY (the oracle): the product path never imports this module.

Source: "FlashMLA 与 DSA：内核、流水线和正确性边界", section 3.2 (the merge
``out = sum_j acc_j e^{m_j - m} / sum_j l_j e^{m_j - m}``), and "FlashMLA Sparse Decode
完整计算过程详解", step 14.2 (a split stores ``lse2 = log2(L) + M`` in base 2, or -inf when
L = 0) and step 16 (combine: M = max_j lse2_j, weights 2^(lse2_j - M), weighted mean of
the normalised partial outputs, final lse in natural log).

Reading (the pages are silent here): when every split has lse2 = -inf the merged output is 0 and the
merged lse is +inf, the same convention as an unsplit row with no valid slot.
"""

from __future__ import annotations

import math

import numpy as np


def combine(lse2: np.ndarray, o: np.ndarray, attn_sink=None) -> tuple[np.ndarray, float]:
    """Merge splits for one (token, head).

    lse2: [n_splits] base-2 log-sum-exp of each split (-inf for an empty split).
    o:    [n_splits, d_v] each split's output, already divided by its own exp-sum.
    attn_sink: optional sink value of this head: the merged output is then multiplied by
          1 / (1 + exp(attn_sink - lse)) with the merged lse ("FlashMLA 与 DSA", section
          4.3); the lse itself is returned unchanged.
    Returns (merged output [d_v], merged natural-log lse).
    """
    lse2 = np.asarray(lse2, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    m = float(np.max(lse2)) if lse2.size else -math.inf
    if m == -math.inf:
        return np.zeros(o.shape[-1], dtype=np.float64), math.inf
    w = np.exp2(lse2 - m)
    total = float(np.sum(w))
    merged = (w[:, None] * o).sum(axis=0) / total
    lse = (m + math.log2(total)) * math.log(2.0)
    if attn_sink is not None:
        with np.errstate(over="ignore"):
            merged = merged / (1.0 + np.exp(np.float64(attn_sink) - lse))
    return merged, lse


def weights(lse2: np.ndarray) -> np.ndarray:
    """Normalised merge weights 2^(lse2_j - M) / sum_k 2^(lse2_k - M)."""
    lse2 = np.asarray(lse2, dtype=np.float64)
    w = np.exp2(lse2 - np.max(lse2))
    return w / w.sum()
