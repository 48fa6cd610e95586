"""Decode variants on top of the sparse attention definition: per-token top-k length and
attention sink, in fp64.

TEST INFRASTRUCTURE ONLY (the oracle): the product path never imports this module.

Source: "FlashMLA 与 DSA：内核、流水线和正确性边界", section 4.3 (the reference
semantics: a slot is invalid when its index is -1 or when its position in the token's
top-k list is at or beyond that token's ``topk_length``; with an attention sink the output
is multiplied by ``1 / (1 + exp(attn_sink - lse))``, lse being the log-sum-exp of the real
scores), and "FlashMLA Sparse Decode 完整计算过程详解", step 13 (the same factor folded
into the kernel's output scale for an unsplit row, in the base-2 domain:
``o_scale = 1 / (L + 2^(attn_sink * log2(e) - M))``, with a worked example).

Also from the first page, section 3.2 (the split decision counts ``topk + extra_topk``) and
section 6.1 (an ``extra_kv`` cache beside the main one): a second KV cache with its own
index list per query token.

Readings:
  * ``topk_length`` holds one length per query token ([b, s_q]); a length above topk
    keeps every slot and a length <= 0 masks them all.
  * ``extra_kv``: a second pool of 656-byte rows with its own indices [b, s_q, extra_topk]
    (physical ids into that pool, masked by the same rule against that pool's size) and an
    optional ``extra_topk_length``; the attention runs over the union of the two slot lists,
    main slots first.
  * The sink is one value per query head ([h_q]); it changes the output only, never the
    returned lse.  A row with no valid slot keeps out = 0 and lse = +inf.
"""

from __future__ import annotations

import math

import numpy as np

LOG2E = 1.0 / math.log(2.0)


def mask_beyond_length(indices: np.ndarray, topk_length) -> np.ndarray:
    """Copy of ``indices`` [b, s_q, topk] with every slot at position >= the token's
    length replaced by -1 (the masked value)."""
    idx = np.array(indices, dtype=np.int32, copy=True)
    if topk_length is None:
        return idx
    lens = np.asarray(topk_length, dtype=np.int64).reshape(idx.shape[0], idx.shape[1])
    pos = np.arange(idx.shape[2], dtype=np.int64)[None, None, :]
    idx[pos >= lens[:, :, None]] = -1
    return idx


def join_extra(kv, indices, extra_kv, extra_indices, extra_topk_length=None):
    """One pool and one slot list equivalent to the union of the main and extra lists: the extra
    pool's pages are appended after the main pool's, valid extra ids are shifted past the main
    rows, invalid ones become -1, and each token's extra slots follow its main slots."""
    kv = np.asarray(kv, dtype=np.uint8)
    kv = kv.reshape(kv.shape[0], kv.shape[1], kv.shape[-1])
    ekv = np.asarray(extra_kv, dtype=np.uint8)
    ekv = ekv.reshape(ekv.shape[0], ekv.shape[1], ekv.shape[-1])
    assert ekv.shape[1:] == kv.shape[1:], "the extra pool has the main pool's page and row size"
    main_rows = kv.shape[0] * kv.shape[1]
    extra_rows = ekv.shape[0] * ekv.shape[1]
    eidx = mask_beyond_length(extra_indices, extra_topk_length).astype(np.int64)
    ok = (eidx >= 0) & (eidx < extra_rows)
    eidx = np.where(ok, eidx + main_rows, -1).astype(np.int32)
    pool = np.ascontiguousarray(np.concatenate([kv, ekv], axis=0))
    idx = np.ascontiguousarray(np.concatenate([np.asarray(indices, dtype=np.int32), eidx], axis=2))
    return pool, idx


def sink_factor(lse, attn_sink):
    """1 / (1 + exp(attn_sink - lse)) elementwise (natural log); 1 where lse = +inf."""
    lse = np.asarray(lse, dtype=np.float64)
    sink = np.asarray(attn_sink, dtype=np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(sink - lse))


def o_scale_kernel_form(l_sum: float, m2: float, attn_sink: float) -> float:
    """Output scale of an unsplit row as the kernel folds the sink in: exp-sum L taken
    against the base-2 running max M, sink converted to base 2."""
    return 1.0 / (l_sum + math.pow(2.0, attn_sink * LOG2E - m2))
