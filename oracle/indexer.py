"""Lightning-indexer scores over a paged FP8 key cache, in fp64 (the scores the top-k selects
from).

TEST INFRASTRUCTURE ONLY (the oracle): the product path never imports this module.

Source: "FlashMLA 与 DSA：内核、流水线和正确性边界", section 4.1 (I[t, s] = sum over the
indexer heads j of w[t, j] * ReLU(q[t, j] . k[s]); e4m3 q and k, one key per cached token
shared by the 64 heads) and section 5.3 (the cache page layout: 64 tokens x 128 e4m3 codes,
then their 64 fp32 scales, 8448 bytes a page; the per-token key scale multiplies the sum over
heads); "sparse-attention co-design", section 5, steps one to four (the query scale and the
normalisations are folded into w, so the scorer reads the e4m3 codes of q as they are).

Reading: ``I[t, s] = k_scale[s] * sum_j w[t, j] * max(q8[t, j] . k8[s], 0)`` with q8, k8 the
decoded e4m3 values, for the positions s < valid_len[t]; token t belongs to request t // s_q
and reads that request's pages through the block table.
"""

from __future__ import annotations

import numpy as np

from . import e4m3_decode

PAGE_TOKENS, DIM, HEADS = 64, 128, 64
PAGE_BYTES = PAGE_TOKENS * DIM + PAGE_TOKENS * 4  # 8448


def page_keys(cache: np.ndarray, page: int):
    """(keys fp64 [64, 128], scales fp64 [64]) of one cache page."""
    raw = np.asarray(cache[page], dtype=np.uint8)
    codes = raw[: PAGE_TOKENS * DIM].reshape(PAGE_TOKENS, DIM)
    scales = raw[PAGE_TOKENS * DIM:].copy().view("<f4").astype(np.float64)
    return e4m3_decode(codes.reshape(-1)).reshape(PAGE_TOKENS, DIM), scales


def indexer_scores(q_codes: np.ndarray, w: np.ndarray, cache: np.ndarray, block_table: np.ndarray,
                   valid_len, s_q: int, ld: int) -> np.ndarray:
    """q_codes uint8 [n_tok, 64, 128], w [n_tok, 64], cache uint8 [pages, 8448], block_table
    int [b, max_pages].  Returns fp64 [n_tok, ld] with NaN past each token's valid prefix."""
    n_tok = q_codes.shape[0]
    out = np.full((n_tok, ld), np.nan)
    q = e4m3_decode(np.asarray(q_codes, dtype=np.uint8).reshape(-1)).reshape(n_tok, HEADS, DIM)
    w = np.asarray(w, dtype=np.float64)
    for t in range(n_tok):
        n = max(0, min(int(valid_len[t]), ld))
        if n == 0:
            continue
        pages = (n + PAGE_TOKENS - 1) // PAGE_TOKENS
        keys, scales = zip(*(page_keys(cache, int(block_table[t // s_q][i])) for i in range(pages)))
        k = np.concatenate(keys)[:n]          # [n, 128]
        ks = np.concatenate(scales)[:n]       # [n]
        z = q[t] @ k.T                        # [64 heads, n]
        out[t, :n] = ks * (w[t] @ np.maximum(z, 0.0))
    return out
