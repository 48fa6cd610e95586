"""Pins for the indexer-score oracle (no GPU): a per-element triple loop with the key
dequantised first (the pages' claim that the per-token scale may be applied after the head
sum), one-hot weights picking single heads, the ReLU on signed products, the paging through
the block table, and the valid prefix."""

import numpy as np

from oracle import indexer as oix
from oracle import e4m3_decode


def _inputs(n_tok=3, s_q=1, pages=4, seed=0):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 256, size=(n_tok, 64, 128), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38  # no NaN codes
    w = rng.uniform(-1, 1, size=(n_tok, 64))
    cache = np.zeros((pages * 2, oix.PAGE_BYTES), dtype=np.uint8)
    kc = rng.integers(0, 256, size=(pages * 2, 64 * 128), dtype=np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x30
    cache[:, : 64 * 128] = kc
    cache[:, 64 * 128:] = rng.uniform(0.01, 2.0, size=(pages * 2, 64)).astype("<f4").view(np.uint8).reshape(pages * 2, 256)
    b = (n_tok + s_q - 1) // s_q
    table = np.stack([rng.permutation(pages * 2)[:pages] for _ in range(b)])
    return codes, w, cache, table


def _slow(codes, w, cache, table, valid_len, s_q, ld):
    out = np.full((codes.shape[0], ld), np.nan)
    for t in range(codes.shape[0]):
        q = e4m3_decode(codes[t].reshape(-1)).reshape(64, 128)
        for s in range(min(int(valid_len[t]), ld)):
            page = int(table[t // s_q][s // 64])
            raw = cache[page]
            k = e4m3_decode(raw[(s % 64) * 128:(s % 64) * 128 + 128])
            scale = float(raw[8192 + 4 * (s % 64):8192 + 4 * (s % 64) + 4].view("<f4")[0])
            kd = k * scale  # dequantise first
            tot = 0.0
            for j in range(64):
                tot += w[t, j] * max(float(np.dot(q[j], kd)), 0.0)
            out[t, s] = tot
    return out


def test_matches_triple_loop_with_key_dequantised_first():
    codes, w, cache, table = _inputs(n_tok=4, s_q=2, pages=3, seed=1)
    lens = [150, 64, 1, 192]
    got = oix.indexer_scores(codes, w, cache, table, lens, 2, 192)
    want = _slow(codes, w, cache, table, lens, 2, 192)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.allclose(got[ok], want[ok], rtol=1e-12, atol=1e-9)


def test_one_hot_weights_and_relu():
    codes, w, cache, table = _inputs(n_tok=1, pages=2, seed=2)
    q = e4m3_decode(codes[0].reshape(-1)).reshape(64, 128)
    keys, scales = oix.page_keys(cache, int(table[0][0]))
    for j in (0, 17, 63):
        w1 = np.zeros((1, 64)); w1[0, j] = 1.0
        got = oix.indexer_scores(codes, w1, cache, table, [64], 1, 64)[0]
        z = keys @ q[j]
        assert np.allclose(got, scales * np.maximum(z, 0.0), rtol=1e-12, atol=0)
        assert np.all(got[z < 0] == 0.0)  # negative products contribute nothing
    # negative weights subtract
    w2 = -np.ones((1, 64))
    got = oix.indexer_scores(codes, w2, cache, table, [64], 1, 64)[0]
    assert np.all(got <= 0.0)


def test_valid_prefix_and_paging():
    codes, w, cache, table = _inputs(n_tok=2, s_q=1, pages=3, seed=3)
    got = oix.indexer_scores(codes, w, cache, table, [0, 100], 1, 192)
    assert np.all(np.isnan(got[0]))
    assert np.all(~np.isnan(got[1, :100])) and np.all(np.isnan(got[1, 100:]))
    # a permuted page table permutes whole 64-token blocks of the scores
    t2 = table.copy()
    t2[1, [0, 1]] = t2[1, [1, 0]]
    g2 = oix.indexer_scores(codes, w, cache, t2, [0, 128], 1, 192)
    g1 = oix.indexer_scores(codes, w, cache, table, [0, 128], 1, 192)
    assert np.allclose(g2[1, :64], g1[1, 64:128]) and np.allclose(g2[1, 64:128], g1[1, :64])
