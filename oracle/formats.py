"""The later KV-cache formats, decoded and attended in fp64.

TEST INFRASTRUCTURE ONLY (the oracle): the product path never imports this module.

Sources, "FlashMLA 与 DSA：内核、流水线和正确性边界":

* section 3.1: after the 656-byte V3.2 row, the V4 and V4.1 caches store a page block as
  structure-of-arrays (the page's data rows first, then its scale rows), the scales become
  float8_e8m0 with groups of 64 / 32 / 16, and the bytes per token are 656 / 584 / 528 / 288;
* section 2.1 (the kernel table): the d_qk = 512 decode reads "FP8 e4m3 / e8m0, optional FP4
  extra", and the FP4 form is e2m1 values with e4m3 scales;
* section 6.4: the scale granularities per format, per-128 (V3.2) / per-64 (V4) / per-32
  (V4.1) / per-16 (FP4), with fp32 / e8m0 / e8m0 / e4m3 scales;
* section 6.1: FP4 is accepted only as the extra cache beside a V4.1 main cache; d_qk is 512
  or 576 and d_v is 512;
* section 4.3: out = exp(s - lse) @ gathered_kv[..., :d_v], so with d_qk = d_v = 512 the value
  is the whole decoded key.
"FlashMLA Sparse Decode 完整计算过程详解", step 2.3: d_qk = 576 selects the V3.2 model type,
d_qk = 512 the later one.

Readings (where the pages give the totals but not every byte): a V4 token is 448 e4m3 NoPE
codes then 64 bf16 RoPE values (576 data bytes), then 7 e8m0 scales (one per 64 NoPE dims) and
one pad byte (8 scale bytes) -- 584; a V4.1 token is 512 e4m3 codes over all 512 dims, then 16
e8m0 scales (one per 32 dims) -- 528; an FP4 token is 512 e2m1 values, two per byte with the
even element in the low nibble, then 32 e4m3 scales (one per 16 dims) -- 288.  Within a page of
64 tokens, token t's data row starts at t * data_bytes and its scale row at
64 * data_bytes + t * scale_bytes.  e8m0 is 2^(e - 127) with 0xFF = NaN; e2m1 has a sign bit,
two exponent bits (bias 1) and one mantissa bit, +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}.
"""

from __future__ import annotations

import math

import numpy as np

from . import bf16_decode, e4m3_decode, variants

PAGE = 64
D = 512  # d_qk = d_v = 512 for these formats


class Fmt:
    """Byte layout of one token of a format (data row + scale row in the page's two arrays)."""

    def __init__(self, name, data_bytes, scale_bytes):
        self.name, self.data_bytes, self.scale_bytes = name, data_bytes, scale_bytes

    @property
    def row_bytes(self) -> int:
        return self.data_bytes + self.scale_bytes

    @property
    def page_bytes(self) -> int:
        return PAGE * self.row_bytes


FORMATS = {
    "v4": Fmt("v4", 448 + 64 * 2, 8),
    "v41": Fmt("v41", 512, 16),
    "v41_fp4": Fmt("v41_fp4", 256, 32),
}


def e8m0_decode(codes) -> np.ndarray:
    """Decode e8m0 scale bytes: 2^(e - 127), NaN for 0xFF."""
    e = np.asarray(codes, dtype=np.int64)
    out = np.ldexp(1.0, e - 127)
    return np.where(e == 255, np.nan, out)


def e2m1_decode(nibbles) -> np.ndarray:
    """Decode 4-bit e2m1 values from their fields (sign, exponent with bias 1, mantissa)."""
    v = np.asarray(nibbles, dtype=np.int64) & 0xF
    s = np.where(v & 0x8, -1.0, 1.0)
    e = (v >> 1) & 0x3
    m = v & 0x1
    mag = np.where(e == 0, m * 0.5, np.ldexp(1.0 + m * 0.5, e - 1))
    return s * mag


def token_bytes(pool: np.ndarray, token: int, fmt: Fmt):
    """(data row, scale row) of physical token id ``token`` in a pool of pages."""
    flat = np.asarray(pool, dtype=np.uint8).reshape(-1)
    page, off = divmod(int(token), PAGE)
    base = page * fmt.page_bytes
    data = flat[base + off * fmt.data_bytes: base + (off + 1) * fmt.data_bytes]
    sbase = base + PAGE * fmt.data_bytes + off * fmt.scale_bytes
    return data, flat[sbase: sbase + fmt.scale_bytes]


def decode_token(pool: np.ndarray, token: int, fmt: Fmt) -> np.ndarray:
    """The 512 dims of one token (key, and the value in full)."""
    data, sc = token_bytes(pool, token, fmt)
    if fmt.name == "v4":
        nope = e4m3_decode(data[:448]) * np.repeat(e8m0_decode(sc[:7]), 64)
        rope = bf16_decode(data[448:].view("<u2"))
        return np.concatenate([nope, rope])
    if fmt.name == "v41":
        return e4m3_decode(data) * np.repeat(e8m0_decode(sc), 32)
    if fmt.name == "v41_fp4":
        vals = np.empty(D, dtype=np.float64)
        vals[0::2] = e2m1_decode(data & 0xF)
        vals[1::2] = e2m1_decode(data >> 4)
        return vals * np.repeat(e4m3_decode(sc), 16)
    raise ValueError(fmt.name)


def num_tokens(pool: np.ndarray, fmt: Fmt) -> int:
    return np.asarray(pool).size // fmt.page_bytes * PAGE


def sparse_mla_decode_fmt(q_bits, pool, indices, sm_scale, fmt: str, tokens=None,
                          slot_range=None, attn_sink=None, topk_length=None, extra_pool=None,
                          extra_fmt=None, extra_indices=None, extra_topk_length=None):
    """Sparse decode over a cache in one of the later formats (d_qk = d_v = 512), in fp64.

    q_bits: uint16 bf16 bits [b, s_q, h_q, 512]; pool: uint8 pages (any shape, whole pages);
    indices: int32 [b, s_q, topk] physical token ids (invalid: outside the pool, or beyond
    topk_length).  The optional extra cache (its own format, index list and lengths) joins
    after the main list; slot_range then indexes the joined list.  Returns (out [n, h, 512],
    lse [n, h], n_valid [n]) over ``tokens`` (default all, flattened b * s_q + s)."""
    f = FORMATS[fmt]
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    b, s_q, h, d = q_bits.shape
    assert d == D
    q = bf16_decode(q_bits.reshape(-1)).reshape(b * s_q, h, D)
    if topk_length is not None:
        indices = variants.mask_beyond_length(indices, topk_length)
    idx = np.asarray(indices, dtype=np.int64).reshape(b * s_q, -1)
    n_main = num_tokens(pool, f)
    lists = [(idx, pool, f, n_main)]
    if extra_indices is not None:
        ef = FORMATS[extra_fmt]
        eidx = extra_indices
        if extra_topk_length is not None:
            eidx = variants.mask_beyond_length(eidx, extra_topk_length)
        lists.append((np.asarray(eidx, dtype=np.int64).reshape(b * s_q, -1), extra_pool, ef,
                      num_tokens(extra_pool, ef)))
    if tokens is None:
        tokens = np.arange(b * s_q)
    tokens = np.asarray(tokens, dtype=np.int64)
    out = np.zeros((tokens.size, h, D))
    lse = np.full((tokens.size, h), math.inf)
    nv = np.zeros(tokens.size, dtype=np.int32)
    for n, t in enumerate(tokens):
        keys = []
        for lidx, lpool, lf, lrows in lists:
            for j in lidx[t]:
                keys.append((j, lpool, lf, lrows))
        lo, hi = (0, len(keys)) if slot_range is None else slot_range
        rows = [decode_token(p, j, ff) for j, p, ff, nr in keys[lo:hi] if 0 <= j < nr]
        nv[n] = len(rows)
        if not rows:
            continue
        k = np.stack(rows)                      # [n_valid, 512]
        s = q[t] @ k.T * sm_scale               # [h, n_valid]
        m = s.max(axis=1, keepdims=True)        # NaN or +inf propagate as in the definition
        l = m + np.log(np.exp(s - m).sum(axis=1, keepdims=True))
        lse[n] = l[:, 0]
        out[n] = np.exp(s - l) @ k              # V = K: all 512 dims
    if attn_sink is not None:
        assert slot_range is None, "the sink scales whole rows, not one split's share"
        out *= variants.sink_factor(lse, np.asarray(attn_sink, dtype=np.float64).reshape(1, h))[:, :, None]
    return out, lse, nv


def sparse_mla_decode_fmt_full(q_bits, pool, indices, sm_scale, fmt, **kw):
    """Library layouts: out [b, s_q, h, 512], lse [b, h, s_q]."""
    b, s_q, h, _ = q_bits.shape
    out, lse, _ = sparse_mla_decode_fmt(q_bits, pool, indices, sm_scale, fmt, **kw)
    return out.reshape(b, s_q, h, D), lse.reshape(b, s_q, h).transpose(0, 2, 1).copy()


__all__ = ["FORMATS", "Fmt", "e8m0_decode", "e2m1_decode", "decode_token", "token_bytes",
           "sparse_mla_decode_fmt", "sparse_mla_decode_fmt_full"]
