"""Pins for the later-format oracle (``oracle/formats.py``; no GPU).

Each test ties it to something other than itself: the library decoders of torch for e8m0, the
format's field definition for e2m1, the byte counts printed on the pages, hand-built pages, the
quantiser's error bound, the independent C oracle of the 656-byte format on rows built to
decode to the same values, closed forms, the split/combine identity and the extra-cache
union."""

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import combine as ocomb
from oracle import formats as F


def _bits(x: torch.Tensor) -> np.ndarray:
    return x.contiguous().view(torch.int16).numpy().view("uint16")


# ------------------------------------------------------------------------- field decoders

def test_e8m0_all_codes_match_library():
    codes = np.arange(256, dtype=np.uint8)
    mine = F.e8m0_decode(codes)
    lib = torch.from_numpy(codes.copy()).view(torch.float8_e8m0fnu).double().numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(lib)) and np.isnan(mine[255])
    ok = ~np.isnan(lib)
    assert np.array_equal(mine[ok], lib[ok])
    assert mine[127] == 1.0 and mine[0] == 2.0 ** -127 and mine[254] == 2.0 ** 127


def test_e2m1_codes():
    # sign, two exponent bits with bias 1, one mantissa bit: 0, 0.5 (subnormal), 1, 1.5, 2, 3,
    # 4, 6, and the negatives (code 8 is -0)
    want = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    got = F.e2m1_decode(np.arange(16))
    assert list(got[:8]) == want and list(-got[8:]) == want
    assert math.copysign(1.0, got[8]) < 0
    # the generator's rounding lands every representable value on its own code
    v = torch.tensor(want + [-x for x in want[1:]], dtype=torch.float32)
    assert np.array_equal(F.e2m1_decode(workloads._e2m1(v).numpy()), v.numpy())


def test_bytes_per_token_match_the_pages():
    # "FlashMLA 与 DSA", section 3.1: 656 / 584 / 528 / 288 bytes a token
    assert workloads.ROW_BYTES == 656
    assert [F.FORMATS[f].row_bytes for f in ("v4", "v41", "v41_fp4")] == [584, 528, 288]
    for f in F.FORMATS:
        assert sum(workloads.FMT_BYTES[f]) == F.FORMATS[f].row_bytes


def test_soa_addressing_on_a_hand_built_page():
    # two V4.1 pages; token 70 = page 1, row 6: its data row and scale row carry markers
    f = F.FORMATS["v41"]
    pool = np.zeros((2, f.page_bytes), dtype=np.uint8)
    pool[:, : 64 * 512] = 0x38                      # e4m3 1.0 everywhere
    pool[:, 64 * 512:] = 127                        # e8m0 1.0 everywhere
    pool[1, 6 * 512 + 33] = 0x40                    # e4m3 2.0 at dim 33 of token 70
    pool[1, 64 * 512 + 6 * 16 + 1] = 129            # scale 4 for dims 32..63 of token 70
    k = F.decode_token(pool, 70, f)
    assert k[33] == 8.0 and k[32] == 4.0 and k[63] == 4.0 and k[31] == 1.0 and k[64] == 1.0
    assert np.all(F.decode_token(pool, 69, f) == 1.0) and np.all(F.decode_token(pool, 6, f) == 1.0)
    # V4: the last 128 data bytes are bf16 RoPE values, the 8th scale byte is padding
    f4 = F.FORMATS["v4"]
    p4 = np.zeros((1, f4.page_bytes), dtype=np.uint8)
    p4[0, 64 * 576 + 5 * 8 + 7] = 0xFF              # the pad byte of token 5: not a scale
    p4[0, 64 * 576 + 5 * 8: 64 * 576 + 5 * 8 + 7] = 127
    p4[0, 5 * 576: 5 * 576 + 448] = 0x38
    p4[0, 5 * 576 + 448: 5 * 576 + 576] = np.frombuffer(
        np.full(64, 0x3FC0, dtype="<u2").tobytes(), np.uint8)  # bf16 1.5
    k4 = F.decode_token(p4, 5, f4)
    assert np.all(k4[:448] == 1.0) and np.all(k4[448:] == 1.5) and not np.isnan(k4).any()
    # FP4: the even element in the low nibble
    ff = F.FORMATS["v41_fp4"]
    pf = np.zeros((1, ff.page_bytes), dtype=np.uint8)
    pf[0, 0] = 0x72                                 # element 0: code 2 (1.0), element 1: 7 (6.0)
    pf[0, 64 * 256: 64 * 256 + 32] = 0x38           # e4m3 scale 1.0
    kf = F.decode_token(pf, 0, ff)
    assert kf[0] == 1.0 and kf[1] == 6.0 and np.all(kf[2:] == 0.0)


@pytest.mark.parametrize("fmt", ["v4", "v41", "v41_fp4"])
def test_quantiser_round_trip_within_its_bound(fmt):
    g = torch.Generator().manual_seed(7)
    x = torch.randn(64 * 3, 512, generator=g).to(torch.bfloat16)
    f = F.FORMATS[fmt]
    pool = np.zeros((3, f.page_bytes), dtype=np.uint8)
    data, sc = workloads.quantize_fmt(x, fmt)
    pool[:, : 64 * f.data_bytes] = data.view(3, -1).numpy()
    pool[:, 64 * f.data_bytes:] = sc.view(3, -1).numpy()
    dec = np.stack([F.decode_token(pool, t, f) for t in range(64 * 3)])
    xf = x.double().numpy()
    if fmt == "v41_fp4":
        # e2m1 keeps two significant bits: rms error about a tenth of the rms value
        assert np.sqrt(np.mean((dec - xf) ** 2)) < 0.15 * np.sqrt(np.mean(xf ** 2))
        return
    n_q = 448 if fmt == "v4" else 512
    gsz = 64 if fmt == "v4" else 32
    grp = xf[:, :n_q].reshape(-1, n_q // gsz, gsz)
    amax = np.abs(grp).max(-1, keepdims=True)
    scale = 2.0 ** np.ceil(np.log2(amax / 448.0))
    err = np.abs(dec[:, :n_q].reshape(grp.shape) - grp)
    assert np.all(err <= scale * np.maximum(np.abs(grp) / scale * 2.0 ** -4, 2.0 ** -10))
    if fmt == "v4":
        assert np.array_equal(dec[:, 448:], xf[:, 448:])  # RoPE stays bf16


# ------------------------------------------------------------------------- attention

def _v32_twin(keys_codes, keys_scale128, rope_bf16_bits=None):
    """656-byte rows whose NoPE decodes to codes * per-128 scale (fp32 powers of two) and whose
    RoPE is the given bf16 bits (zero by default)."""
    n = keys_codes.shape[0]
    rows = np.zeros((n, 656), dtype=np.uint8)
    rows[:, :512] = keys_codes
    rows[:, 512:528] = np.asarray(keys_scale128, dtype="<f4").reshape(n, 4).view(np.uint8)
    if rope_bf16_bits is not None:
        rows[:, 528:] = np.asarray(rope_bf16_bits, dtype="<u2").reshape(n, 64).view(np.uint8)
    pages = -(-n // 64)
    pool = np.zeros((pages * 64, 656), dtype=np.uint8)
    pool[:n] = rows
    return pool.reshape(pages, 64, 656)


def _pool_from(data, sc, fmt):
    f = F.FORMATS[fmt]
    n = data.shape[0]
    pages = -(-n // 64)
    pool = np.zeros((pages, f.page_bytes), dtype=np.uint8)
    d = np.zeros((pages * 64, f.data_bytes), np.uint8)
    s = np.zeros((pages * 64, f.scale_bytes), np.uint8)
    d[:n], s[:n] = data, sc
    pool[:, : 64 * f.data_bytes] = d.reshape(pages, -1)
    pool[:, 64 * f.data_bytes:] = s.reshape(pages, -1)
    return pool


@pytest.mark.parametrize("fmt", ["v41", "v4", "v41_fp4"])
def test_attention_equals_the_656_byte_oracle_on_twin_rows(fmt):
    # rows built so that the format's decode equals a 656-byte row's NoPE exactly (power-of-
    # two scales equal within each 128-dim group, RoPE values on the e4m3 grid); with zero
    # RoPE in the 656-byte rows and zero q there, the independent C oracle's attention over
    # 576 dims must equal this one's over 512 dims (V = K = the 512 dims)
    rng = np.random.default_rng(3)
    n, h, topk = 150, 4, 96
    e128 = rng.integers(120, 132, size=(n, 4))               # e8m0 exponent per 128 dims
    s128 = np.ldexp(1.0, e128 - 127)
    if fmt == "v41_fp4":
        nib = rng.integers(0, 16, size=(n, 512))
        vals = F.e2m1_decode(nib)                                # exactly e4m3 too
        codes = torch.from_numpy(vals).float().to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        data = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
        # e4m3 scale per 16 dims = the group's power of two (e4m3 holds 2^-9 .. 2^8)
        e4 = torch.from_numpy(np.repeat(s128, 8, axis=1)).float().to(torch.float8_e4m3fn)
        sc = e4.view(torch.uint8).numpy()
    else:
        codes = rng.integers(0, 256, size=(n, 512)).astype(np.uint8)
        codes[(codes & 0x7F) == 0x7F] = 0x38                    # no NaN code here
        if fmt == "v41":
            data, sc = codes, np.repeat(e128, 4, axis=1).astype(np.uint8)
        else:  # v4: dims 448..511 are bf16 RoPE holding the same e4m3 values times the scale
            rope = oracle.e4m3_decode(codes[:, 448:].reshape(-1)).reshape(n, 64) * s128[:, 3:4]
            rope_bits = _bits(torch.from_numpy(rope).to(torch.bfloat16))
            assert np.array_equal(oracle.bf16_decode(rope_bits.reshape(-1)).reshape(n, 64), rope)
            data = np.concatenate([codes[:, :448], rope_bits.view(np.uint8).reshape(n, 128)], 1)
            sc = np.concatenate([np.repeat(e128, 2, axis=1)[:, :7].astype(np.uint8),
                                 np.zeros((n, 1), np.uint8)], 1)
    pool = _pool_from(data, sc, fmt)
    twin = _v32_twin(codes, s128.astype(np.float32))
    q = torch.randn(2, 1, h, 512, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    q576 = torch.cat([q, torch.zeros(2, 1, h, 64, dtype=torch.bfloat16)], -1)
    idx = np.stack([rng.permutation(n)[:topk] for _ in range(2)]).astype(np.int32).reshape(2, 1, topk)
    idx[0, 0, 5] = -1
    idx[1, 0, 7] = 10_000                                  # beyond both pools: masked
    sm = 1.0 / math.sqrt(512.0)
    if fmt == "v41_fp4":
        # FP4 is an extra cache only: an empty main list, the rows as the extra list
        empty_main = np.full((2, 1, 1), -1, np.int32)
        vmain = _pool_from(np.zeros((1, 512), np.uint8), np.full((1, 16), 127, np.uint8), "v41")
        out, lse = F.sparse_mla_decode_fmt_full(_bits(q), vmain, empty_main, sm, "v41",
                                                extra_pool=pool, extra_fmt="v41_fp4",
                                                extra_indices=idx)
    else:
        out, lse = F.sparse_mla_decode_fmt_full(_bits(q), pool, idx, sm, fmt)
    ro, rl = oracle.sparse_mla_decode_full(_bits(q576), twin, idx, sm)
    assert np.max(np.abs(out - ro)) <= 1e-12 * max(1.0, np.max(np.abs(ro)))
    assert np.max(np.abs(lse - rl)) <= 1e-12


def _fmt_tiny(fmt="v41", b=2, s_q=2, h=4, topk=80, ctx=256, seed=0, **kw):
    wl = workloads.small(b=b, s_q=s_q, h_q=h, topk=topk, ctx=ctx, seed=seed, kv_format=fmt, **kw)
    return wl, _bits(wl.q), wl.kv.numpy(), wl.indices.numpy()


@pytest.mark.parametrize("fmt", ["v4", "v41"])
def test_closed_forms(fmt):
    wl, q, pool, idx = _fmt_tiny(fmt, b=1, s_q=1, topk=6)
    f = F.FORMATS[fmt]
    k = np.stack([F.decode_token(pool, j, f) for j in idx[0, 0]])
    qf = oracle.bf16_decode(q.reshape(-1)).reshape(q.shape)[0, 0]
    # one slot: out = its key (V = K, all 512 dims), lse = its score
    one = idx.copy()
    one[0, 0, 1:] = -1
    out, lse = F.sparse_mla_decode_fmt_full(q, pool, one, wl.sm_scale, fmt)
    assert np.array_equal(out[0, 0], np.broadcast_to(k[0], (4, 512)))
    assert np.allclose(lse[0, :, 0], qf @ k[0] * wl.sm_scale, rtol=1e-14, atol=1e-14)
    # zero query: the mean of the keys, lse = ln n
    out, lse = F.sparse_mla_decode_fmt_full(np.zeros_like(q), pool, idx, wl.sm_scale, fmt)
    assert np.allclose(out[0, 0], k.mean(0), rtol=1e-13, atol=1e-15)
    assert np.allclose(lse, math.log(6), rtol=1e-14)
    # all masked: 0 and +inf
    out, lse = F.sparse_mla_decode_fmt_full(q, pool, np.full_like(idx, -1), wl.sm_scale, fmt)
    assert np.all(out == 0) and np.all(np.isposinf(lse))


def test_splits_then_combine_equal_whole():
    wl, q, pool, idx = _fmt_tiny("v41", topk=150, seed=3, masked_per_row=4)
    whole, lw, _ = F.sparse_mla_decode_fmt(q, pool, idx, wl.sm_scale, "v41")
    parts = [(0, 64), (64, 100), (100, 150)]
    res = [F.sparse_mla_decode_fmt(q, pool, idx, wl.sm_scale, "v41", slot_range=r) for r in parts]
    for t in range(whole.shape[0]):
        for hh in range(whole.shape[1]):
            lse2 = [np.inf if np.isposinf(r[1][t, hh]) else r[1][t, hh] / math.log(2) for r in res]
            lse2 = [-np.inf if np.isposinf(v) else v for v in lse2]
            o, l = ocomb.combine(np.array(lse2), np.stack([r[0][t, hh] for r in res]))
            assert np.allclose(o, whole[t, hh], rtol=1e-12, atol=1e-14)
            assert abs(l - lw[t, hh]) < 1e-12


def test_extra_fp4_is_the_union():
    # the joined lists give the lse-weighted merge of the two lists taken alone
    wl, q, pool, idx = _fmt_tiny("v41", topk=64, seed=4, masked_per_row=3)
    g = torch.Generator().manual_seed(2)
    x = torch.randn(3 * 64, 512, generator=g).to(torch.bfloat16)
    data, sc = workloads.quantize_fmt(x, "v41_fp4")
    epool = _pool_from(data.numpy(), sc.numpy(), "v41_fp4")
    eidx = np.random.default_rng(9).integers(0, 3 * 64, size=(2, 2, 40)).astype(np.int32)
    eidx[0, 1, 3] = -1
    both, lb, _ = F.sparse_mla_decode_fmt(q, pool, idx, wl.sm_scale, "v41", extra_pool=epool,
                                          extra_fmt="v41_fp4", extra_indices=eidx)
    main, lm, _ = F.sparse_mla_decode_fmt(q, pool, idx, wl.sm_scale, "v41")
    empty = np.full((2, 2, 1), -1, np.int32)
    extra, le, _ = F.sparse_mla_decode_fmt(q, pool, empty, wl.sm_scale, "v41", extra_pool=epool,
                                           extra_fmt="v41_fp4", extra_indices=eidx)
    for t in range(4):
        for hh in range(4):
            o, l = ocomb.combine(np.array([lm[t, hh], le[t, hh]]) / math.log(2),
                                 np.stack([main[t, hh], extra[t, hh]]))
            assert np.allclose(o, both[t, hh], rtol=1e-12, atol=1e-14)
            assert abs(l - lb[t, hh]) < 1e-12


def test_nan_scale_makes_the_token_nan():
    wl, q, pool, idx = _fmt_tiny("v41", b=2, s_q=1, topk=16, seed=6)
    f = F.FORMATS["v41"]
    j = int(idx[0, 0, 2])
    assert j not in set(idx[1, 0].tolist())
    p2 = pool.copy().reshape(-1)
    page, off = divmod(j, 64)
    p2[page * f.page_bytes + 64 * 512 + off * 16 + 5] = 0xFF   # e8m0 NaN
    out, lse = F.sparse_mla_decode_fmt_full(q, p2.reshape(pool.shape), idx, wl.sm_scale, "v41")
    assert np.all(np.isnan(out[0])) and np.all(np.isnan(lse[0]))
    o0, l0 = F.sparse_mla_decode_fmt_full(q, pool, idx, wl.sm_scale, "v41")
    assert np.array_equal(out[1], o0[1]) and np.array_equal(lse[1], l0[1])
