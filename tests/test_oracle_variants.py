"""Pins for the decode variants of the oracle (no GPU): per-token top-k length and the
attention sink.  Each ties ``oracle.variants`` and the options of
``oracle.sparse_mla_decode`` to the printed worked example, to the other page's form of
the same factor, or to a different path through the oracle that must give the same result
(a truncated top-k list; the sink as one extra key whose value vector is zero)."""

import json
import math
import os

import numpy as np
import pytest

import oracle
import workloads
from oracle import combine as ocomb
from oracle import online as oonline
from oracle import variants as ovar

SINK = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "attn_sink.json"),
                      encoding="utf-8"))


def _tiny(b=1, s_q=1, h=4, topk=16, ctx=256, seed=0, **kw):
    wl = workloads.small(b=b, s_q=s_q, h_q=h, topk=topk, ctx=ctx, seed=seed, **kw)
    return wl, *workloads.to_numpy_inputs(wl)


def _rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


# --------------------------------------------------------------------------- attention sink

def test_sink_worked_example():
    g = SINK
    assert abs(g["attn_sink"] * ovar.LOG2E - g["attn_sink_log2_printed"]) < 5e-4
    term = 2.0 ** (g["attn_sink"] * ovar.LOG2E - g["final_M_log2"])
    assert abs(term - g["exp2_term_printed"]) < 5e-4
    assert abs(g["final_L"] + term - g["denominator_printed"]) < 5e-3
    s = ovar.o_scale_kernel_form(g["final_L"], g["final_M_log2"], g["attn_sink"])
    assert abs(s - g["o_scale_printed"]) < 5e-6
    assert abs(g["rO0"] * s - g["out0_printed"]) < 5e-5
    # without the sink the scale would be 1 / L: the printed value is not that
    assert abs(1.0 / g["final_L"] - g["o_scale_printed"]) > 5e-6


def test_sink_two_page_forms_agree():
    # in-kernel form 1 / (L + 2^(sink log2e - M)) against the reference-semantics factor
    # 1 / (1 + exp(sink - lse)) applied to O / L, with lse = ln L + M ln 2
    rng = np.random.default_rng(5)
    cases = [(SINK["final_L"], SINK["final_M_log2"], SINK["attn_sink"])]
    cases += [(float(rng.uniform(1, 3000)), float(rng.uniform(-30, 30)),
               float(rng.uniform(-10, 20))) for _ in range(50)]
    for l_sum, m2, sink in cases:
        lse = math.log(l_sum) + m2 * math.log(2.0)
        a = ovar.o_scale_kernel_form(l_sum, m2, sink)
        b = float(ovar.sink_factor(lse, sink)) / l_sum
        assert abs(a - b) <= 1e-13 * abs(a)


def _with_sink_row(kv, rope_bits):
    """Pool with one page appended whose row 0 has zero NoPE codes (V = 0), unit scales and
    the given bf16 RoPE values; returns (pool, physical id of that row)."""
    nb = kv.shape[0]
    extra = np.zeros((1, 64, 656), dtype=np.uint8)
    extra[0, :, 512:528] = np.frombuffer(np.ones(4, dtype="<f4").tobytes(), np.uint8)
    extra[0, 0, 528:656] = np.frombuffer(rope_bits.astype("<u2").tobytes(), np.uint8)
    return np.ascontiguousarray(np.concatenate([kv, extra], axis=0)), nb * 64


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_sink_is_an_extra_key_with_zero_value(seed):
    # "a pretend sink token with a fixed score": decoding with sink x_h must equal decoding,
    # without a sink, a list with one more slot whose value vector is 0 and whose score for
    # head h is exactly x_h; the returned lse excludes that slot's term
    wl, q, kv, idx = _tiny(h=6, topk=40, ctx=512, masked_per_row=4, seed=seed)
    rng = np.random.default_rng(seed)
    rope = rng.standard_normal(64).astype(np.float32)
    rope_bits = (rope.view(np.uint32) >> 16).astype(np.uint16)  # bf16 by truncation
    rope_f = oracle.bf16_decode(rope_bits)
    kv2, rid = _with_sink_row(kv, rope_bits)
    x = oracle.bf16_decode(q[0, 0, :, 512:]) @ rope_f * wl.sm_scale  # [h] exact-ish in fp64
    out_s, lse_s, _ = oracle.sparse_mla_decode(q, kv, idx, wl.sm_scale, attn_sink=x)
    idx2 = np.ascontiguousarray(np.concatenate([idx, np.full((1, 1, 1), rid, np.int32)], 2))
    out_a, lse_a, _ = oracle.sparse_mla_decode(q, kv2, idx2, wl.sm_scale)
    assert _rel(out_s, out_a) < 1e-12
    assert np.max(np.abs(np.logaddexp(lse_s, x[None, :]) - lse_a)) < 1e-12
    plain, lse_p, _ = oracle.sparse_mla_decode(q, kv, idx, wl.sm_scale)
    assert np.array_equal(lse_s, lse_p)  # the sink leaves the lse alone
    assert _rel(out_s, plain) > 1e-6  # and it did change the output


def test_sink_limits_and_empty_rows():
    wl, q, kv, idx = _tiny(b=2, h=3, topk=24, ctx=256, seed=4)
    idx[1] = -1
    plain, lse, _ = oracle.sparse_mla_decode(q, kv, idx, wl.sm_scale)
    lo, lse_lo, _ = oracle.sparse_mla_decode(q, kv, idx, wl.sm_scale,
                                            attn_sink=np.full(3, -np.inf))
    assert np.array_equal(lo, plain) and np.array_equal(lse_lo, lse)
    hi, _, _ = oracle.sparse_mla_decode(q, kv, idx, wl.sm_scale,
                                        attn_sink=lse[0] + 60.0)
    assert np.max(np.abs(hi[0])) <= np.max(np.abs(plain[0])) * 1e-25
    # a token with no valid slot keeps out = 0 and lse = +inf whatever the sink
    for sink in (np.full(3, -2.5), np.full(3, 40.0)):
        o, l, _ = oracle.sparse_mla_decode(q, kv, idx, wl.sm_scale, attn_sink=sink)
        assert np.all(o[1] == 0.0) and np.all(np.isposinf(l[1]))
    # equal sink and lse halve the output
    half, _, _ = oracle.sparse_mla_decode(q, kv, idx, wl.sm_scale, tokens=[0],
                                          attn_sink=lse[0])
    assert np.allclose(half[0], plain[0] / 2, rtol=1e-13, atol=0)


def test_combine_with_sink_equals_whole():
    wl, q, kv, idx = _tiny(h=4, topk=200, ctx=1024, masked_per_row=20, seed=3)
    sink = np.array([-2.5, 4.0, 6.5, 9.0])
    whole, lw, _ = oracle.sparse_mla_decode(q, kv, idx, wl.sm_scale, attn_sink=sink)
    parts = [(0, 64), (64, 128), (128, 200)]
    res = [oracle.sparse_mla_decode(q, kv, idx, wl.sm_scale, slot_range=r) for r in parts]
    for h in range(4):
        lse2 = np.array([r[1][0, h] for r in res]) * oonline.LOG2E
        o = np.stack([r[0][0, h] for r in res])
        merged, lse = ocomb.combine(lse2, o, attn_sink=sink[h])
        assert np.allclose(merged, whole[0, h], rtol=1e-12, atol=1e-15)
        assert abs(lse - lw[0, h]) < 1e-12


# --------------------------------------------------------------------------- topk_length

def test_topk_length_equals_truncated_list():
    wl, q, kv, idx = _tiny(b=3, s_q=2, h=3, topk=70, ctx=1024, masked_per_row=5, seed=8)
    lens = np.array([[0, 1], [63, 64], [65, 70]], dtype=np.int32)
    out, lse, nv = oracle.sparse_mla_decode(q, kv, idx, wl.sm_scale, topk_length=lens)
    for t in range(6):
        bi, si = divmod(t, 2)
        n = int(lens[bi, si])
        if n == 0:
            assert np.all(out[t] == 0.0) and np.all(np.isposinf(lse[t])) and nv[t] == 0
            continue
        cut = np.ascontiguousarray(idx[:, :, :n])
        o_c, l_c, nv_c = oracle.sparse_mla_decode(q, kv, cut, wl.sm_scale, tokens=[t])
        assert np.array_equal(out[t], o_c[0]) and np.array_equal(lse[t], l_c[0])
        assert nv[t] == nv_c[0] == int(np.sum(idx[bi, si, :n] >= 0))


def test_topk_length_bounds():
    wl, q, kv, idx = _tiny(b=2, s_q=1, h=2, topk=20, seed=9)
    plain, lse, _ = oracle.sparse_mla_decode(q, kv, idx, wl.sm_scale)
    for lens in ([[20], [20]], [[25], [1 << 30]]):
        o, l, _ = oracle.sparse_mla_decode(q, kv, idx, wl.sm_scale, topk_length=lens)
        assert np.array_equal(o, plain) and np.array_equal(l, lse)
    o, l, nv = oracle.sparse_mla_decode(q, kv, idx, wl.sm_scale, topk_length=[[-3], [0]])
    assert np.all(o == 0.0) and np.all(np.isposinf(l)) and np.all(nv == 0)
    # the input array is not modified
    assert np.array_equal(idx, workloads.to_numpy_inputs(wl)[2])


# --------------------------------------------------------------------------- extra_kv

def _extra(b, s_q, h, topk, extra_topk, seed):
    wl, q, kv, idx = _tiny(b=b, s_q=s_q, h=h, topk=topk, ctx=512, masked_per_row=3, seed=seed)
    wx = workloads.small(b=b, s_q=s_q, h_q=h, topk=extra_topk, ctx=256, masked_per_row=2,
                         seed=seed + 50)
    _, ekv, eidx = workloads.to_numpy_inputs(wx)
    return wl, q, kv, idx, ekv, eidx


def test_extra_kv_equals_one_list_in_another_layout():
    # the union of the two lists, rebuilt with the extra pool FIRST and the extra slots first:
    # the same set of (query, key) pairs, so the same result
    wl, q, kv, idx, ekv, eidx = _extra(2, 2, 4, 40, 24, seed=12)
    out, lse, nv = oracle.sparse_mla_decode(q, kv, idx, wl.sm_scale, extra_kv=ekv,
                                            extra_indices=eidx)
    erows = ekv.shape[0] * ekv.shape[1]
    mrows = kv.shape[0] * kv.shape[1]
    pool = np.ascontiguousarray(np.concatenate([ekv, kv], axis=0))
    shifted = np.where((idx >= 0) & (idx < mrows), idx + erows, -1).astype(np.int32)
    both = np.ascontiguousarray(np.concatenate([eidx, shifted], axis=2))
    o2, l2, nv2 = oracle.sparse_mla_decode(q, pool, both, wl.sm_scale)
    assert _rel(out, o2) < 1e-12 and np.max(np.abs(lse - l2)) < 1e-12
    assert np.array_equal(nv, nv2) and np.all(nv == np.sum(idx >= 0, axis=2).reshape(-1)
                                              + np.sum(eidx >= 0, axis=2).reshape(-1))


def test_extra_kv_alone_and_empty():
    wl, q, kv, idx, ekv, eidx = _extra(2, 1, 3, 32, 48, seed=13)
    none = np.full_like(idx, -1)
    o, l, _ = oracle.sparse_mla_decode(q, kv, none, wl.sm_scale, extra_kv=ekv, extra_indices=eidx)
    o2, l2, _ = oracle.sparse_mla_decode(q, ekv, eidx, wl.sm_scale)
    assert np.array_equal(o, o2) and np.array_equal(l, l2)
    plain, lp, _ = oracle.sparse_mla_decode(q, kv, idx, wl.sm_scale)
    o3, l3, _ = oracle.sparse_mla_decode(q, kv, idx, wl.sm_scale, extra_kv=ekv,
                                         extra_indices=np.full_like(eidx, -1))
    assert np.array_equal(o3, plain) and np.array_equal(l3, lp)


def test_extra_kv_masks_against_its_own_pool():
    wl, q, kv, idx, ekv, eidx = _extra(1, 1, 2, 16, 16, seed=14)
    erows = ekv.shape[0] * ekv.shape[1]
    base, lb, _ = oracle.sparse_mla_decode(q, kv, idx, wl.sm_scale, extra_kv=ekv,
                                           extra_indices=eidx)
    bad = eidx.copy()
    bad[0, 0, :4] = [erows, erows + 3, -5, 1 << 30]  # outside the extra pool: masked
    ref = eidx.copy()
    ref[0, 0, :4] = -1
    o1, l1, _ = oracle.sparse_mla_decode(q, kv, idx, wl.sm_scale, extra_kv=ekv, extra_indices=bad)
    o2, l2, _ = oracle.sparse_mla_decode(q, kv, idx, wl.sm_scale, extra_kv=ekv, extra_indices=ref)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # extra_topk_length masks the extra list's tail only
    o3, l3, _ = oracle.sparse_mla_decode(q, kv, idx, wl.sm_scale, extra_kv=ekv, extra_indices=eidx,
                                         extra_topk_length=[[5]])
    cut = np.full_like(eidx, -1)
    cut[..., :5] = eidx[..., :5]
    o4, l4, _ = oracle.sparse_mla_decode(q, kv, idx, wl.sm_scale, extra_kv=ekv, extra_indices=cut)
    assert np.array_equal(o3, o4) and np.array_equal(l3, l4)
    assert not np.array_equal(o3, base)
