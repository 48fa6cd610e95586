"""Pins for the CPU oracle (no GPU).  Each test ties an oracle function to something other
than itself: values printed on the pages, a library routine, a closed form, an invariant
or an independent brute-force path."""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import combine as ocomb
from oracle import online as oonline
from oracle import sched as osched
from tests import brute

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_example.json"),
                      encoding="utf-8"))
SM_SCALE = 1.0 / math.sqrt(576.0)


# --------------------------------------------------------------------------- e4m3 / bf16

def test_e4m3_all_codes_match_library():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_decode(codes)
    lib = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], lib[~nan])
    assert np.array_equal(np.signbit(mine[~nan]), np.signbit(lib[~nan]))


def test_e4m3_spec_facts():
    assert oracle.e4m3_decode([0x7E])[0] == 448.0
    assert oracle.e4m3_decode([0xFE])[0] == -448.0
    assert oracle.e4m3_decode([0x01])[0] == 2.0 ** -9
    assert oracle.e4m3_decode([0x08])[0] == 2.0 ** -6
    assert np.isnan(oracle.e4m3_decode([0x7F])[0]) and np.isnan(oracle.e4m3_decode([0xFF])[0])
    z = oracle.e4m3_decode([0x80])[0]
    assert z == 0.0 and math.copysign(1.0, z) < 0


def test_bf16_all_patterns_match_library():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle.bf16_decode(bits)
    lib = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(
        torch.float64).numpy()
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], lib[~nan])


def _e4m3_code(v: float) -> int:
    return int(torch.tensor([v], dtype=torch.float32).to(torch.float8_e4m3fn).view(
        torch.uint8)[0])


def test_worked_example_dequant():
    g = GOLD["dequant"]
    row = np.zeros(656, dtype=np.uint8)
    for i, v in enumerate(g["e4m3_values"]):
        row[i] = _e4m3_code(v)
    row[512:516] = np.frombuffer(np.float32(g["scale"]).tobytes(), dtype=np.uint8)
    row[516:528] = np.frombuffer(np.ones(3, dtype="<f4").tobytes(), dtype=np.uint8)
    k = oracle.decode_row(row)
    assert np.array_equal(k[:8], np.array(g["expected"]))
    assert np.all(k[8:512] == 0.0) and np.all(k[512:] == 0.0)


def test_decode_row_groups_and_rope_match_library():
    rng = np.random.default_rng(5)
    rows = rng.integers(0, 256, size=(17, 656), dtype=np.uint8)
    rows[:, :512][rows[:, :512] & 0x7F == 0x7F] = 0x10  # no NaN codes
    rows[:, 512:528] = np.frombuffer(rng.uniform(0.001, 3.0, (17, 4)).astype("<f4").tobytes(),
                                     dtype=np.uint8).reshape(17, 16)
    rope = rng.standard_normal((17, 64)).astype(np.float32)
    rows[:, 528:] = torch.from_numpy(rope).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint8).reshape(17, 128)
    ref = brute.decode_rows_lib(rows)
    for i in range(17):
        assert np.array_equal(oracle.decode_row(rows[i]), ref[i])


# --------------------------------------------------------------------------- generator pins

def test_ue8m0_worked_example():
    g = GOLD["ue8m0"]
    assert abs(g["amax"] / 448.0 - g["amax_over_448"]) < 5e-7
    s = workloads.ue8m0_scale(torch.tensor([g["amax"] / 448.0], dtype=torch.float32))
    assert float(s[0]) == g["scale_ue8m0"]
    x = torch.zeros(1, 576, dtype=torch.bfloat16)
    x[0, 0] = g["x0"]
    x[0, 1] = g["amax"]
    row = workloads.quantize_rows(x, ue8m0=True)[0].numpy()
    assert row[512:516].view("<f4")[0] == g["scale_ue8m0"]
    assert oracle.e4m3_decode([row[0]])[0] == g["code0_value"]


def test_quantiser_roundtrip_bound():
    x = torch.randn(64, 576, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    rows = workloads.quantize_rows(x).numpy()
    k = np.stack([oracle.decode_row(r) for r in rows])
    xf = x.double().numpy()
    # e4m3 keeps 3 mantissa bits: relative error <= 2^-4 of the group amax in the worst case
    amax = np.abs(xf[:, :512]).reshape(64, 4, 128).max(-1)
    err = np.abs(k[:, :512] - xf[:, :512]).reshape(64, 4, 128).max(-1)
    assert np.all(err <= amax * 2.0 ** -4 + 1e-12)
    assert np.array_equal(k[:, 512:], xf[:, 512:])  # RoPE stored exactly


# --------------------------------------------------------------------------- attention core

def _tiny(b=2, s_q=2, h=4, topk=8, ctx=256, seed=0, **kw):
    wl = workloads.small(b=b, s_q=s_q, h_q=h, topk=topk, ctx=ctx, seed=seed, **kw)
    return wl, *workloads.to_numpy_inputs(wl)


def _rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_oracle_matches_bruteforce(seed):
    wl, q, kv, idx = _tiny(seed=seed, masked_per_row=2)
    out, lse = oracle.sparse_mla_decode_full(q, kv, idx, wl.sm_scale)
    bo, bl = brute.sparse_attention(q, kv, idx, wl.sm_scale)
    assert _rel(out, bo) < 1e-12
    assert np.max(np.abs(lse - bl)) < 1e-12


def test_addressing_worked_example():
    g = GOLD["addressing"]
    assert divmod(g["index"], g["page_block_size"]) == (g["block"], g["offset"])
    # Token id 47 must read page 0, row 47: make that the only valid slot and check O = V.
    wl, q, kv, idx = _tiny(b=1, s_q=1, h=2, topk=4, ctx=128)
    idx[:] = -1
    idx[0, 0, 1] = g["index"]
    out, lse = oracle.sparse_mla_decode_full(q, kv, idx, wl.sm_scale)
    v = brute.decode_rows_lib(kv.reshape(-1, 656)[[g["block"] * 64 + g["offset"]]])[0]
    assert np.array_equal(out[0, 0, 0], v[:512])


def test_topk_equal_ctx_is_dense_mla():
    ctx = 192  # three pages per sequence, scattered in the pool
    wl, q, kv, idx = _tiny(b=2, s_q=1, h=3, topk=ctx, ctx=ctx, seed=7, extra_pool_pages=5)
    # every position of each sequence, in a random order
    bt = wl.block_table.numpy()
    rng = np.random.default_rng(3)
    for s in range(2):
        pos = rng.permutation(ctx)
        idx[s, 0] = bt[s, pos // 64] * 64 + pos % 64
    out, lse = oracle.sparse_mla_decode_full(q, kv, idx, wl.sm_scale)
    for s in range(2):
        do, dl = brute.dense_attention(q, kv, bt, ctx, wl.sm_scale, s)
        assert _rel(out[s], do) < 1e-12
        assert np.max(np.abs(lse[s].T - dl)) < 1e-12


def _keys(kv, ids):
    return np.stack([oracle.decode_row(kv.reshape(-1, 656)[i]) for i in ids])


def test_closed_form_topk1():
    wl, q, kv, idx = _tiny(b=1, s_q=1, h=4, topk=1)
    out, lse = oracle.sparse_mla_decode_full(q, kv, idx, wl.sm_scale)
    k = _keys(kv, [idx[0, 0, 0]])[0]
    qf = oracle.bf16_decode(q[0, 0])
    assert np.array_equal(out[0, 0], np.broadcast_to(k[:512], (4, 512)))
    assert np.allclose(lse[0, :, 0], qf @ k * wl.sm_scale, rtol=1e-14, atol=1e-14)


def test_closed_form_zero_query():
    wl, q, kv, idx = _tiny(b=1, s_q=1, h=2, topk=16, masked_per_row=3)
    q[:] = 0
    out, lse = oracle.sparse_mla_decode_full(q, kv, idx, wl.sm_scale)
    valid = idx[0, 0][idx[0, 0] >= 0]
    k = _keys(kv, valid)
    assert np.allclose(out[0, 0], k[:, :512].mean(0), rtol=1e-13, atol=1e-15)
    assert np.allclose(lse[0, :, 0], math.log(len(valid)), rtol=1e-14)


def test_closed_form_two_slots():
    wl, q, kv, idx = _tiny(b=1, s_q=1, h=3, topk=6)
    idx[0, 0, 2:] = -1
    out, lse = oracle.sparse_mla_decode_full(q, kv, idx, wl.sm_scale)
    k = _keys(kv, idx[0, 0, :2])
    qf = oracle.bf16_decode(q[0, 0])
    s = qf @ k.T * wl.sm_scale  # [h, 2]
    sig = 1.0 / (1.0 + np.exp(-(s[:, 0] - s[:, 1])))
    want = sig[:, None] * k[0, :512] + (1 - sig)[:, None] * k[1, :512]
    assert np.allclose(out[0, 0], want, rtol=1e-12, atol=1e-15)
    assert np.allclose(lse[0, :, 0], np.logaddexp(s[:, 0], s[:, 1]), rtol=1e-14)


def test_invariants_lse_permutation_masking_duplicates():
    wl, q, kv, idx = _tiny(b=1, s_q=2, h=4, topk=32, ctx=512, seed=11)
    out, lse = oracle.sparse_mla_decode_full(q, kv, idx, wl.sm_scale)
    qf = oracle.bf16_decode(q)
    # lse = ln sum exp(s_j), recomputed from the decoded rows
    for si in range(2):
        k = _keys(kv, idx[0, si])
        s = qf[0, si] @ k.T * wl.sm_scale
        m = s.max(1)
        assert np.allclose(lse[0, :, si], m + np.log(np.exp(s - m[:, None]).sum(1)), rtol=1e-13)
    # permutation of the slots
    perm = np.random.default_rng(1).permutation(32)
    o2, l2 = oracle.sparse_mla_decode_full(q, kv, idx[:, :, perm].copy(), wl.sm_scale)
    assert _rel(o2, out) < 1e-12 and np.max(np.abs(l2 - lse)) < 1e-12
    # inserting -1 and out-of-range slots changes nothing
    nrows = kv.shape[0] * 64
    pad = np.concatenate([idx, np.full((1, 2, 5), -1, np.int32),
                          np.full((1, 2, 3), nrows, np.int32),
                          np.full((1, 2, 2), -7, np.int32)], axis=2)
    o3, l3 = oracle.sparse_mla_decode_full(q, kv, np.ascontiguousarray(pad), wl.sm_scale)
    assert _rel(o3, out) < 1e-12 and np.max(np.abs(l3 - lse)) < 1e-12
    # a duplicated slot counts twice: same as adding ln 2 to that slot's score
    dup = np.concatenate([idx, idx[:, :, :1]], axis=2)
    o4, l4 = oracle.sparse_mla_decode_full(q, kv, np.ascontiguousarray(dup), wl.sm_scale)
    k = _keys(kv, idx[0, 0])
    s = qf[0, 0] @ k.T * wl.sm_scale
    s[:, 0] += math.log(2.0)
    w = np.exp(s - s.max(1, keepdims=True))
    w /= w.sum(1, keepdims=True)
    assert np.allclose(o4[0, 0], w @ k[:, :512], rtol=1e-12, atol=1e-15)


def test_all_masked_row_defined_output():
    wl, q, kv, idx = _tiny(b=2, s_q=1, h=2, topk=8)
    idx[1] = -1
    out, lse = oracle.sparse_mla_decode_full(q, kv, idx, wl.sm_scale)
    assert np.all(out[1] == 0.0) and np.all(np.isposinf(lse[1]))
    assert np.all(np.isfinite(lse[0]))


def test_non_finite_key_values_follow_the_definition():
    # the plain definition in exact arithmetic: a NaN anywhere in a valid key row makes every
    # score of that token NaN, hence its whole output and lse; a +inf score gives inf - inf =
    # NaN in the softmax; a -inf score only adds exp(-inf) = 0, the same as masking the slot
    wl, q, kv, idx = _tiny(b=2, s_q=1, h=4, topk=8, seed=5)
    out0, lse0 = oracle.sparse_mla_decode_full(q, kv, idx, wl.sm_scale)
    flat = kv.reshape(-1, 656)
    r = int(idx[0, 0, 3])
    assert r not in set(idx[1, 0].tolist())
    for where, patch in (("nope", {17: 0x7F}), ("rope", {528 + 2 * 5: 0xC0, 529 + 2 * 5: 0x7F})):
        kv2 = kv.copy()
        f2 = kv2.reshape(-1, 656)
        for byte, v in patch.items():
            f2[r, byte] = v
        out, lse = oracle.sparse_mla_decode_full(q, kv2, idx, wl.sm_scale)
        assert np.all(np.isnan(out[0])) and np.all(np.isnan(lse[0])), where
        assert np.array_equal(out[1], out0[1]) and np.array_equal(lse[1], lse0[1]), where
    # bf16 +inf in RoPE dim 5: heads whose q there is positive see +inf (NaN row), heads
    # with a negative value see -inf (the slot drops out, as if it were masked)
    kv3 = kv.copy()
    f3 = kv3.reshape(-1, 656)
    f3[r, 528 + 10], f3[r, 529 + 10] = 0x80, 0x7F
    out, lse = oracle.sparse_mla_decode_full(q, kv3, idx, wl.sm_scale)
    masked = idx.copy()
    masked[0, 0, 3] = -1
    om, lm = oracle.sparse_mla_decode_full(q, kv, masked, wl.sm_scale)
    qr = oracle.bf16_decode(q[0, 0, :, 512 + 5])
    assert np.all(qr != 0)
    for h in range(4):
        if qr[h] > 0:
            assert np.all(np.isnan(out[0, 0, h])) and np.isnan(lse[0, h, 0])
        else:
            assert _rel(out[0, 0, h], om[0, 0, h]) < 1e-12 and abs(lse[0, h, 0] - lm[0, h, 0]) < 1e-12
    assert (qr > 0).any() and (qr < 0).any()


# --------------------------------------------------------------------------- splits / combine

def test_combine_worked_example_corrected():
    g = GOLD["combine"]
    lse2 = np.array(g["lse2"])
    assert np.allclose(np.exp2(lse2 - g["max_lse"]), g["terms"], atol=1e-6)
    assert abs(np.exp2(lse2 - g["max_lse"]).sum() - g["sum"]) < 1e-6
    assert np.allclose(ocomb.weights(lse2), g["weights"], atol=1e-6)
    o = np.eye(3)
    merged, lse = ocomb.combine(lse2, o)
    assert np.allclose(merged, g["weights"], atol=1e-6)
    assert abs(lse - g["lse_natural"]) < 1e-6
    # the page's printed third term is e^-2, which the base-2 formula does not give
    assert abs(np.exp2(g["lse2"][2] - g["max_lse"]) - g["page_printed_terms_wrong"][2]) > 0.05


def test_combine_all_empty():
    o, lse = ocomb.combine(np.array([-np.inf, -np.inf]), np.zeros((2, 512)))
    assert np.all(o == 0) and lse == math.inf


def test_splits_then_combine_equal_whole():
    wl, q, kv, idx = _tiny(b=1, s_q=1, h=4, topk=200, ctx=1024, masked_per_row=20, seed=3)
    whole, lw, _ = oracle.sparse_mla_decode(q, kv, idx, wl.sm_scale)
    parts = [(0, 64), (64, 128), (128, 200)]
    res = [oracle.sparse_mla_decode(q, kv, idx, wl.sm_scale, slot_range=r) for r in parts]
    for h in range(4):
        lse2 = np.array([r[1][0, h] for r in res]) * oonline.LOG2E
        o = np.stack([r[0][0, h] for r in res])
        merged, lse = ocomb.combine(lse2, o)
        assert np.allclose(merged, whole[0, h], rtol=1e-12, atol=1e-15)
        assert abs(lse - lw[0, h]) < 1e-12


# --------------------------------------------------------------------------- online softmax

def test_online_softmax_worked_example():
    g = GOLD["softmax"]
    scale_log2 = SM_SCALE * oonline.LOG2E
    assert abs(scale_log2 - g["scale_log2_printed"]) < 5e-5
    st = oonline.State()
    p, a = st.update(np.array(g["block1_scores"]), scale_log2)
    assert abs(st.m - g["block1_max_scaled"]) < 5e-4
    assert a == 0.0  # first block: old output discarded
    assert np.allclose(p, g["block1_p"], atol=1e-3)
    m1 = st.m
    p, a = st.update(np.array(g["block2_scores"]), scale_log2)
    assert abs(g["block2_scores"][0] * scale_log2 - g["block2_max_scaled"]) < 5e-4
    assert st.m == m1 and a == g["block2_rescale"]
    assert np.allclose(p, g["block2_p"], atol=1e-3)
    st.l, st.m = g["final_L"], g["final_M"]
    assert abs(st.lse() - g["final_lse"]) < 1e-3


def test_online_softmax_matches_two_pass():
    rng = np.random.default_rng(0)
    s = rng.standard_normal(300) * 30
    v = rng.standard_normal((300, 16))
    valid = rng.random(300) > 0.1
    o, lse = oonline.run(s, v, SM_SCALE * oonline.LOG2E, valid=valid)
    t = s[valid] * SM_SCALE
    w = np.exp(t - t.max())
    assert np.allclose(o, (w / w.sum()) @ v[valid], rtol=1e-12)
    assert abs(lse - (t.max() + math.log(w.sum()))) < 1e-12
    o0, l0 = oonline.run(s, v, 0.1, valid=np.zeros(300, bool))
    assert np.all(o0 == 0) and l0 == math.inf


# --------------------------------------------------------------------------- scheduler

def test_scheduler_worked_example():
    g = GOLD["scheduler"]
    parts = osched.num_sm_parts(g["num_sms"], g["s_q"])
    assert parts == g["num_sm_parts"]
    plan, prefix = osched.plan([g["topk"]] * g["b"], parts)
    assert prefix == g["num_splits_prefix"]
    for want, got in zip(g["partitions"], plan):
        assert (got.begin_req, got.end_req, got.begin_block, got.end_block,
                got.is_first_req_splitted, got.is_last_req_splitted) == (
            want["begin_req"], want["end_req"], want["begin_block"], want["end_block"],
            want["is_first_req_splitted"], want["is_last_req_splitted"])
    assert all(p.empty(g["b"]) for p in plan[len(g["partitions"]):])
    assert [p.begin_split_idx for p in plan[:4]] == [0, 1, 2, 3]


@pytest.mark.parametrize("b,topk,parts", [(64, 2048, 76), (32, 2048, 76), (128, 2048, 38),
                                          (1, 2048, 1), (3, 100, 7), (5, 0, 4), (200, 64, 3),
                                          (7, 1, 76), (2, 65, 76), (33, 4096, 76), (76, 640, 76),
                                          (9, 2048 + 64 * 7, 37), (1, 64, 76)])
def test_scheduler_covers_every_block_once(b, topk, parts):
    plan, prefix = osched.plan([topk] * b, parts)
    nb = -(-topk // 64)
    seen = np.zeros((b, max(nb, 1)), dtype=int)
    reqs_touched = np.zeros(b, dtype=int)
    slots = set()
    for p in plan:
        if p.empty(b):
            continue
        for r in range(p.begin_req, p.end_req + 1):
            lo, hi = osched.block_range(p, r, nb)
            # every request a partition touches gets at least one of its blocks (the decode
            # kernel relies on it: each (position, request) item has a last block)
            assert 0 <= lo < hi <= nb if nb else lo == hi == 0
            seen[r, lo:hi] += 1
            reqs_touched[r] += 1
            slot = p.begin_split_idx if r == p.begin_req else prefix[r]
            assert prefix[r] <= slot < prefix[r + 1]
            assert slot not in slots
            slots.add(slot)
    if nb:
        assert np.all(seen[:, :nb] == 1)
    assert np.array_equal(np.diff(prefix), reqs_touched)
    assert len(slots) == prefix[-1]
