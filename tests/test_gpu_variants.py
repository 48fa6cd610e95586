"""GPU parity of the decode variants (attention sink, per-token top-k length) through the C
ABI against the fp64 oracle: small cases in full on unsplit and split plans, the combine
kernel with a sink on synthetic partials, and the full-size b=64 / h=128 / topk=2048
workload with both variants on every query token."""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import sched as osched
import workloads
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(cuda_ok):
    import sparse_mla_attention_decode_gb300 as smla
    smla.lib()
    return torch.device("cuda:0")


def _full(wl, num_sms, what, sink=None, lens=None):
    out, lse, _ = gu.run_cuda(wl, num_sms=num_sms, attn_sink=sink, topk_length=lens)
    q, kv, idx = workloads.to_numpy_inputs(wl)
    ro, rl = oracle.sparse_mla_decode_full(
        q, kv, idx, wl.sm_scale,
        attn_sink=None if sink is None else sink.double().cpu().numpy(),
        topk_length=None if lens is None else lens.cpu().numpy())
    h = wl.spec.h_q
    go = out.double().cpu().numpy().reshape(-1, h, 512)
    gl = lse.double().cpu().numpy().transpose(0, 2, 1).reshape(-1, h)
    m = gu.compare(go, gl, ro.reshape(-1, h, 512), rl.transpose(0, 2, 1).reshape(-1, h), what)
    return m, go


CASES = [
    # (name, workload kwargs, num_sms, sink, lengths)
    ("sink_nosplit_h128", dict(b=3, h_q=128, topk=300, ctx=2048, masked_per_row=20), 8,
     True, False),
    ("sink_split_h128", dict(b=3, h_q=128, topk=300, ctx=2048, masked_per_row=20), 132,
     True, False),
    ("sink_split_h64_sq2", dict(b=2, s_q=2, h_q=64, topk=256, ctx=1024, causal_base=700), 48,
     True, False),
    ("len_nosplit_h128", dict(b=7, h_q=128, topk=200, ctx=1024, masked_per_row=9), 8,
     False, True),
    ("len_split_h64", dict(b=4, s_q=2, h_q=64, topk=330, ctx=2048), 64, False, True),
    ("both_split_h128", dict(b=7, h_q=128, topk=320, ctx=4096, ue8m0=True), 152, True, True),
    ("both_nosplit_h64", dict(b=9, h_q=64, topk=130, ctx=1024, masked_per_row=5), 6,
     True, True),
]


@pytest.mark.parametrize("name,kw,num_sms,use_sink,use_len", CASES, ids=[c[0] for c in CASES])
def test_variant_parity(dev, name, kw, num_sms, use_sink, use_len):
    seed = 500 + sum(map(ord, name))
    wl = workloads.small(device=dev, seed=seed, **kw)
    sink = workloads.attn_sink(wl.spec.h_q, seed, device=dev) if use_sink else None
    lens = (workloads.topk_lengths(wl.spec.b, wl.spec.s_q, wl.spec.topk, seed, device=dev)
            if use_len else None)
    m, go = _full(wl, num_sms, name, sink, lens)
    print(name, m)
    # the variant must have changed the result: compare with the plain decode
    plain, _, _ = gu.run_cuda(wl, num_sms=num_sms)
    diff = np.abs(go - plain.double().cpu().numpy().reshape(go.shape)).max()
    assert diff > 2 * gu.O_MAX_ABS, f"{name}: the variant left the output unchanged ({diff})"


def test_combine_kernel_with_sink(dev):
    import sparse_mla_attention_decode_gb300 as smla
    from oracle import combine as ocomb
    b, s_q, h = 3, 2, 64
    op = smla.SparseMLADecode(b, s_q, h, 2048, 64, device=dev, num_sms=40)
    st = torch.cuda.current_stream().cuda_stream
    smla.sparse_mla_sched_meta(op.dims, op.num_sms, op.sched.data_ptr(), op.sched_bytes, st)
    torch.cuda.synchronize()
    parts = max(op.num_sms // s_q // 2, 1)
    # the oracle planner's split layout (the GPU plan must equal it)
    _, pre = osched.plan([2048] * b, osched.num_sm_parts(op.num_sms, s_q))
    assert op.plan()[1].tolist() == pre
    max_splits, lse_off = gu.accum_layout(pre, s_q, h)
    g = torch.Generator(device="cpu").manual_seed(14)
    o_acc = torch.randn(max_splits, s_q, h, 512, generator=g)
    l_acc = torch.randn(max_splits, s_q, h, generator=g) * 4 + 6
    l_acc[pre[1]:pre[2], 1, 7] = -math.inf  # a row whose splits are all empty
    sink = workloads.attn_sink(h, 3)
    sink[5] = 60.0   # far above every lse: output about 0
    sink[6] = -60.0  # far below: no effect
    ws = op.workspace
    ws[: o_acc.numel() * 4].copy_(o_acc.view(torch.uint8).view(-1).to(dev))
    ws[lse_off:lse_off + l_acc.numel() * 4].copy_(l_acc.contiguous().view(torch.uint8).view(-1).to(dev))
    out = torch.full((b, s_q, h, 512), 7.0, dtype=torch.bfloat16, device=dev)
    lse = torch.full((b, h, s_q), 7.0, dtype=torch.float32, device=dev)
    sink_d = sink.to(dev)
    opts = smla.smla_decode_opts(sink_d.data_ptr(), None)
    smla.sparse_mla_combine_ex(op.dims, op.num_sms, opts, op.sched.data_ptr(), ws.data_ptr(),
                               op.accum_bytes, out.data_ptr(), lse.data_ptr(), st)
    torch.cuda.synchronize()
    out, lse = out.double().cpu().numpy(), lse.double().cpu().numpy()
    checked = 0
    for r in range(b):
        n = pre[r + 1] - pre[r]
        for s in range(s_q):
            for hh in range(h):
                if n <= 1:
                    assert np.all(out[r, s, hh] == 7.0) and lse[r, hh, s] == 7.0
                    continue
                ro, rl = ocomb.combine(l_acc[pre[r]:pre[r + 1], s, hh].double().numpy(),
                                       o_acc[pre[r]:pre[r + 1], s, hh].double().numpy(),
                                       attn_sink=float(sink[hh]))
                if math.isinf(rl):
                    assert np.all(out[r, s, hh] == 0) and np.isposinf(lse[r, hh, s])
                else:
                    assert np.max(np.abs(out[r, s, hh] - ro)) <= 1e-2 * max(1, np.abs(ro).max())
                    assert abs(lse[r, hh, s] - rl) <= 1e-4
                    checked += 1
    assert checked > 100


def test_full_size_workload_with_variants(dev):
    spec = workloads.CONFIGS["c2_b64_h128_k2048_mask5"]
    wl = workloads.make(spec, device=dev)
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sink = workloads.attn_sink(spec.h_q, 77, device=dev)
    lens = workloads.topk_lengths(spec.b, spec.s_q, spec.topk, 77, device=dev)
    out, lse, _ = gu.run_cuda(wl, num_sms=num_sms, attn_sink=sink, topk_length=lens)
    tokens = np.arange(spec.b * spec.s_q)  # every query token
    ro, rl = gu.oracle_tokens(wl, tokens, attn_sink=sink, topk_length=lens)
    go, gl = gu.gpu_tokens(out, lse, wl, tokens)
    print(gu.compare(go, gl, ro, rl, "c2 with sink and lengths"))


# ----------------------------------------------------------------------------- bf16 partials

BF16_CASES = [
    ("bf16p_many_splits_h128", dict(b=1, h_q=128, topk=2048, ctx=8192), 152, False),
    ("bf16p_split_h64_sq2", dict(b=3, s_q=2, h_q=64, topk=640, ctx=4096, masked_per_row=30), 60,
     False),
    ("bf16p_split_sink_h128", dict(b=4, h_q=128, topk=512, ctx=4096, ue8m0=True), 120, True),
]


@pytest.mark.parametrize("name,kw,num_sms,use_sink", BF16_CASES, ids=[c[0] for c in BF16_CASES])
def test_bf16_partials_parity(dev, name, kw, num_sms, use_sink):
    seed = 900 + sum(map(ord, name))
    wl = workloads.small(device=dev, seed=seed, **kw)
    sink = workloads.attn_sink(wl.spec.h_q, seed, device=dev) if use_sink else None
    out, lse, op = gu.run_cuda(wl, num_sms=num_sms, attn_sink=sink, partials_bf16=True)
    _, pre = op.plan()
    assert int((pre[1:] - pre[:-1]).max()) > 1, "the case must have split requests"
    q, kv, idx = workloads.to_numpy_inputs(wl)
    ro, rl = oracle.sparse_mla_decode_full(
        q, kv, idx, wl.sm_scale, attn_sink=None if sink is None else sink.double().cpu().numpy())
    h = wl.spec.h_q
    go = out.double().cpu().numpy().reshape(-1, h, 512)
    gl = lse.double().cpu().numpy().transpose(0, 2, 1).reshape(-1, h)
    print(name, gu.compare(go, gl, ro.reshape(-1, h, 512), rl.transpose(0, 2, 1).reshape(-1, h),
                           name))
    # against the fp32-partial path: the same lse, outputs a few bf16 steps apart at most
    out32, lse32, _ = gu.run_cuda(wl, num_sms=num_sms, attn_sink=sink)
    assert torch.allclose(lse, lse32, rtol=0, atol=1e-5)
    d = (out.float() - out32.float()).abs()
    assert d.max().item() <= 4 * 2.0 ** -8 * max(1.0, out32.float().abs().max().item())
    assert d.max().item() > 0, "the bf16-partial path gave bit-identical results"


def test_combine_kernel_bf16_partials(dev):
    import sparse_mla_attention_decode_gb300 as smla
    from oracle import combine as ocomb
    b, s_q, h = 2, 3, 128
    op = smla.SparseMLADecode(b, s_q, h, 2048, 64, device=dev, num_sms=60)
    st = torch.cuda.current_stream().cuda_stream
    smla.sparse_mla_sched_meta(op.dims, op.num_sms, op.sched.data_ptr(), op.sched_bytes, st)
    torch.cuda.synchronize()
    parts = max(op.num_sms // s_q // 2, 1)
    # the oracle planner's split layout (the GPU plan must equal it)
    _, pre = osched.plan([2048] * b, osched.num_sm_parts(op.num_sms, s_q))
    assert op.plan()[1].tolist() == pre
    max_splits, lse_off = gu.accum_layout(pre, s_q, h)
    g = torch.Generator(device="cpu").manual_seed(15)
    o_acc = torch.randn(max_splits, s_q, h, 512, generator=g).to(torch.bfloat16)
    l_acc = torch.randn(max_splits, s_q, h, generator=g) * 3
    l_acc[pre[0], 1, :9] = -math.inf
    ws = op.workspace
    ws[: o_acc.numel() * 2].copy_(o_acc.view(torch.uint8).view(-1).to(dev))
    ws[lse_off:lse_off + l_acc.numel() * 4].copy_(l_acc.contiguous().view(torch.uint8).view(-1).to(dev))
    out = torch.full((b, s_q, h, 512), 7.0, dtype=torch.bfloat16, device=dev)
    lse = torch.full((b, h, s_q), 7.0, dtype=torch.float32, device=dev)
    opts = smla.smla_decode_opts(None, None, 1)
    smla.sparse_mla_combine_ex(op.dims, op.num_sms, opts, op.sched.data_ptr(), ws.data_ptr(),
                               op.accum_bytes, out.data_ptr(), lse.data_ptr(), st)
    torch.cuda.synchronize()
    out, lse = out.double().cpu().numpy(), lse.double().cpu().numpy()
    checked = 0
    for r in range(b):
        n = pre[r + 1] - pre[r]
        if n <= 1:
            continue
        for s in range(s_q):
            for hh in range(h):
                ro, rl = ocomb.combine(l_acc[pre[r]:pre[r + 1], s, hh].double().numpy(),
                                       o_acc[pre[r]:pre[r + 1], s, hh].double().numpy())
                assert np.max(np.abs(out[r, s, hh] - ro)) <= 1e-2 * max(1, np.abs(ro).max())
                assert abs(lse[r, hh, s] - rl) <= 1e-4
                checked += 1
    assert checked >= 2 * 128


# ----------------------------------------------------------------------------- extra_kv

def _extra_inputs(wl, extra_topk, ctx, seed, masked=0, out_of_range=0):
    """A second cache (its own pool) and index list for the tokens of ``wl``; some slots are
    masked and slots 3.. hold ids just past the extra pool (which must be masked, not read
    from any other pool)."""
    wx = workloads.small(b=wl.spec.b, s_q=wl.spec.s_q, h_q=wl.spec.h_q, topk=extra_topk,
                         ctx=ctx, masked_per_row=masked, seed=seed, device=wl.q.device)
    eidx = wx.indices.clone()
    if out_of_range:
        erows = wx.kv.shape[0] * 64
        eidx[..., 3:3 + out_of_range] = erows + torch.arange(out_of_range, device=eidx.device,
                                                             dtype=eidx.dtype)
    return wx.kv.contiguous(), eidx.contiguous()


EXTRA_CASES = [
    # (name, main workload kwargs, extra_topk, num_sms, with lengths, with sink)
    ("extra_nosplit_h128", dict(b=3, h_q=128, topk=200, ctx=2048, masked_per_row=10), 130, 8,
     False, False),
    ("extra_split_h128_lens_sink", dict(b=2, h_q=128, topk=256, ctx=2048), 192, 132, True,
     True),
    ("extra_split_h64_sq2", dict(b=2, s_q=2, h_q=64, topk=100, ctx=1024, causal_base=700), 77,
     48, True, False),
    ("extra_only_topk0", dict(b=3, h_q=128, topk=0, ctx=512), 150, 24, False, True),
    ("extra_ragged_main", dict(b=4, h_q=128, topk=65, ctx=1024, ue8m0=True), 63, 20, True,
     False),
]


@pytest.mark.parametrize("name,kw,extra_topk,num_sms,use_len,use_sink", EXTRA_CASES,
                         ids=[c[0] for c in EXTRA_CASES])
def test_extra_kv_parity(dev, name, kw, extra_topk, num_sms, use_len, use_sink):
    seed = 1300 + sum(map(ord, name))
    wl = workloads.small(device=dev, seed=seed, **kw)
    ekv, eidx = _extra_inputs(wl, extra_topk, ctx=768, seed=seed + 1, masked=7, out_of_range=3)
    lens = elens = sink = None
    if use_len:
        lens = workloads.topk_lengths(wl.spec.b, wl.spec.s_q, max(wl.spec.topk, 1), seed, device=dev)
        elens = workloads.topk_lengths(wl.spec.b, wl.spec.s_q, extra_topk, seed + 2, device=dev)
    if use_sink:
        sink = workloads.attn_sink(wl.spec.h_q, seed, device=dev)
    out, lse, _ = gu.run_cuda(wl, num_sms=num_sms, attn_sink=sink, topk_length=lens,
                              extra_kv=ekv, extra_indices=eidx, extra_topk_length=elens)
    q, kv, idx = workloads.to_numpy_inputs(wl)
    ro, rl = oracle.sparse_mla_decode_full(
        q, kv, idx, wl.sm_scale,
        attn_sink=None if sink is None else sink.double().cpu().numpy(),
        topk_length=None if lens is None else lens.cpu().numpy(),
        extra_kv=ekv.cpu().numpy().reshape(-1, 64, 656), extra_indices=eidx.cpu().numpy(),
        extra_topk_length=None if elens is None else elens.cpu().numpy())
    h = wl.spec.h_q
    go = out.double().cpu().numpy().reshape(-1, h, 512)
    gl = lse.double().cpu().numpy().transpose(0, 2, 1).reshape(-1, h)
    print(name, gu.compare(go, gl, ro.reshape(-1, h, 512), rl.transpose(0, 2, 1).reshape(-1, h),
                           name))
    if wl.spec.topk > 0:  # the extra list changed the result
        plain, _, _ = gu.run_cuda(wl, num_sms=num_sms, attn_sink=sink, topk_length=lens)
        assert np.abs(go - plain.double().cpu().numpy().reshape(go.shape)).max() > 2 * gu.O_MAX_ABS


def test_full_size_workload_with_extra_kv(dev):
    spec = workloads.CONFIGS["c2_b64_h128_k2048_mask5"]
    wl = workloads.make(spec, device=dev)
    ekv, eidx = _extra_inputs(wl, 512, ctx=4096, seed=991, masked=20, out_of_range=2)
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out, lse, _ = gu.run_cuda(wl, num_sms=num_sms, extra_kv=ekv, extra_indices=eidx)
    tokens = np.arange(spec.b * spec.s_q)  # every query token
    ro, rl = gu.oracle_tokens_extra(wl, tokens, ekv, eidx)
    go, gl = gu.gpu_tokens(out, lse, wl, tokens)
    print(gu.compare(go, gl, ro, rl, "c2 with a 512-slot extra list"))
