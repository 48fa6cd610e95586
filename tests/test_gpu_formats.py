"""GPU parity of the later KV-cache formats (V4, V4.1, and FP4 as the extra cache of a V4.1
cache; d_qk = d_v = 512, structure-of-arrays pages) against the format oracle, through the C
ABI: unsplit, several-requests and split plans, h_q 64 and 128, masked and out-of-range slots,
per-token lengths, the attention sink, a NaN scale, and a decode-shaped workload at full size
on sampled tokens."""

import numpy as np
import pytest
import torch

import sparse_mla_attention_decode_gb300 as smla
import workloads
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(cuda_ok):
    smla.lib()
    return torch.device("cuda:0")


def _check(wl, num_sms, what, tokens=None, **kw):
    ext = {k: v for k, v in kw.items() if k in ("extra_kv", "extra_indices", "extra_topk_length")}
    out, lse, op = gu.run_cuda(wl, num_sms=num_sms, check_status=True, **kw)
    n = wl.spec.b * wl.spec.s_q
    toks = np.arange(n) if tokens is None else np.asarray(tokens)
    og, lg = gu.gpu_tokens(out, lse, wl, toks)
    orf, lrf = gu.oracle_tokens_fmt(wl, toks, attn_sink=kw.get("attn_sink"),
                                    topk_length=kw.get("topk_length"), **ext)
    return gu.compare(og, lg, orf, lrf, what)


CASES = [  # (b, s_q, h_q, topk, ctx, masked, num_sms)
    (2, 1, 128, 128, 512, 0, 152),
    (3, 2, 128, 200, 1024, 7, 4),      # several requests per partition, ragged tail
    (3, 2, 64, 200, 1024, 5, 4),       # the same at h_q = 64 (Q stays in one key-tile stage)
    (2, 1, 64, 300, 2048, 5, 152),     # h_q = 64, requests split over partitions
    (4, 1, 128, 17, 256, 0, 8),        # one short block
    (2, 2, 128, 2048, 8192, 100, 152), # split, full-length list
]


@pytest.mark.parametrize("fmt", ["v41", "v4"])
@pytest.mark.parametrize("case", CASES)
def test_formats_small(dev, fmt, case):
    b, s_q, h, topk, ctx, masked, nsm = case
    wl = workloads.small(b=b, s_q=s_q, h_q=h, topk=topk, ctx=ctx, masked_per_row=masked,
                         seed=71 + topk, device=dev, kv_format=fmt)
    if masked:
        wl.indices.view(-1)[3] = wl.kv.shape[0] * 64 + 5   # beyond the pool: masked too
    m = _check(wl, nsm, f"{fmt} {case}")
    print("FMT", fmt, case, m)


@pytest.mark.parametrize("fmt", ["v41", "v4"])
def test_formats_variants(dev, fmt):
    wl = workloads.small(b=4, s_q=2, h_q=128, topk=300, ctx=2048, masked_per_row=3, seed=81,
                         device=dev, kv_format=fmt)
    lens = workloads.topk_lengths(4, 2, 300, seed=3, device=dev)
    sink = workloads.attn_sink(128, seed=4, device=dev)
    _check(wl, 152, f"{fmt} lengths", topk_length=lens)
    _check(wl, 6, f"{fmt} lengths, several requests", topk_length=lens)
    _check(wl, 152, f"{fmt} sink", attn_sink=sink)


def _fp4_extra(b, s_q, etopk, epages, seed, dev):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(epages * 64, 512, generator=g).to(torch.bfloat16)
    data, sc = workloads.quantize_fmt(x, "v41_fp4")
    pool = torch.empty(epages, 64 * 288, dtype=torch.uint8)
    pool[:, : 64 * 256] = data.view(epages, -1)
    pool[:, 64 * 256:] = sc.view(epages, -1)
    eidx = torch.randint(0, epages * 64, (b, s_q, etopk), generator=g, dtype=torch.int32)
    eidx.view(-1)[::11] = -1
    return pool.to(dev), eidx.to(dev)


@pytest.mark.parametrize("nsm", [152, 4])
def test_v41_with_fp4_extra(dev, nsm):
    wl = workloads.small(b=3, s_q=2, h_q=128, topk=150, ctx=1024, masked_per_row=4, seed=91,
                         device=dev, kv_format="v41")
    ekv, eidx = _fp4_extra(3, 2, 96, 6, seed=5, dev=dev)
    _check(wl, nsm, f"v41 + fp4 extra ({nsm} SMs)", extra_kv=ekv, extra_indices=eidx)
    elen = torch.tensor([[5, 96], [0, 64], [65, 200]], dtype=torch.int32, device=dev)
    _check(wl, nsm, "v41 + fp4 extra, lengths", extra_kv=ekv, extra_indices=eidx,
           extra_topk_length=elen)


def test_nan_scale_propagates(dev):
    wl = workloads.small(b=3, s_q=1, h_q=128, topk=128, ctx=512, seed=95, device=dev,
                         kv_format="v41")
    j = int(wl.indices[2, 0, 70].item())
    page, off = divmod(j, 64)
    wl.kv[page, 64 * 512 + off * 16 + 3] = 0xFF  # e8m0 NaN: dims 96..127 of that token
    out, lse, op = gu.run_cuda(wl, num_sms=152, check_status=False)
    assert op.device_status() & smla.SMLA_DEV_NAN_INPUT
    og, lg = gu.gpu_tokens(out, lse, wl, np.arange(3))
    orf, lrf = gu.oracle_tokens_fmt(wl, np.arange(3))
    nan = np.isnan(orf).any(-1)
    assert nan[2].all() and np.array_equal(np.isnan(og).all(-1), nan)
    gu.compare(og[~nan], lg[~nan], orf[~nan], lrf[~nan], "v41 NaN scale, other tokens")


def test_v41_decode_shape_full_size(dev):
    # the decode-shaped workload (b = 64, topk = 2048 of 32768 tokens, 5 % masked) in V4.1
    spec = workloads.Spec("c2_v41", b=64, s_q=1, h_q=128, topk=2048, ctx=32768,
                          masked_per_row=102, seed=1, kv_format="v41")
    wl = workloads.make(spec, device=dev)
    toks = np.arange(0, 64, 7)
    m = _check(wl, 0, "c2-shaped v41", tokens=toks)
    print("FMT full c2-shaped v41", m)
