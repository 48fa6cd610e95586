"""GPU parity of the indexer scores (sparse_mla_indexer_scores: e4m3 x e4m3 tensor-core MMAs,
ReLU and the weighted 64-head sum in the epilogue) against the fp64 oracle, and the whole
selection pipeline: indexer scores -> exact top-k with the page-table emit -> sparse
attention, against the same three steps in the oracle."""

import numpy as np
import pytest
import torch

import oracle
import sparse_mla_attention_decode_gb300 as smla
import workloads
from oracle import indexer as oix
from oracle import topk as otk
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(cuda_ok):
    smla.lib()
    return torch.device("cuda:0")


def _compare(got, ref, lens, ld):
    got = got.double().cpu().numpy()
    for t in range(ref.shape[0]):
        n = min(int(lens[t]), ld)
        g, r = got[t, :n], ref[t, :n]
        tol = 2e-5 * max(1.0, float(np.abs(r).max(initial=0.0))) + 1e-6
        err = float(np.abs(g - r).max(initial=0.0))
        assert err <= tol, (t, err, tol)


@pytest.mark.parametrize("s_q", [1, 2, 3, 4, 5])
def test_indexer_parity(dev, s_q):
    b, pages, ld = 3, 40, 2560
    n_tok = b * s_q
    cache = workloads.indexer_cache(pages * 2, seed=10 + s_q, device=dev)
    q8, w = workloads.indexer_queries(n_tok, seed=20 + s_q, device=dev)
    g = torch.Generator().manual_seed(s_q)
    table = torch.stack([torch.randperm(pages * 2, generator=g)[:pages] for _ in range(b)]).to(torch.int32).to(dev)
    edge = [0, 1, 63, 64, 65, 127, 128, 129, 2048, 2560, 2999]
    lens = torch.tensor((edge * 3)[:n_tok], dtype=torch.int32).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = smla.indexer_scores(q8, w, cache, table, lens, s_q, ld, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oix.indexer_scores(q8.cpu().numpy(), w.cpu().double().numpy(), cache.cpu().numpy(),
                             table.cpu().numpy(), lens.cpu().numpy(), s_q, ld)
    _compare(out, ref, lens.cpu().numpy(), ld)


def test_indexer_bad_page_ids_score_zero(dev):
    pages, ld = 8, 512
    cache = workloads.indexer_cache(pages, seed=3, device=dev)
    q8, w = workloads.indexer_queries(1, seed=4, device=dev)
    table = torch.tensor([[2, 9999, 5, -3, 1, 0, 7, 6]], dtype=torch.int32, device=dev)
    lens = torch.tensor([300], dtype=torch.int32, device=dev)
    out = smla.indexer_scores(q8, w, cache, table, lens, 1, ld)
    torch.cuda.synchronize()
    o = out.cpu().numpy()[0]
    assert np.all(o[64:128] == 0.0) and np.all(o[192:256] == 0.0)  # pages outside the cache
    good = table.clone()
    good[0, 1], good[0, 3] = 3, 4
    ref = oix.indexer_scores(q8.cpu().numpy(), w.cpu().double().numpy(), cache.cpu().numpy(),
                             good.cpu().numpy(), [300], 1, ld)
    ok = np.r_[0:64, 128:192, 256:300]
    assert np.allclose(o[ok], ref[0, ok], rtol=1e-4, atol=1e-5)


def test_indexer_decode_workload_shape(dev):
    # b = 64 requests, one query token each, 32768 cached tokens (512 pages) per request
    b, pages, ld = 64, 512, 32768
    cache = workloads.indexer_cache(b * pages, seed=5, device=dev)
    q8, w = workloads.indexer_queries(b, seed=6, device=dev)
    table = torch.randperm(b * pages, generator=torch.Generator().manual_seed(7)).to(torch.int32).view(b, pages).to(dev)
    lens = torch.full((b,), ld, dtype=torch.int32, device=dev)
    lens[5] = 1000
    out = smla.indexer_scores(q8, w, cache, table, lens, 1, ld)
    torch.cuda.synchronize()
    rows = [0, 5, 31, 63]
    ref = oix.indexer_scores(q8[rows].cpu().numpy(), w[rows].cpu().double().numpy(),
                             cache.cpu().numpy(), table[rows].cpu().numpy(),
                             lens[rows].cpu().numpy(), 1, ld)
    _compare(out[rows], ref, lens[rows].cpu().numpy(), ld)


def test_indexer_topk_attention_pipeline(dev):
    # scores -> top-k -> attention on the GPU against the same three steps in the oracle; the
    # scores are continuous (fp32 weights and scales), so the selected sets are unique
    wl = workloads.small(b=3, s_q=2, h_q=128, topk=256, ctx=2048, device=dev, seed=70,
                         causal_base=1500)
    b, s_q = wl.spec.b, wl.spec.s_q
    n_tok = b * s_q
    pages = wl.block_table.shape[1]
    num_pages = wl.kv.shape[0]
    cache = workloads.indexer_cache(num_pages, seed=71, device=dev)  # one indexer page per KV page
    q8, w = workloads.indexer_queries(n_tok, seed=72, device=dev)
    table = wl.block_table.contiguous()
    lens = (1501 + torch.arange(n_tok, device=dev) % s_q).to(torch.int32)
    scores = smla.indexer_scores(q8, w, cache, table, lens, s_q, wl.spec.ctx)
    idx = smla.topk_page_table(scores, lens, table, s_q, 256)
    wl.indices = idx.view(b, s_q, 256).contiguous()
    out, lse, _ = gu.run_cuda(wl, num_sms=24)
    # each step against the oracle on the step's own GPU input: the scores within tolerance,
    # the selection exactly (on the GPU's fp32 scores, whose ties do not occur here), and the
    # attention over the selection
    rs = oix.indexer_scores(q8.cpu().numpy(), w.cpu().double().numpy(), cache.cpu().numpy(),
                            table.cpu().numpy(), lens.cpu().numpy(), s_q, wl.spec.ctx)
    _compare(scores, rs, lens.cpu().numpy(), wl.spec.ctx)
    gs = scores.double().cpu().numpy()
    ridx, _ = otk.topk_page_table(gs, lens.cpu().numpy(), table.cpu().numpy(), s_q, 256)
    got_sets = [set(r) for r in idx.cpu().numpy().tolist()]
    want_sets = [set(r) for r in ridx.tolist()]
    assert got_sets == want_sets
    q, kv, _ = workloads.to_numpy_inputs(wl)
    ro, rl = oracle.sparse_mla_decode_full(q, kv, ridx.reshape(b, s_q, 256), wl.sm_scale)
    h = wl.spec.h_q
    gu.compare(out.double().cpu().numpy().reshape(-1, h, 512),
               lse.double().cpu().numpy().transpose(0, 2, 1).reshape(-1, h),
               ro.reshape(-1, h, 512), rl.transpose(0, 2, 1).reshape(-1, h), "indexer pipeline")
