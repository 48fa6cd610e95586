"""GPU parity of the exact top-k with the page-table emit (sparse_mla_topk_page_table) against
the full-sort oracle: every output row is checked for what is unique (all positions scoring
above the k-th largest value are selected) and for validity (no duplicate, selected positions
inside the valid prefix and at least the k-th value, -1 after the selected ids).  bf16 and
fp32 scores, ragged and degenerate lengths, tie-heavy rows that overflow the candidate list,
signed zeros and infinities, the workload shapes, and the selection feeding the attention."""

import numpy as np
import pytest
import torch

import oracle
import sparse_mla_attention_decode_gb300 as smla
import workloads
from oracle import topk as otk
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(cuda_ok):
    smla.lib()
    return torch.device("cuda:0")


def _table(b, pages, seed, dev):
    g = torch.Generator().manual_seed(seed)
    return torch.stack([torch.randperm(pages * 4, generator=g)[:pages] for _ in range(b)]).to(
        torch.int32).to(dev)


def _check(out, scores, lens, table, s_q, k, rows=None):
    out = out.cpu().numpy()
    sc = scores.float().cpu().numpy().astype(np.float64)
    tb = table.cpu().numpy()
    ln = lens.cpu().numpy()
    for t in (range(out.shape[0]) if rows is None else rows):
        otk.check_row(out[t], sc[t], int(ln[t]), k, tb[t // s_q])


# up to 76 rows (half the SMs) an fp32 row runs on a pair of CTAs, above that on one CTA (bf16
# rows always on one): n_tok 12 and 96 take the two kernels
@pytest.mark.parametrize("n_tok", [12, 96])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("ld,k", [(4096, 2048), (1000, 64), (24576, 2048), (64, 64)])
def test_topk_parity(dev, dtype, ld, k, n_tok):
    s_q = 3
    scores = workloads.index_scores(n_tok, ld, dtype, seed=ld + k, device=dev)
    edge = [0, 1, k - 1, k, k + 1, ld, ld + 5, -3]
    g = torch.Generator().manual_seed(k)
    lens = torch.tensor(edge + torch.randint(0, ld + 1, (n_tok - len(edge),), generator=g).tolist(),
                        dtype=torch.int32)[:n_tok].to(dev)
    table = _table(n_tok // s_q, (ld + 63) // 64, seed=ld, dev=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = smla.topk_page_table(scores, lens, table, s_q, k, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _check(out, scores, lens, table, s_q, k)


@pytest.mark.parametrize("n_tok", [4, 96])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("levels", [1, 3, 40])
def test_topk_tie_heavy_rows(dev, dtype, levels, n_tok):
    # few distinct values: the threshold bin holds far more than the candidate list (8192)
    ld, k = 40000, 2048
    scores = workloads.index_scores(n_tok, ld, dtype, seed=levels, device=dev, levels=levels)
    lens = torch.tensor([ld, ld - 7, 30000, 9000] * (n_tok // 4), dtype=torch.int32, device=dev)
    table = _table(n_tok, (ld + 63) // 64, seed=1, dev=dev)
    out = smla.topk_page_table(scores, lens, table, 1, k)
    torch.cuda.synchronize()
    _check(out, scores, lens, table, 1, k)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_topk_signed_zero_and_infinities(dev, dtype):
    n_tok, ld, k = 3, 5000, 100
    g = torch.Generator().manual_seed(2)
    base = torch.randn(n_tok, ld, generator=g)
    base[0] = torch.where(torch.rand(ld, generator=g) < 0.5, torch.tensor(0.0), torch.tensor(-0.0))
    base[0, :37] = 1.0
    base[1, ::7] = float("inf")
    base[1, 1::5] = float("-inf")
    base[2] = -torch.rand(ld, generator=g) - 1.0  # all negative
    scores = base.to(dtype).to(dev)
    lens = torch.full((n_tok,), ld, dtype=torch.int32, device=dev)
    table = _table(n_tok, (ld + 63) // 64, seed=3, dev=dev)
    out = smla.topk_page_table(scores, lens, table, 1, k)
    torch.cuda.synchronize()
    _check(out, scores, lens, table, 1, k)


@pytest.mark.parametrize("n_tok", [4, 96])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("shift,k", [(-5.0, 2048), (0.0, 12288), (0.0, 19661), (3.0, 100)])
def test_topk_boundary_sign(dev, dtype, shift, k, n_tok):
    # where the sampled boundary falls decides how the full pass tests a candidate: on its raw
    # bits when the boundary is non-negative, on its key otherwise.  All-negative rows, a
    # boundary near zero (half the row selected), one below zero (80 %) and a high one.
    ld = 24576
    g = torch.Generator().manual_seed(int(k + 10 * shift))
    base = torch.randn(n_tok, ld, generator=g) + shift
    base[:, ::97] = 0.0
    base[:, 1::89] = -0.0
    scores = base.to(dtype).to(dev)
    lens = torch.tensor([ld, ld - 3, k + 1000, ld // 2 + 17] * (n_tok // 4), dtype=torch.int32,
                        device=dev)
    table = _table(n_tok, ld // 64, seed=9, dev=dev)
    out = smla.topk_page_table(scores, lens, table, 1, k)
    torch.cuda.synchronize()
    _check(out, scores, lens, table, 1, k)


def test_topk_strided_rows_and_table_flag(dev):
    n_tok, ld, k = 4, 8192, 512
    big = workloads.index_scores(n_tok, ld + 64, torch.bfloat16, seed=5, device=dev)
    scores = big[:, :ld]  # a row stride above the row length
    lens = torch.tensor([ld, 7000, 600, 513], dtype=torch.int32, device=dev)
    table = _table(n_tok, ld // 64, seed=6, dev=dev)
    out = smla.topk_page_table(scores, lens, table, 1, k)
    torch.cuda.synchronize()
    _check(out, scores, lens, table, 1, k)
    # a page table too short for the valid prefix: the flag is raised, no fault
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    short = table[:, :4].contiguous()
    smla.topk_page_table(scores, lens, short, 1, k, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & smla.SMLA_DEV_TOPK_TABLE


@pytest.mark.parametrize("cfg", ["c2_b64_h128_k2048_mask5", "c4_b32_h128_k2048_ue8m0_perm",
                                 "c3_b128_sq2_h64_k2048", "c5_b1_sq4096_h128_k2048"])
def test_topk_workload_shapes(dev, cfg):
    spec = workloads.CONFIGS[cfg]
    n_tok = spec.b * spec.s_q
    scores = workloads.index_scores(n_tok, spec.ctx, torch.bfloat16, seed=spec.seed, device=dev)
    if spec.causal_base is not None:
        lens = (spec.causal_base + 1 + torch.arange(n_tok) % spec.s_q).clamp(max=spec.ctx)
    else:
        lens = torch.full((n_tok,), spec.ctx)
    lens = lens.to(torch.int32).to(dev)
    table = _table(spec.b, spec.pages_per_seq, seed=spec.seed, dev=dev)
    out = smla.topk_page_table(scores, lens, table, spec.s_q, spec.topk)
    torch.cuda.synchronize()
    rows = sorted(set([0, n_tok - 1] + list(np.random.default_rng(1).integers(0, n_tok, 10))))
    _check(out, scores, lens, table, spec.s_q, spec.topk, rows=rows)


def test_topk_feeds_the_attention(dev):
    # fp32 scores (no ties at the threshold): the selected set is unique, so the attention
    # over the GPU's selection equals the oracle's attention over the oracle's selection
    wl = workloads.small(b=3, h_q=128, topk=256, ctx=2048, device=dev, seed=40)
    n_tok = wl.spec.b
    scores = workloads.index_scores(n_tok, wl.spec.ctx, torch.float32, seed=41, device=dev)
    lens = torch.tensor([2048, 1500, 200], dtype=torch.int32, device=dev)
    idx = smla.topk_page_table(scores, lens, wl.block_table.contiguous(), 1, 256)
    wl.indices = idx.view(n_tok, 1, 256).contiguous()
    out, lse, _ = gu.run_cuda(wl, num_sms=16)
    ref_idx, _ = otk.topk_page_table(scores.cpu().double().numpy(), lens.cpu().numpy(),
                                     wl.block_table.cpu().numpy(), 1, 256)
    q, kv, _ = workloads.to_numpy_inputs(wl)
    ro, rl = oracle.sparse_mla_decode_full(q, kv, ref_idx.reshape(n_tok, 1, 256), wl.sm_scale)
    h = wl.spec.h_q
    gu.compare(out.double().cpu().numpy().reshape(-1, h, 512),
               lse.double().cpu().numpy().transpose(0, 2, 1).reshape(-1, h),
               ro.reshape(-1, h, 512), rl.transpose(0, 2, 1).reshape(-1, h), "top-k -> attention")
