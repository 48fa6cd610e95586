"""Non-finite values in valid key rows follow the definition, as the oracle computes it: a NaN
e4m3 code or a NaN bf16 RoPE value in a row that a token selects makes every head of that token
NaN (out and lse); a bf16 +inf in RoPE makes the heads whose query is positive there NaN and
drops the slot for the others (a -inf score adds exp(-inf) = 0).  The CUDA path must give the
same NaN pattern, the oracle's values elsewhere and SMLA_DEV_NAN_INPUT in the status word, on
the unsplit path and through the split partials and the combine.  (Inputs only: a NaN input
is an ordinary value for every instruction on the path; nothing here can fault.)"""

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


def _check(wl, num_sms, what):
    out, lse, op = gu.run_cuda(wl, num_sms=num_sms, check_status=False)
    word = op.device_status()
    n_tok = wl.spec.b * wl.spec.s_q
    toks = np.arange(n_tok)
    o_gpu, l_gpu = gu.gpu_tokens(out, lse, wl, toks)
    o_ref, l_ref = gu.oracle_tokens(wl, toks)
    nan_ref = np.isnan(o_ref).any(-1)  # [tok, h]: a NaN row of the oracle is NaN throughout
    assert np.array_equal(np.isnan(o_ref).all(-1), nan_ref)
    assert nan_ref.any(), what
    assert np.array_equal(np.isnan(o_gpu).all(-1), nan_ref), what
    assert np.array_equal(np.isnan(o_gpu).any(-1), nan_ref), what
    assert np.array_equal(np.isnan(l_gpu), np.isnan(l_ref)), what
    assert np.array_equal(np.isnan(l_ref), nan_ref), what
    fin = ~nan_ref
    gu.compare(o_gpu[fin], l_gpu[fin], o_ref[fin], l_ref[fin], what)
    assert word & smla.SMLA_DEV_NAN_INPUT, (what, word)
    return nan_ref


# (b, topk, ctx, num_sms): several requests per partition, one partition per request, and
# requests split over many partitions (partials + combine)
CASES = [(6, 192, 1024, 4), (6, 192, 1024, 152), (2, 1024, 4096, 152)]


@pytest.mark.parametrize("b,topk,ctx,num_sms", CASES)
def test_nan_code_in_a_valid_row(dev, b, topk, ctx, num_sms):
    wl = workloads.small(b=b, h_q=128, topk=topk, ctx=ctx, device=dev, seed=61)
    assert gu.run_cuda(wl, num_sms=num_sms, check_status=False)[2].device_status() == 0
    flat = wl.kv.view(-1, 656)
    row = int(wl.indices[b - 1, 0, topk - 5].item())  # the last block of the last request
    flat[row, 300] = 0x7F  # e4m3 NaN (S.1111.111)
    nan = _check(wl, num_sms, "e4m3 NaN")
    assert nan[b - 1].all()


@pytest.mark.parametrize("b,topk,ctx,num_sms", CASES)
def test_nan_and_inf_rope_in_a_valid_row(dev, b, topk, ctx, num_sms):
    wl = workloads.small(b=b, h_q=128, topk=topk, ctx=ctx, device=dev, seed=62)
    flat = wl.kv.view(-1, 656)
    kv0 = wl.kv.clone()
    row = int(wl.indices[0, 0, 70].item())  # second block of the first request
    flat[row, 528 + 2 * 9] = 0xC0  # bf16 NaN 0x7FC0 in RoPE dim 9
    flat[row, 529 + 2 * 9] = 0x7F
    nan = _check(wl, num_sms, "bf16 NaN")
    assert nan[0].all()
    wl.kv = kv0.clone()
    flat = wl.kv.view(-1, 656)
    flat[row, 528 + 2 * 9] = 0x80  # bf16 +inf 0x7F80
    flat[row, 529 + 2 * 9] = 0x7F
    nan = _check(wl, num_sms, "bf16 +inf")
    qd = wl.q[0, 0, :, 512 + 9].float().cpu().numpy()
    assert np.array_equal(nan[0], qd >= 0)  # +inf (or 0 * inf) only where q is not negative
