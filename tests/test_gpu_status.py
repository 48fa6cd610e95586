"""The device status word reports inputs outside the fp16 range the kernel computes in: a query
value that would overflow fp16 (from the first and from a later request of a partition), and
a KV scale whose product with 256 leaves the fp16 normal range.  Clean inputs give 0; the
largest scale in range does not trip the scale check.  (Valid inputs only: nothing here can fault.)"""

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


def _status(wl, num_sms):
    _, _, op = gu.run_cuda(wl, num_sms=num_sms, check_status=False)
    return op.device_status()


@pytest.mark.parametrize("num_sms", [4, 152])  # several requests per partition / one each
def test_query_range_flag(dev, num_sms):
    wl = workloads.small(b=6, h_q=128, topk=128, ctx=1024, device=dev, seed=31)
    assert _status(wl, num_sms) == 0
    q0 = wl.q.clone()
    for bi, h, d, v in ((5, 17, 3, 70000.0), (0, 100, 560, -70000.0), (3, 0, 0, float("nan"))):
        wl.q = q0.clone()
        wl.q[bi, 0, h, d] = v
        assert _status(wl, num_sms) & smla.SMLA_DEV_Q_RANGE, (bi, h, d, v)
    wl.q = q0.clone()
    wl.q[5, 0, 17, 3] = 65280.0  # the largest bf16 value that is finite in fp16
    wl.q[0, 0, 3, 511] = -65280.0
    assert _status(wl, num_sms) == 0


def test_query_range_flag_h64_unused_rows(dev):
    # h_q = 64: the tensor-memory rows 64-127 are unused and must not raise the flag
    wl = workloads.small(b=2, h_q=64, topk=96, ctx=512, device=dev, seed=32)
    assert _status(wl, 16) == 0
    wl.q[1, 0, 63, 575] = 1.0e5
    assert _status(wl, 16) & smla.SMLA_DEV_Q_RANGE


def test_scale_range_flag(dev):
    wl = workloads.small(b=2, h_q=128, topk=64, ctx=512, device=dev, seed=33)
    assert _status(wl, 8) == 0
    kv0 = wl.kv.clone()
    row = int(wl.indices[1, 0, 5].item())
    for scale in (300.0, 1e-8):
        wl.kv = kv0.clone()
        flat = wl.kv.view(-1, 656)
        flat[row, 512 + 4:512 + 8] = torch.tensor([scale], dtype=torch.float32).view(torch.uint8).to(dev)
        assert _status(wl, 8) & smla.SMLA_DEV_SCALE_RANGE, scale
    # the largest scale the fp16 path takes (255 * 256 = 65280) is not a scale-range error;
    # with large codes in that group the products themselves overflow fp16, which the
    # non-finite-score bit reports instead
    wl.kv = kv0.clone()
    flat = wl.kv.view(-1, 656)
    flat[row, 512:516] = torch.tensor([255.0], dtype=torch.float32).view(torch.uint8).to(dev)
    assert not _status(wl, 8) & smla.SMLA_DEV_SCALE_RANGE
    # and with codes small enough (|code| <= 1) the key stays finite: the word is clean
    flat[row, 0:128] = torch.tensor([0x38, 0xB8], dtype=torch.uint8, device=dev).repeat(64)
    assert _status(wl, 8) == 0
