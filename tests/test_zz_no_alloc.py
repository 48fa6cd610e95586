"""sparse_mla_decode_static: the decode on the library's fixed scratch gives the results of
the three-call sequence on caller buffers, call after call, and rejects problems that do not
fit its scratch before launching anything."""

import numpy as np
import pytest

import sparse_mla_attention_decode_gb300 as smla
import workloads
from tests.gpu_util import compare, gpu_tokens


def _static_run(wl, num_sms):
    import torch
    d = smla.dims_for(wl.spec.b, wl.spec.s_q, wl.spec.h_q, wl.spec.topk, wl.kv.shape[0])
    out = torch.empty(wl.spec.b, wl.spec.s_q, wl.spec.h_q, 512, dtype=torch.bfloat16,
                      device=wl.q.device)
    lse = torch.empty(wl.spec.b, wl.spec.h_q, wl.spec.s_q, dtype=torch.float32, device=wl.q.device)
    out.fill_(7.0)  # stale values must all be overwritten
    lse.fill_(-3.0)
    st = torch.cuda.current_stream(wl.q.device).cuda_stream
    smla.sparse_mla_decode_static(d, num_sms, wl.q.data_ptr(), wl.kv.data_ptr(),
                                  wl.indices.data_ptr(), wl.sm_scale, out.data_ptr(),
                                  lse.data_ptr(), st)
    return out, lse


def _check_same(wl, out_s, lse_s, out_r, lse_r, what):
    tokens = np.arange(wl.spec.b * wl.spec.s_q)
    o_s, l_s = gpu_tokens(out_s, lse_s, wl, tokens)
    o_r, l_r = gpu_tokens(out_r, lse_r, wl, tokens)
    compare(o_s, l_s, o_r, l_r, what)


def test_static_rejects_problem_above_scratch():
    # b = 1, s_q = 4096, h_q = 128: two splits x 4096 x 128 x 512 fp32 partials = 2 GiB
    d = smla.dims_for(1, 4096, 128, 2048, 1024)
    with pytest.raises(smla.SparseMLAError) as e:
        smla.sparse_mla_decode_static(d, 152, 16, 16, 16, 0.04, 16, 16, 0)
    assert e.value.code == smla.SMLA_ERR_WORKSPACE
    assert str(smla.STATIC_SCRATCH_BYTES) in str(e.value)


@pytest.mark.gpu
@pytest.mark.parametrize("case", [
    dict(b=6, s_q=1, h_q=128, topk=448, ctx=4096, masked_per_row=40, seed=21),
    dict(b=3, s_q=2, h_q=64, topk=200, ctx=2048, ue8m0=True, seed=22),
])
def test_static_matches_three_call_sequence(cuda_ok, case):
    import torch
    dev = torch.device("cuda:0")
    nsm = 16  # several partitions per request: split rows and the combine are exercised
    wl_a = workloads.small(device=dev, **case)
    wl_b = workloads.small(device=dev, **{**case, "seed": case["seed"] + 100})
    ref = {}
    for name, wl in (("a", wl_a), ("b", wl_b)):
        op = smla.SparseMLADecode(wl.spec.b, wl.spec.s_q, wl.spec.h_q, wl.spec.topk,
                                  wl.kv.shape[0], device=dev, num_sms=nsm)
        ref[name] = op.run(wl.q, wl.kv, wl.indices, wl.sm_scale)
    # two calls in a row on the same scratch, with different inputs
    out1, lse1 = _static_run(wl_a, nsm)
    out2, lse2 = _static_run(wl_b, nsm)
    torch.cuda.synchronize(dev)
    _check_same(wl_a, out1, lse1, *ref["a"], "first static call")
    _check_same(wl_b, out2, lse2, *ref["b"], "second static call")


@pytest.mark.gpu
def test_static_matches_on_full_size_workload(cuda_ok):
    import torch
    dev = torch.device("cuda:0")
    wl = workloads.make(workloads.CONFIGS["c2_b64_h128_k2048_mask5"], device=dev)
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    op = smla.SparseMLADecode(wl.spec.b, wl.spec.s_q, wl.spec.h_q, wl.spec.topk,
                              wl.kv.shape[0], device=dev, num_sms=nsm)
    out_r, lse_r = op.run(wl.q, wl.kv, wl.indices, wl.sm_scale)
    for call in range(2):
        out_s, lse_s = _static_run(wl, nsm)
        torch.cuda.synchronize(dev)
        _check_same(wl, out_s, lse_s, out_r, lse_r, f"static call {call}")
