"""sparse_mla_decode_static: the decode on the library's fixed scratch gives the results of
the three-call sequence on caller buffers, call after call (and after a device reset), its
device status word reads back clean, and it rejects problems that do not fit its scratch
before launching anything."""

import os
import subprocess
import sys

import numpy as np
import pytest

import sparse_mla_attention_decode_gb300 as smla
import workloads
from tests.gpu_util import compare, gpu_tokens


def _static_run(wl, num_sms):
    import torch
    d = smla.dims_for(wl.spec.b, wl.spec.s_q, wl.spec.h_q, wl.spec.topk, wl.kv.shape[0],
                      kv_format=wl.spec.kv_format)
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


def _dims(wl):
    return smla.dims_for(wl.spec.b, wl.spec.s_q, wl.spec.h_q, wl.spec.topk, wl.kv.shape[0])


def _check_same(wl, out_s, lse_s, out_r, lse_r, what):
    tokens = np.arange(wl.spec.b * wl.spec.s_q)
    o_s, l_s = gpu_tokens(out_s, lse_s, wl, tokens)
    o_r, l_r = gpu_tokens(out_r, lse_r, wl, tokens)
    compare(o_s, l_s, o_r, l_r, what)


def test_static_rejects_problem_above_scratch():
    # b = 64, s_q = 8, h_q = 128 on 152 SMs: 9 partitions per position split 8 requests, and
    # the split partials of 71 slots x 8 positions x 128 heads x 512 fp32 exceed 48 MiB.  The
    # pointers are null: if the size check ever let this through, the decode call would reject
    # them before launching anything (only the planner would have run, on the scratch itself).
    d = smla.dims_for(64, 8, 128, 2048, 1024)
    sb, ab = smla.sparse_mla_workspace_size(d, 152)
    assert ab > smla.STATIC_SCRATCH_BYTES
    with pytest.raises(smla.SparseMLAError) as e:
        smla.sparse_mla_decode_static(d, 152, 0, 0, 0, 0.04, 0, 0, 0)
    assert e.value.code == smla.SMLA_ERR_WORKSPACE
    assert str(smla.STATIC_SCRATCH_BYTES) in str(e.value)
    rc, _ = smla.sparse_mla_static_read_status(d, 152)
    assert rc == smla.SMLA_ERR_WORKSPACE


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
    assert smla.sparse_mla_static_read_status(_dims(wl_a), nsm) == (0, 0)
    out2, lse2 = _static_run(wl_b, nsm)
    assert smla.sparse_mla_static_read_status(_dims(wl_b), nsm) == (0, 0)
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
        assert smla.sparse_mla_static_read_status(_dims(wl), nsm) == (0, 0)
        _check_same(wl, out_s, lse_s, out_r, lse_r, f"static call {call}")


@pytest.mark.gpu
def test_static_runs_the_prefill_shaped_workload(cuda_ok):
    """b = 1, s_q = 4096, h_q = 128: the plan splits no request, so the scratch holds only the
    plan; the static call's result equals the three-call sequence bit for bit."""
    import torch
    dev = torch.device("cuda:0")
    wl = workloads.make(workloads.CONFIGS["c5_b1_sq4096_h128_k2048"], device=dev)
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    op = smla.SparseMLADecode(wl.spec.b, wl.spec.s_q, wl.spec.h_q, wl.spec.topk,
                              wl.kv.shape[0], device=dev, num_sms=nsm)
    assert op.accum_bytes == 0
    out_r, lse_r = op.run(wl.q, wl.kv, wl.indices, wl.sm_scale)
    out_s, lse_s = _static_run(wl, nsm)
    torch.cuda.synchronize(dev)
    assert smla.sparse_mla_static_read_status(_dims(wl), nsm) == (0, 0)
    assert torch.equal(out_s.view(torch.int16), out_r.view(torch.int16))
    assert torch.equal(lse_s.view(torch.int32), lse_r.view(torch.int32))


@pytest.mark.gpu
def test_static_survives_a_device_reset(cuda_ok):
    """A device reset ends the context whose module holds the scratch array; the next static
    call must find the array again (run in a child process that owns its device memory
    through the CUDA runtime, so no torch state is left dangling by the reset)."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-m", "tests.static_reset_child"], cwd=root,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "STATIC RESET CHILD OK" in r.stdout


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", ["v41", "v4"])
def test_static_runs_the_later_formats(cuda_ok, fmt):
    # the static scratch takes any problem that fits, whatever the cache format
    import torch
    from tests.gpu_util import run_cuda
    smla.lib()
    dev = torch.device("cuda:0")
    wl = workloads.small(b=3, s_q=2, h_q=128, topk=300, ctx=2048, masked_per_row=5, seed=57,
                         device=dev, kv_format=fmt)
    out_r, lse_r, _ = run_cuda(wl, num_sms=152)
    out_s, lse_s = _static_run(wl, 152)
    torch.cuda.synchronize()
    assert torch.equal(out_s, out_r) and torch.equal(lse_s, lse_r)
    d = smla.dims_for(3, 2, 128, 300, wl.kv.shape[0], kv_format=fmt)
    rc, word = smla.sparse_mla_static_read_status(d, 152)
    assert rc == smla.SMLA_OK and word == 0
