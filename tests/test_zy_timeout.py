"""The failure path on the GPU without a fault: the test_stall hook makes every partition's
MMA issuer wait on a barrier that nothing arrives at.  Every waiting role gives up after its
bounded wait, the kernel returns, the device status word reports SMLA_DEV_TIMEOUT and records
the first wait that ran out, and the context stays usable: the next call is correct and
clean.  (Runs last: it takes about a second of wall time.)"""

import time

import numpy as np
import pytest
import torch

import oracle
import sparse_mla_attention_decode_gb300 as smla
import workloads
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_the_context_stays_usable(cuda_ok):
    dev = torch.device("cuda:0")
    wl = workloads.small(b=3, h_q=128, topk=256, ctx=1024, device=dev, seed=61)
    op = smla.SparseMLADecode(wl.spec.b, wl.spec.s_q, wl.spec.h_q, wl.spec.topk,
                              wl.kv.shape[0], device=dev, num_sms=16)
    st = torch.cuda.current_stream(dev).cuda_stream
    out = torch.empty(3, 1, 128, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(3, 128, 1, dtype=torch.float32, device=dev)
    opts = smla.smla_decode_opts()
    opts.test_stall = 1
    smla.sparse_mla_sched_meta(op.dims, op.num_sms, op.sched.data_ptr(), op.sched_bytes, st)
    t0 = time.perf_counter()
    smla.sparse_mla_decode_fwd_ex(op.dims, op.num_sms, wl.q.data_ptr(), wl.kv.data_ptr(),
                                  wl.indices.data_ptr(), wl.sm_scale, opts, op.sched.data_ptr(),
                                  op.workspace.data_ptr(), op.accum_bytes, out.data_ptr(),
                                  lse.data_ptr(), st)
    smla.sparse_mla_combine_ex(op.dims, op.num_sms, opts, op.sched.data_ptr(),
                               op.workspace.data_ptr(), op.accum_bytes, out.data_ptr(),
                               lse.data_ptr(), st)
    rc, word = smla.sparse_mla_read_device_status(op.dims, op.num_sms, op.sched.data_ptr(), st)
    waited = time.perf_counter() - t0
    assert rc == smla.SMLA_ERR_TIMEOUT and word & smla.SMLA_DEV_TIMEOUT
    assert waited > 0.5  # the bounded waits (one second) ran out; nothing returned early
    # status word 1: the first wait that ran out (marker bit, CTA rank, role, barrier, parity)
    meta, pre = op.plan()
    parts = meta.shape[0]
    status_off = ((parts * 32 + (3 + 1) * 4) + 15) // 16 * 16
    words = op.sched.cpu()[status_off:status_off + 8].view(torch.int32)
    assert int(words[1]) & 0x80000000 == 0x80000000 or int(words[1]) < 0
    # the context is usable: the same problem again, normally
    out2, lse2 = op.run(wl.q, wl.kv, wl.indices, wl.sm_scale)
    torch.cuda.synchronize(dev)
    assert op.device_status() == 0
    q, kv, idx = workloads.to_numpy_inputs(wl)
    ro, rl = oracle.sparse_mla_decode_full(q, kv, idx, wl.sm_scale)
    gu.compare(out2.double().cpu().numpy().reshape(-1, 128, 512),
               lse2.double().cpu().numpy().transpose(0, 2, 1).reshape(-1, 128),
               ro.reshape(-1, 128, 512), rl.transpose(0, 2, 1).reshape(-1, 128), "after a timeout")


def test_indexer_bounded_wait_runs_out_and_the_context_stays_usable(cuda_ok):
    # the indexer's MMA issuer waits on a barrier nothing arrives at: the producer (after
    # waiting for the copies it issued), the epilogue and the issuer all leave their bounded
    # waits, the status word reports SMLA_DEV_TIMEOUT, no score is written, and the next call
    # on the same context is correct and clean
    from oracle import indexer as oix
    dev = torch.device("cuda:0")
    b, pages, ld = 2, 40, 2560
    cache = workloads.indexer_cache(pages, seed=90, device=dev)
    q8, w = workloads.indexer_queries(b, seed=91, device=dev)
    table = torch.arange(pages, dtype=torch.int32, device=dev).view(1, pages).repeat(b, 1).contiguous()
    lens = torch.tensor([ld, 1000], dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.full((b, ld), 7.0, dtype=torch.float32, device=dev)
    d = smla.smla_indexer_dims(b, 1, 64, 128, pages, ld, pages)
    d.test_stall = 1
    st = torch.cuda.current_stream(dev).cuda_stream
    t0 = time.perf_counter()
    smla.sparse_mla_indexer_scores(d, 8, q8.data_ptr(), w.data_ptr(), cache.data_ptr(),
                                   table.data_ptr(), lens.data_ptr(), out.data_ptr(),
                                   status.data_ptr(), st)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) & smla.SMLA_DEV_TIMEOUT
    assert 0.5 < elapsed < 10.0, elapsed
    assert bool(torch.all(out == 7.0)), "no tile reached the epilogue, so no score is written"
    status.zero_()
    got = smla.indexer_scores(q8, w, cache, table, lens, 1, ld, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oix.indexer_scores(q8.cpu().numpy(), w.cpu().double().numpy(), cache.cpu().numpy(),
                             table.cpu().numpy(), lens.cpu().numpy(), 1, ld)
    g = got.double().cpu().numpy()
    for t in range(b):
        n = int(lens[t])
        tol = 2e-5 * max(1.0, float(np.abs(ref[t, :n]).max())) + 1e-6
        assert float(np.abs(g[t, :n] - ref[t, :n]).max()) <= tol


def test_chained_selection_reports_an_indexer_timeout(cuda_ok):
    # the chained indexer -> top-k call with the indexer's stall hook: the indexer's waits run
    # out, the top-k then selects from whatever the scratch holds, and the required status word
    # carries SMLA_DEV_TIMEOUT, so the caller sees that the ids are not valid; the next chained
    # call on the same context is clean
    dev = torch.device("cuda:0")
    b, pages, ld, k = 2, 40, 2560, 64
    cache = workloads.indexer_cache(pages, seed=92, device=dev)
    q8, w = workloads.indexer_queries(b, seed=93, device=dev)
    table = torch.arange(pages, dtype=torch.int32, device=dev).view(1, pages).repeat(b, 1).contiguous()
    lens = torch.tensor([ld, 1000], dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty(b, k, dtype=torch.int32, device=dev)
    d = smla.smla_indexer_dims(b, 1, 64, 128, pages, ld, pages)
    d.test_stall = 1
    scratch = torch.empty(smla.sparse_mla_indexer_topk_scratch_size(d), dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream(dev).cuda_stream
    smla.sparse_mla_indexer_topk(d, k, 8, q8.data_ptr(), w.data_ptr(), cache.data_ptr(),
                                 table.data_ptr(), lens.data_ptr(), scratch.data_ptr(),
                                 scratch.numel(), out.data_ptr(), status.data_ptr(), st)
    torch.cuda.synchronize()
    assert int(status.item()) & smla.SMLA_DEV_TIMEOUT
    status.zero_()
    smla.indexer_topk(q8, w, cache, table, lens, 1, ld, k, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
