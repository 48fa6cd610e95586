"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and compare with the
oracle.  Tolerances come from the accuracy target of this project: O max-abs <= 2e-2,
relative L2 <= 5e-3 over the compared tensor, LSE abs <= 1e-3 with +inf matching +inf."""

from __future__ import annotations

import numpy as np
import torch

import oracle
import sparse_mla_attention_decode_gb300 as smla
import workloads

O_MAX_ABS = 2e-2
O_REL_L2 = 5e-3
LSE_ABS = 1e-3


def run_cuda(wl: workloads.Workload, num_sms: int = 0, check_status: bool = True,
             attn_sink=None, topk_length=None, partials_bf16: bool = False, extra_kv=None,
             extra_indices=None, extra_topk_length=None):
    dev = wl.q.device
    ek = 0 if extra_indices is None else extra_indices.shape[-1]
    enb = 0 if extra_kv is None else extra_kv.shape[0]
    op = smla.SparseMLADecode(wl.spec.b, wl.spec.s_q, wl.spec.h_q, wl.spec.topk,
                              wl.kv.shape[0], device=dev, num_sms=num_sms, extra_topk=ek,
                              extra_num_blocks=enb, kv_format=wl.spec.kv_format)
    out, lse = op.run(wl.q, wl.kv, wl.indices, wl.sm_scale, attn_sink=attn_sink,
                      topk_length=topk_length, partials_bf16=partials_bf16, extra_kv=extra_kv,
                      extra_indices=extra_indices, extra_topk_length=extra_topk_length)
    torch.cuda.synchronize(dev)
    if check_status:
        word = op.device_status()
        assert word == 0, f"device status word {word:#x}"
    return out, lse, op


def accum_layout(prefix, s_q: int, h_q: int):
    """(slots, lse byte offset) of the split-partial workspace of a plan with this num_splits
    prefix, as include/sparse_mla.h documents it: slots = prefix[r + 1] for the last request r
    that the plan splits (0 when none is), fp32 partial O [slots][s_q][h_q][512], then the
    base-2 lse [slots][s_q][h_q] at the next 256-byte boundary."""
    prefix = [int(x) for x in prefix]
    split = [r for r in range(len(prefix) - 1) if prefix[r + 1] - prefix[r] > 1]
    slots = prefix[split[-1] + 1] if split else 0
    return slots, ((slots * s_q * h_q * 512 * 4) + 255) // 256 * 256


def compact_inputs(wl: workloads.Workload, tokens: np.ndarray):
    """Oracle inputs restricted to ``tokens``: the rows those tokens select are gathered (with
    torch, from the seeded inputs) into a small pool and their indices renumbered.  Invalid
    slots stay invalid."""
    b, s_q = wl.spec.b, wl.spec.s_q
    nrows = wl.kv.shape[0] * 64
    idx = wl.indices.view(b * s_q, -1)[torch.as_tensor(tokens, device=wl.indices.device)]
    valid = (idx >= 0) & (idx < nrows)
    used = torch.unique(idx[valid])
    remap = torch.full((nrows,), -1, dtype=torch.int64, device=idx.device)
    remap[used] = torch.arange(used.numel(), device=idx.device)
    new_idx = torch.where(valid, remap[idx.clamp(0, nrows - 1).long()], torch.full_like(idx, -1).long())
    npages = (used.numel() + 63) // 64
    pool = torch.zeros(max(npages, 1) * 64, 656, dtype=torch.uint8, device=idx.device)
    pool[: used.numel()] = wl.kv.view(nrows, 656)[used]
    q = wl.q.view(b * s_q, wl.spec.h_q, 576)[torch.as_tensor(tokens, device=wl.q.device)]
    n = len(tokens)
    qb = q.cpu().contiguous().view(torch.int16).numpy().view("uint16").reshape(n, 1, wl.spec.h_q, 576)
    kvn = pool.cpu().numpy().reshape(-1, 64, 656)
    idn = new_idx.to(torch.int32).cpu().numpy().reshape(n, 1, -1)
    return qb, kvn, idn


def compact_pool(kv: torch.Tensor, idx_rows: torch.Tensor):
    """(small pool [pages, 64, 656] numpy, renumbered int32 indices numpy) holding only the
    rows that ``idx_rows`` [n, k] selects from ``kv``; invalid slots stay invalid."""
    nrows = kv.shape[0] * 64
    valid = (idx_rows >= 0) & (idx_rows < nrows)
    used = torch.unique(idx_rows[valid])
    remap = torch.full((max(nrows, 1),), -1, dtype=torch.int64, device=idx_rows.device)
    remap[used] = torch.arange(used.numel(), device=idx_rows.device)
    new_idx = torch.where(valid, remap[idx_rows.clamp(0, max(nrows - 1, 0)).long()],
                          torch.full_like(idx_rows, -1).long())
    npages = (used.numel() + 63) // 64
    pool = torch.zeros(max(npages, 1) * 64, 656, dtype=torch.uint8, device=idx_rows.device)
    if used.numel():
        pool[: used.numel()] = kv.reshape(nrows, 656)[used]
    return pool.cpu().numpy().reshape(-1, 64, 656), new_idx.to(torch.int32).cpu().numpy()


def oracle_tokens_extra(wl: workloads.Workload, tokens, extra_kv, extra_indices,
                        extra_topk_length=None, attn_sink=None, topk_length=None):
    """oracle_tokens with an extra cache and list (both pools compacted to the used rows)."""
    tokens = np.asarray(tokens, dtype=np.int64)
    qb, kvn, idn = compact_inputs(wl, tokens)
    n = len(tokens)
    t = torch.as_tensor(tokens, device=extra_indices.device)
    ekv, eidx = compact_pool(extra_kv, extra_indices.reshape(wl.spec.b * wl.spec.s_q, -1)[t])
    sink = None if attn_sink is None else attn_sink.double().cpu().numpy()
    lens = None if topk_length is None else topk_length.reshape(-1).cpu().numpy()[tokens].reshape(-1, 1)
    elens = (None if extra_topk_length is None
             else extra_topk_length.reshape(-1).cpu().numpy()[tokens].reshape(-1, 1))
    out, lse, _ = oracle.sparse_mla_decode(qb, kvn, idn, wl.sm_scale, attn_sink=sink,
                                           topk_length=lens, extra_kv=ekv,
                                           extra_indices=eidx.reshape(n, 1, -1),
                                           extra_topk_length=elens)
    return out, lse


def oracle_tokens(wl: workloads.Workload, tokens, threads: int = 0, attn_sink=None,
                  topk_length=None):
    """Oracle (out [n, h, 512], lse [n, h]) for the given flattened query tokens, with the
    optional decode variants (sink [h_q], per-token lengths [b, s_q]) as host tensors."""
    tokens = np.asarray(tokens, dtype=np.int64)
    qb, kvn, idn = compact_inputs(wl, tokens)
    sink = None if attn_sink is None else attn_sink.double().cpu().numpy()
    lens = None
    if topk_length is not None:
        lens = topk_length.reshape(-1).cpu().numpy()[tokens].reshape(-1, 1)
    out, lse, _ = oracle.sparse_mla_decode(qb, kvn, idn, wl.sm_scale, threads=threads,
                                           attn_sink=sink, topk_length=lens)
    return out, lse


def gpu_tokens(out: torch.Tensor, lse: torch.Tensor, wl: workloads.Workload, tokens):
    b, s_q, h = wl.spec.b, wl.spec.s_q, wl.spec.h_q
    t = torch.as_tensor(np.asarray(tokens), device=out.device)
    o = out.view(b * s_q, h, 512)[t].double().cpu().numpy()
    l = lse.permute(0, 2, 1).reshape(b * s_q, h)[t].double().cpu().numpy()
    return o, l


def compare(o_gpu, l_gpu, o_ref, l_ref, what: str = ""):
    """Assert the tolerances; returns the metrics."""
    assert o_gpu.shape == o_ref.shape and l_gpu.shape == l_ref.shape
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite output"
    inf_ref = np.isposinf(l_ref)
    assert np.array_equal(np.isposinf(l_gpu), inf_ref), f"{what}: +inf lse mismatch"
    assert np.all(np.isfinite(l_gpu[~inf_ref])), f"{what}: non-finite lse"
    err = np.abs(o_gpu - o_ref)
    max_abs = float(err.max()) if err.size else 0.0
    denom = float(np.linalg.norm(o_ref))
    rel = float(np.linalg.norm(o_gpu - o_ref) / denom) if denom > 0 else float(np.linalg.norm(o_gpu))
    rows = np.linalg.norm(o_gpu - o_ref, axis=-1) / np.maximum(np.linalg.norm(o_ref, axis=-1), 1e-30)
    worst_row = float(rows[np.linalg.norm(o_ref, axis=-1) > 0].max()) if np.any(
        np.linalg.norm(o_ref, axis=-1) > 0) else 0.0
    lse_err = float(np.abs(l_gpu[~inf_ref] - l_ref[~inf_ref]).max()) if np.any(~inf_ref) else 0.0
    assert np.all(o_gpu[inf_ref] == 0.0), f"{what}: all-masked rows must be 0"
    assert max_abs <= O_MAX_ABS, f"{what}: max abs {max_abs}"
    assert rel <= O_REL_L2, f"{what}: rel L2 {rel}"
    assert lse_err <= LSE_ABS, f"{what}: lse abs {lse_err}"
    return {"max_abs": max_abs, "rel_l2": rel, "worst_row_rel": worst_row, "lse_abs": lse_err}


def oracle_tokens_fmt(wl: workloads.Workload, tokens, attn_sink=None, topk_length=None,
                      extra_kv=None, extra_indices=None, extra_topk_length=None):
    """Later-format oracle (out [n, h, 512], lse [n, h]) for the given flattened tokens; the
    pool is read on the host (whole), the FP4 extra cache likewise."""
    from oracle import formats as ofmt
    q = wl.q.cpu().contiguous().view(torch.int16).numpy().view("uint16")
    pool = wl.kv.cpu().numpy()
    kw = {}
    if attn_sink is not None:
        kw["attn_sink"] = attn_sink.double().cpu().numpy()
    if topk_length is not None:
        kw["topk_length"] = topk_length.cpu().numpy()
    if extra_indices is not None:
        kw.update(extra_pool=extra_kv.cpu().numpy(), extra_fmt="v41_fp4",
                  extra_indices=extra_indices.cpu().numpy())
        if extra_topk_length is not None:
            kw["extra_topk_length"] = extra_topk_length.cpu().numpy()
    out, lse, _ = ofmt.sparse_mla_decode_fmt(q, pool, wl.indices.cpu().numpy(), wl.sm_scale,
                                             wl.spec.kv_format, tokens=np.asarray(tokens), **kw)
    return out, lse
