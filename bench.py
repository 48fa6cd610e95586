"""Benchmark: sparse MLA decode on GB300 (TFLOPS, gathered KV tokens/s, fraction of roofline).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step = the whole hot path on one batch: split-KV plan (sched_meta), decode pass, combine,
all through the C ABI, inputs resident in HBM.  L2 is flushed between steps (a 256 MiB
write, then a 256 MiB read of another buffer that writes the dirty lines back); the flush is
outside the step time.  Prints one JSON line (rank 0).

--impl reference times the fp64 CPU oracle on the host cores on a bounded sample of the same
workload (the reference arm of this project: the pages ship no runnable code).
Under torchrun (N > 1) every rank runs an independent replica of the workload on its own GPU
(no collective on the data path) and the job value is the sum of work over the max time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(ROOT, "sparse_mla_attention_decode_gb300", "csrc")
FLUSH_NOTE = ("flushed between steps (256 MiB write, then a 256 MiB read of another buffer so "
              "no dirty line is left; outside the step time)")
sys.path.insert(0, ROOT)

METRIC = "sparse MLA decode TFLOPS & gathered KV tokens/s, % of roofline (1×GB300)"
# The headline is the largest single-GPU workload of the five (the prefill-shaped one, 2.3
# TFLOP a step); the other four are measured in the same run and reported under per_config.
DEFAULT_WORKLOAD = "c5_b1_sq4096_h128_k2048"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


def max_over_ranks(values, device="cpu"):
    """Element-wise maximum of ``values`` over the ranks of the default process group (the
    values unchanged when there is none)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def code_sha256(path: str) -> str:
    """sha256 of a source file's code: // and /* */ comments removed, whitespace collapsed, so
    that a comment edit does not make a profile of an unchanged kernel stale."""
    txt = open(path, encoding="utf-8").read()
    txt = re.sub(r"/\*.*?\*/", " ", txt, flags=re.S)
    txt = re.sub(r"//[^\n]*", " ", txt)
    return hashlib.sha256(" ".join(txt.split()).encode()).hexdigest()


def traffic_from_profiles(kernel_src: str, profile: str, alg_bytes=None):
    """DRAM bytes per launch from a committed ncu summary, or None when the summary is missing
    or was taken on different kernel code (its code_sha256, or else its source_sha256, against
    the current file).  A summary captured on a smaller case than the bench's records its own
    algorithmic bytes; its traffic is then scaled by the ratio of the algorithmic bytes (the
    kernel reads each valid input byte once, so traffic grows in proportion)."""
    path = os.path.join(ROOT, "profiles", profile)
    if not os.path.exists(path):
        return None
    txt = open(path, encoding="utf-8").read()
    m_code = re.search(r"code_sha256:\s*([0-9a-f]{64})", txt)
    m_src = re.search(r"source_sha256:\s*([0-9a-f]{64})", txt)
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not m_b or not (m_code or m_src):
        return None
    if m_code:
        if m_code.group(1) != code_sha256(kernel_src):
            return None
    elif m_src.group(1) != hashlib.sha256(open(kernel_src, "rb").read()).hexdigest():
        return None
    traffic = float(m_b.group(1))
    m_a = re.search(r"alg_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if alg_bytes is not None and m_a:
        traffic *= float(alg_bytes) / float(m_a.group(1))
    return traffic


def decode_config(spec, wl, ws: int) -> dict:
    """The decode line's ``config``, the same for both arms (the workload, not how it is
    timed: the reference arm's token sample is in its ``cpu_baseline.sample``)."""
    return {"workload": spec.name, "b": spec.b, "s_q": spec.s_q, "h_q": spec.h_q,
            "topk": spec.topk, "ctx": spec.ctx, "num_blocks": int(wl.kv.shape[0]),
            "valid_slots": int(wl.num_valid),
            "parallelism": f"replicas x{ws}" if ws > 1 else "1 GPU", "l2": FLUSH_NOTE}


def traffic_from_pair_profile(sources, profile: str):
    """DRAM bytes per step of a chain of kernels from one committed ncu summary that lists a
    ``code_sha256 <file>: <hash>`` line per kernel source and their summed
    ``dram_bytes_per_step``; None when the summary is missing or any source has changed."""
    path = os.path.join(ROOT, "profiles", profile)
    if not os.path.exists(path):
        return None
    txt = open(path, encoding="utf-8").read()
    for src in sources:
        m = re.search(r"code_sha256 %s:\s*([0-9a-f]{64})" % re.escape(os.path.basename(src)), txt)
        if not m or m.group(1) != code_sha256(src):
            return None
    m_b = re.search(r"dram_bytes_per_step:\s*([0-9.eE+]+)", txt)
    return float(m_b.group(1)) if m_b else None


def rotated_index_sets(indices, block_table, num_blocks: int, n_sets: int, shift_pages: int = 128):
    """n_sets index tensors (int32, host): the given one, then the same slots with every valid
    position of a sequence moved by j * shift_pages pages (cyclically within the sequence's
    pages) and mapped back through its page table; masked slots stay -1, so the valid count
    and the FLOPs are the same."""
    import torch
    bt = block_table.long().cpu()
    b, pages = bt.shape
    inv = torch.zeros(num_blocks, dtype=torch.int64)  # physical page -> its logical index
    inv[bt.reshape(-1)] = torch.arange(pages).repeat(b)
    base = indices.long().cpu()
    seq = torch.arange(b).view(b, *([1] * (base.dim() - 1))).expand_as(base)
    ok = base >= 0
    pos = inv[base.clamp(min=0) // 64] * 64 + base.clamp(min=0) % 64
    out = [indices.cpu().to(torch.int32).contiguous()]
    for j in range(1, n_sets):
        moved = (pos + j * shift_pages * 64) % (pages * 64)
        phys = bt[seq, moved // 64] * 64 + moved % 64
        out.append(torch.where(ok, phys, base).to(torch.int32).contiguous())
    return out


class L2Flush:
    """Leaves L2 holding none of the next step's inputs and no dirty line: a 256 MiB write
    (larger than L2), then a 256 MiB read of a second buffer, which writes the dirty lines back
    before the timed step starts instead of during it."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(256 << 20, dtype=torch.uint8, device=dev)

    def __call__(self, k: int = 1):
        self.w.fill_(k & 0xFF)
        self.r.max()


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "samples": len(sm),
                "reasons": sorted(reasons)}


def compact_for_oracle(wl, tokens):
    """Inputs restricted to ``tokens`` with the rows they select gathered into a small pool
    (indices renumbered, invalid slots kept invalid), as numpy arrays for the oracle."""
    import numpy as np
    import torch
    b, s_q, h = wl.spec.b, wl.spec.s_q, wl.spec.h_q
    nrows = wl.kv.shape[0] * 64
    t = torch.as_tensor(tokens, device=wl.indices.device)
    idx = wl.indices.view(b * s_q, -1)[t].long()
    valid = (idx >= 0) & (idx < nrows)
    used = torch.unique(idx[valid])
    remap = torch.full((nrows,), -1, dtype=torch.int64, device=idx.device)
    remap[used] = torch.arange(used.numel(), device=idx.device)
    new_idx = torch.where(valid, remap[idx.clamp(0, nrows - 1)], torch.full_like(idx, -1))
    pool = torch.zeros(max((used.numel() + 63) // 64, 1) * 64, 656, dtype=torch.uint8,
                       device=idx.device)
    pool[: used.numel()] = wl.kv.view(nrows, 656)[used]
    n = len(tokens)
    q = wl.q.view(b * s_q, h, 576)[t].cpu().contiguous().view(torch.int16).numpy().view("uint16")
    return (q.reshape(n, 1, h, 576), pool.cpu().numpy().reshape(-1, 64, 656),
            new_idx.to(torch.int32).cpu().numpy().reshape(n, 1, -1),
            int(valid.sum().item()))


def time_oracle(wl, budget_s: float, max_tokens: int | None = None):
    """Run the oracle over the workload's query tokens (4 at a time, all heads) until
    ``budget_s`` of oracle time is spent, going round the tokens again if one pass is shorter;
    with ``max_tokens``, one pass over that many tokens.  Input compaction is not timed."""
    import oracle
    import workloads
    n_tok = wl.spec.b * wl.spec.s_q
    chunk = 4
    limit = n_tok if max_tokens is None else min(n_tok, max_tokens)
    cache = {}
    done, valid, elapsed = 0, 0, 0.0
    while elapsed < budget_s or done == 0:
        start = done % limit
        if max_tokens is not None and done >= limit:
            break
        if start not in cache:
            cache[start] = compact_for_oracle(wl, list(range(start, min(limit, start + chunk))))
        q, kv, idx, nv = cache[start]
        t0 = time.perf_counter()
        oracle.sparse_mla_decode(q, kv, idx, wl.sm_scale)
        elapsed += time.perf_counter() - t0
        done += q.shape[0]
        valid += nv
    flops = 2.0 * wl.spec.h_q * (workloads.D_QK + workloads.D_V) * valid
    return {"flops": flops, "seconds": elapsed, "tokens": done, "valid_slots": valid,
            "threads": oracle.max_threads(), "passes": done / limit, "pool": limit}


def roofline_of(wl, t_dec: float, peaks) -> dict:
    """The decode kernel against its roofline: T_roof = max(valid-slot FLOPs / bf16 tensor peak,
    algorithmic bytes / HBM bandwidth); frac = T_roof / measured time; bound = the larger."""
    import workloads
    flops = workloads.flops_valid(wl)
    alg = workloads.alg_bytes(wl)
    t_tensor = flops / (float(peaks["bf16_tflops"]) * 1e12)
    t_hbm = alg / (float(peaks["hbm_gbs"]) * 1e9)
    bound = "tensor" if t_tensor >= t_hbm else "hbm"
    return {"bound": bound, "t_roof_us": max(t_tensor, t_hbm) * 1e6,
            "frac": max(t_tensor, t_hbm) / t_dec,
            "tflops": flops / t_dec / 1e12, "hbm_gbs": alg / t_dec / 1e9,
            "tensor_frac": t_tensor / t_dec, "hbm_frac": t_hbm / t_dec}


def measure_decode(spec, wl, dev, steps: int, warmup: int, flush, gpu_index: int,
                   barrier=None):
    """Time plan + decode + combine (one step) and the decode kernel alone on one workload with
    CUDA events on the launching stream, L2 flushed before every step (outside the events),
    nvidia-smi clocks sampled during the timed region.  Returns a dict of raw times, the op and
    the output buffers."""
    import torch

    import sparse_mla_attention_decode_gb300 as smla
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    op = smla.SparseMLADecode(spec.b, spec.s_q, spec.h_q, spec.topk, wl.kv.shape[0], device=dev,
                              num_sms=num_sms, kv_format=spec.kv_format)
    out = torch.empty(spec.b, spec.s_q, spec.h_q, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(spec.b, spec.h_q, spec.s_q, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    st = stream.cuda_stream
    d = op.dims

    def sched():
        smla.sparse_mla_sched_meta(d, num_sms, op.sched.data_ptr(), op.sched_bytes, st)

    def decode():
        smla.sparse_mla_decode_fwd(d, num_sms, wl.q.data_ptr(), wl.kv.data_ptr(),
                                   wl.indices.data_ptr(), wl.sm_scale, op.sched.data_ptr(),
                                   op.workspace.data_ptr(), op.accum_bytes, out.data_ptr(),
                                   lse.data_ptr(), st)

    def combine():
        smla.sparse_mla_combine(d, num_sms, op.sched.data_ptr(), op.workspace.data_ptr(),
                                op.accum_bytes, out.data_ptr(), lse.data_ptr(), st)

    launches_per_step = 3 if smla.sparse_mla_plan_has_splits(d, num_sms) else 2

    # One step = plan + decode + combine, back to back on the stream (events only around the
    # whole step, so the launches overlap as they do in use).
    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        sched()
        decode()
        combine()
        if ev is not None:
            ev[1].record(stream)

    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize(dev)
    if op.device_status() != 0:
        raise RuntimeError(f"{spec.name}: device status word set during warm-up")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    dec_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    sampler = ClockSampler(gpu_index)
    if barrier is not None:
        barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    t0 = time.perf_counter()
    for k in range(steps):
        flush(k)
        step(evs[k])
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t0
    # the decode kernel alone (for the roofline): events on the launching stream around it
    for k in range(steps):
        flush(k)
        sched()
        dec_evs[k][0].record(stream)
        decode()
        dec_evs[k][1].record(stream)
        combine()
    torch.cuda.synchronize(dev)
    if barrier is not None:
        barrier()
    clocks = sampler.stop()
    if op.device_status() != 0:
        raise RuntimeError(f"{spec.name}: device status word set during the timed steps")
    step_ms = [e[0].elapsed_time(e[1]) for e in evs]
    dec_ms = [e[0].elapsed_time(e[1]) for e in dec_evs]
    return {"op": op, "out": out, "lse": lse, "step_ms": step_ms, "dec_ms": dec_ms,
            "wall": wall, "clocks": clocks, "launches_per_step": launches_per_step}


def per_config_entry(spec, wl, r, peaks) -> dict:
    import workloads
    t_step = sum(r["step_ms"]) / len(r["step_ms"]) / 1e3
    t_dec = sum(r["dec_ms"]) / len(r["dec_ms"]) / 1e3
    rf = roofline_of(wl, t_dec, peaks)
    return {"step_us": t_step * 1e6, "decode_us": t_dec * 1e6,
            "step_tflops": workloads.flops_valid(wl) / t_step / 1e12,
            "decode_tflops": rf["tflops"], "decode_hbm_gbs": rf["hbm_gbs"],
            "gathered_tokens_per_s": wl.num_valid / t_step,
            "roofline": {"bound": rf["bound"], "t_roof_us": rf["t_roof_us"], "frac": rf["frac"],
                         "tensor_frac": rf["tensor_frac"], "hbm_frac": rf["hbm_frac"]},
            "valid_slots": wl.num_valid, "launches_per_step": r["launches_per_step"],
            "clocks": r["clocks"]}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import torch
    import workloads
    import oracle
    oracle.build()
    spec = workloads.CONFIGS[args.workload]
    dev = "cuda:0" if torch.cuda.is_available() else "cpu"
    wl = workloads.make(spec, device=dev)
    per_step_tokens = max(1, min(spec.b * spec.s_q, args.ref_tokens))
    for _ in range(args.warmup):
        time_oracle(wl, 1e9, max_tokens=per_step_tokens)
    secs, flops, valid = [], 0.0, 0
    for _ in range(args.steps):
        r = time_oracle(wl, 1e9, max_tokens=per_step_tokens)
        secs.append(r["seconds"])
        flops += r["flops"]
        valid += r["valid_slots"]
    total = sum(secs)
    tflops = flops / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": tflops, "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": decode_config(spec, wl, ws),
        "gathered_tokens_per_s": valid / total,
        "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": oracle.max_threads(),
                         "kind": "oracle",
                         "sample": f"{per_step_tokens} of {spec.b * spec.s_q} query tokens of "
                                   f"{spec.name} per step, all heads"},
        "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_topk(args):
    """The exact top-k with the page-table emit on prefill-shaped index scores: --topk-rows
    query tokens of one request over a 65536-token context, causal (query i sees positions
    [0, 61440 + i]), bf16 N(0, 1) scores, k = 2048.  HBM-bound: the algorithmic bytes are the
    valid score bytes read once plus the int32 ids written.  The scores (512 MB at the
    default) are larger than L2, so no flush is needed between steps."""
    import torch

    import sparse_mla_attention_decode_gb300 as smla
    import workloads

    dev = torch.device("cuda:0")
    n_tok, ld, k = args.topk_rows, 65536, 2048
    scores = workloads.index_scores(n_tok, ld, torch.bfloat16, seed=4, device=dev)
    lens = (61441 + torch.arange(n_tok, device=dev)).clamp(max=ld).to(torch.int32)
    table = torch.randperm(ld // 64 * 2, generator=torch.Generator().manual_seed(5))[: ld // 64]
    table = table.to(torch.int32).view(1, -1).to(dev)
    out = torch.empty(n_tok, k, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        smla.topk_page_table(scores, lens, table, n_tok, k, out=out)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(args.steps):
        smla.topk_page_table(scores, lens, table, n_tok, k, out=out)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    t = e0.elapsed_time(e1) / 1e3 / args.steps
    alg = int(lens.sum().item()) * 2 + n_tok * k * 4
    peaks, peak_src = load_peaks()
    peak = float(peaks["hbm_gbs"])
    achieved = alg / t / 1e9
    traffic = traffic_from_profiles(os.path.join(CSRC, "topk.cu"),
                                    "topk_kernel_prefill_1024x65536_k2048.md", alg)
    print(json.dumps({
        "metric": "exact top-k + page-table emit, index-score bytes/s", "impl": "gb300",
        "value": achieved, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"topk_prefill_{n_tok}x{ld}_k{k}", "rows": n_tok, "ld": ld,
                   "topk": k, "causal_base": 61440, "l2": "inputs larger than L2"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_kind": f"{peak_src} copy bandwidth", "alg_bytes_per_launch": alg},
        "gpu_launches": args.steps, "clocks": clocks}), flush=True)


def run_indexer(args):
    """The lightning-indexer scores.  --indexer-shape decode (default): 64 requests, one query
    token each, over 32768 cached tokens (512 indexer pages of 8448 bytes) per request;
    HBM-bound: the algorithmic bytes are the key pages read once per request (132 bytes a
    token), the fp32 scores written and the e4m3 Q and fp32 weights read.  L2 is flushed
    between steps (the 277 MB of pages are larger than L2 too).  --indexer-shape prefill: one
    request, 4096 query tokens over a 65536-token cache, causal (query i sees positions
    [0, 61441 + i]); tensor-bound (2 * 64 * 128 flop per query token and visible position,
    e4m3 MMAs), against the FP8 dense peak taken as twice the measured bf16 one."""
    import torch

    import sparse_mla_attention_decode_gb300 as smla
    import workloads

    dev = torch.device("cuda:0")
    prefill = args.indexer_shape == "prefill"
    b, s_q, ctx = (1, 4096, 65536) if prefill else (64, 1, 32768)
    n_tok = b * s_q
    pages = ctx // 64
    cache = workloads.indexer_cache(b * pages, seed=1, device=dev)
    q8, w = workloads.indexer_queries(n_tok, seed=2, device=dev)
    table = torch.randperm(b * pages, generator=torch.Generator().manual_seed(3))
    table = table.to(torch.int32).view(b, pages).to(dev)
    if prefill:
        lens = (61441 + torch.arange(n_tok, device=dev)).clamp(max=ctx).to(torch.int32)
    else:
        lens = torch.full((n_tok,), ctx, dtype=torch.int32, device=dev)
    out = torch.empty(n_tok, ctx, dtype=torch.float32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        flush()
        smla.indexer_scores(q8, w, cache, table, lens, s_q, ctx, out=out)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.3)
    ts = []
    for _ in range(args.steps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        smla.indexer_scores(q8, w, cache, table, lens, s_q, ctx, out=out)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ts.append(e0.elapsed_time(e1) / 1e3)
    clocks = sampler.stop()
    t = sum(ts) / len(ts)
    visible = int(lens.sum().item())
    # the pages of a request are read once (its query tokens share them)
    req_len = int(lens.view(b, s_q).max(dim=1).values.sum().item())
    alg = req_len * 132 + visible * 4 + n_tok * (64 * 128 + 64 * 4)
    flops = 2.0 * 64 * 128 * visible
    peaks, peak_src = load_peaks()
    workload = f"indexer_prefill_sq{s_q}_ctx{ctx}" if prefill else f"indexer_decode_b{b}_ctx{ctx}"
    config = {"workload": workload, "requests": b, "query_tokens": n_tok, "ctx": ctx,
              "heads": 64, "dim": 128, "l2": FLUSH_NOTE}
    if prefill:
        config["causal_base"] = 61441
        peak = 2.0 * float(peaks["bf16_tflops"])
        achieved = flops / t / 1e12
        metric = ("lightning-indexer scores (e4m3 tensor-core MMA + ReLU + weighted head sum), "
                  "TFLOP/s")
        traffic = traffic_from_profiles(os.path.join(CSRC, "indexer.cu"),
                                        f"indexer_kernel_prefill_sq{s_q}_ctx{ctx}.md", alg)
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": traffic,
                    "peak_kind": f"2 x the {peak_src} bf16 burst (FP8 dense = 2 x bf16 nominal)",
                    "alg_bytes_per_launch": alg}
        value, unit = achieved, "TFLOP/s"
    else:
        peak = float(peaks["hbm_gbs"])
        achieved = alg / t / 1e9
        traffic = traffic_from_profiles(os.path.join(CSRC, "indexer.cu"),
                                        f"indexer_kernel_decode_b{b}_ctx{ctx}.md", alg)
        metric = ("lightning-indexer scores (e4m3 tensor-core MMA + ReLU + weighted head sum), "
                  "bytes/s")
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                    "frac": achieved / peak, "traffic": traffic,
                    "peak_kind": f"{peak_src} copy bandwidth", "alg_bytes_per_launch": alg}
        value, unit = achieved, "GB/s"
    print(json.dumps({
        "metric": metric, "impl": "gb300", "value": value, "unit": unit, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
        "higher_is_better": True, "dtype": "e4m3 x e4m3 -> f32", "data": "synthetic",
        "config": config, "roofline": roofline, "tflops": flops / t / 1e12,
        "gpu_launches": args.steps, "clocks": clocks}), flush=True)


def run_select(args):
    """The two selection steps chained (indexer scores -> exact top-k with the page-table emit,
    the scores only in an L2-sized scratch) on the decode workload's shape: 64 requests, one
    query token each, 32768 cached tokens, k = 2048.  HBM-bound; the algorithmic bytes are the
    indexer pages read once, Q and weights, and the ids written (the scores never reach HBM by
    design, so they are not counted).  L2 is flushed between steps."""
    import torch

    import sparse_mla_attention_decode_gb300 as smla
    import workloads

    dev = torch.device("cuda:0")
    b, ctx, k = 64, 32768, 2048
    pages = ctx // 64
    cache = workloads.indexer_cache(b * pages, seed=1, device=dev)
    q8, w = workloads.indexer_queries(b, seed=2, device=dev)
    table = torch.randperm(b * pages, generator=torch.Generator().manual_seed(3))
    table = table.to(torch.int32).view(b, pages).to(dev)
    lens = torch.full((b,), ctx, dtype=torch.int32, device=dev)
    out = torch.empty(b, k, dtype=torch.int32, device=dev)
    d = smla.smla_indexer_dims(b, 1, 64, 128, pages, ctx, b * pages)
    scratch = torch.empty(smla.sparse_mla_indexer_topk_scratch_size(d), dtype=torch.uint8, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        smla.indexer_topk(q8, w, cache, table, lens, 1, ctx, k, out=out, scratch=scratch)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.3)
    ts = []
    for _ in range(args.steps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ts.append(e0.elapsed_time(e1) / 1e3)
    clocks = sampler.stop()
    t = sum(ts) / len(ts)
    alg = b * pages * 8448 + b * (64 * 128 + 64 * 4) + b * k * 4
    # both kernels of a step (the scores between them stay in L2 by design)
    traffic = traffic_from_pair_profile(
        [os.path.join(CSRC, "indexer.cu"), os.path.join(CSRC, "topk.cu")],
        f"select_kernels_decode_b{b}_ctx{ctx}_k{k}.md")
    peaks, peak_src = load_peaks()
    peak = float(peaks["hbm_gbs"])
    achieved = alg / t / 1e9
    print(json.dumps({
        "metric": "indexer scores + exact top-k chained (scores kept in L2), bytes/s",
        "impl": "gb300", "value": achieved, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
        "dtype": "e4m3 x e4m3 -> f32 scores", "data": "synthetic",
        "config": {"workload": f"select_decode_b{b}_ctx{ctx}_k{k}", "requests": b, "ctx": ctx,
                   "topk": k, "scratch_bytes": scratch.numel(), "l2": FLUSH_NOTE},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_kind": f"{peak_src} copy bandwidth", "alg_bytes_per_launch": alg},
        "gpu_launches": 2 * args.steps, "clocks": clocks}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle time for the cpu_baseline leg")
    ap.add_argument("--ref-tokens", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only --workload (skip the per_config block)")
    ap.add_argument("--kernel", default="decode", choices=["decode", "topk", "indexer", "select"],
                    help="decode: the attention path (the default line); topk: the top-k "
                         "selection with the page-table emit; indexer: the indexer scores; "
                         "select: the two chained; each on its own line")
    ap.add_argument("--topk-rows", type=int, default=4096)
    ap.add_argument("--indexer-shape", default="decode", choices=["decode", "prefill"],
                    help="--kernel indexer: the decode shape (64 requests x 32768, HBM-bound) or "
                         "the prefill shape (4096 query tokens x 65536, tensor-bound)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        return run_reference(args)
    if args.kernel == "topk":
        return run_topk(args)
    if args.kernel == "indexer":
        return run_indexer(args)
    if args.kernel == "select":
        return run_select(args)

    import numpy as np
    import torch

    import sparse_mla_attention_decode_gb300 as smla
    import workloads

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    smla.lib()
    peaks, peak_kind = load_peaks()
    flush = L2Flush(dev)
    barrier = torch.distributed.barrier if ws > 1 else None

    # ---- the other workloads first (one at a time, freed after), single-GPU runs only
    per_config = None
    if ws == 1 and not args.no_per_config:
        per_config = {}
        for name, cfg in list(workloads.CONFIGS.items()) + list(workloads.FORMAT_CONFIGS.items()):
            if name == args.workload:
                continue
            wl_c = workloads.make(cfg, device=dev)
            r = measure_decode(cfg, wl_c, dev, args.steps, args.warmup, flush, local)
            per_config[name] = per_config_entry(cfg, wl_c, r, peaks)
            del wl_c, r
            torch.cuda.empty_cache()

    # the headline is one of the five configurations; a later-format workload may be named
    # too (for a profiling capture of that instance)
    spec = workloads.CONFIGS.get(args.workload) or workloads.FORMAT_CONFIGS[args.workload]
    wl = workloads.make(spec, device=dev)
    r = measure_decode(spec, wl, dev, args.steps, args.warmup, flush, local, barrier)
    op, out, lse = r["op"], r["out"], r["lse"]
    stream = torch.cuda.current_stream(dev)
    step_ms, dec_ms, wall, clocks = r["step_ms"], r["dec_ms"], r["wall"], r["clocks"]
    launches_per_step = r["launches_per_step"]
    t_step = sum(step_ms) / len(step_ms) / 1e3
    t_dec = sum(dec_ms) / len(dec_ms) / 1e3
    if ws > 1:
        t_step, t_dec = max_over_ranks([t_step, t_dec], dev)

    flops = workloads.flops_valid(wl)
    flops_all = 2.0 * spec.h_q * (576 + 512) * spec.b * spec.s_q * spec.topk
    nvalid = wl.num_valid
    alg_bytes = workloads.alg_bytes(wl)
    value = ws * flops / t_step / 1e12
    peak = float(peaks["bf16_tflops"])
    achieved = flops / t_dec / 1e12
    traffic = traffic_from_profiles(os.path.join(CSRC, "decode_fwd.cu"),
                                    f"decode_kernel_{spec.name}.md")

    # ---- end to end through the public API with host buffers (KV cache resident).  Every
    # step copies its q and indices host->device and its out and lse device->host.  Steps are
    # pipelined as a serving loop runs them: the input copy of step k + 1 and the output copy
    # of step k - 1 run on their own streams while step k computes (two device buffers of
    # each, events order the reuse).  Four index sets in rotation (each a shift of the
    # workload's positions by a multiple of 128 pages within every sequence, same mask) keep
    # the rows a step gathers out of L2 from the steps before it where the pool is larger
    # than L2 (the prefill-shaped workload's 43 MB pool stays in L2 by design).
    q_h = wl.q.cpu().pin_memory()
    n_sets = 4
    i_sets = [s.pin_memory() for s in rotated_index_sets(wl.indices, wl.block_table,
                                                         wl.kv.shape[0], n_sets)]
    q_d = [torch.empty_like(wl.q) for _ in range(2)]
    i_d = [torch.empty_like(wl.indices) for _ in range(2)]
    o_d = [torch.empty_like(out) for _ in range(2)]
    l_d = [torch.empty_like(lse) for _ in range(2)]
    o_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    l_h = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(k):
        j = k % 2
        if k >= 2:
            s_in.wait_event(ev_done[j])  # step k - 2 no longer reads q_d[j], i_d[j]
        with torch.cuda.stream(s_in):
            q_d[j].copy_(q_h, non_blocking=True)
            i_d[j].copy_(i_sets[k % n_sets], non_blocking=True)
            ev_in[j].record(s_in)
        stream.wait_event(ev_in[j])
        if k >= 2:
            stream.wait_event(ev_out[j])  # the output copy of step k - 2 has read o_d[j], l_d[j]
        op.run(q_d[j], wl.kv, i_d[j], wl.sm_scale, out=o_d[j], lse=l_d[j], stream=stream)
        ev_done[j].record(stream)
        s_out.wait_event(ev_done[j])
        with torch.cuda.stream(s_out):
            o_h[j].copy_(o_d[j], non_blocking=True)
            l_h[j].copy_(l_d[j], non_blocking=True)
            ev_out[j].record(s_out)

    for k in range(args.warmup):
        e2e_step(k)
    torch.cuda.synchronize(dev)
    if ws > 1:
        torch.distributed.barrier()
    t1 = time.perf_counter()
    for k in range(args.steps):
        e2e_step(args.warmup + k)
    torch.cuda.synchronize(dev)
    t_e2e = (time.perf_counter() - t1) / args.steps
    if ws > 1:
        t_e2e = max_over_ranks([t_e2e], dev)[0]
    # the same with each step alone (copy in, compute, copy out, wait): the latency of a step
    e_times = []
    for k in range(args.steps):
        flush(k)
        torch.cuda.synchronize(dev)
        t2 = time.perf_counter()
        e2e_step(2 * (k % 2))  # no reuse waits needed: everything before has finished
        torch.cuda.synchronize(dev)
        e_times.append(time.perf_counter() - t2)
    t_e2e_serial = sum(e_times) / len(e_times)
    h2d = q_h.numel() * q_h.element_size() + i_sets[0].numel() * i_sets[0].element_size()
    d2h = o_h[0].numel() * o_h[0].element_size() + l_h[0].numel() * l_h[0].element_size()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and spec.kv_format == "v32":
        import oracle
        oracle.build()
        r = time_oracle(wl, args.cpu_budget)
        cpu = {"value": r["flops"] / r["seconds"] / 1e12, "unit": "TFLOP/s",
               "cores": r["threads"], "kind": "oracle",
               "sample": f"{r['passes']:.1f} passes over the {r['pool']} query tokens of "
                         f"{spec.name}, all heads ({r['tokens']} token-evaluations, "
                         f"{r['seconds']:.1f} s of oracle time)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16", "data": "synthetic",
            "config": decode_config(spec, wl, ws),
            "gathered_tokens_per_s": ws * nvalid / t_step,
            "tflops_all_slots": ws * flops_all / t_step / 1e12,
            "kernel_ms": {"decode": statistics.mean(dec_ms),
                          "step_median": statistics.median(step_ms)},
            "wall_s_timed_region": wall,
            "roofline": ({"bound": "tensor", "achieved": achieved, "peak": peak,
                          "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                          "peak_kind": f"{peak_kind} bf16 burst",
                          "frac_of_sustained": achieved / float(peaks["bf16_tflops_sustained"]),
                          "alg_bytes_per_launch": alg_bytes,
                          "hbm_frac_alg_bytes": alg_bytes / t_dec / 1e9 / float(peaks["hbm_gbs"])}
                         if roofline_of(wl, t_dec, peaks)["bound"] == "tensor" else
                         {"bound": "hbm", "achieved": alg_bytes / t_dec / 1e9,
                          "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                          "frac": alg_bytes / t_dec / 1e9 / float(peaks["hbm_gbs"]),
                          "traffic": traffic, "peak_kind": f"{peak_kind} copy bandwidth",
                          "alg_bytes_per_launch": alg_bytes, "tflops": achieved}),
            "roofline_combined": roofline_of(wl, t_dec, peaks),
            "per_config": per_config,
            "cpu_baseline": cpu,
            "e2e": {"value": ws * flops / t_e2e / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": t_e2e * 1e3,
                    "serial_value": ws * flops / t_e2e_serial / 1e12,
                    "serial_ms_per_step": t_e2e_serial * 1e3,
                    "note": "q and indices host->device, out and lse device->host each step "
                            "(pinned buffers, the KV cache resident); steps pipelined: the "
                            "copies of neighbouring steps overlap a step's compute on their own "
                            "streams; four index sets in rotation keep the gathered rows out "
                            "of L2; serial_*: each step alone, copies and compute in turn"},
            # planner + decode (+ combine when a request is split) per timed step
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
