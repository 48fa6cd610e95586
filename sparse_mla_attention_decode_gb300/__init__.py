"""Sparse MLA decode attention for NVIDIA GB300 (sm_103a).

A thin ctypes binding over ``libsparse_mla.so`` (C ABI in ``include/sparse_mla.h``): the
functions below carry the same names as the C entry points and only marshal arguments.
Every step of the computation runs in the library's CUDA kernels; there is no CPU or
PyTorch fallback, and calling into the library without the built extension raises.

PyTorch is used for device memory and streams only (``SparseMLADecode`` allocates the
caller-owned plan, workspace and outputs as torch tensors).
"""

from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "SMLA_OK", "SparseMLAError", "smla_dims", "lib", "build", "library_path",
    "sparse_mla_workspace_size", "sparse_mla_sched_meta", "sparse_mla_decode_fwd",
    "sparse_mla_combine", "sparse_mla_status_string", "sparse_mla_read_device_status",
    "sparse_mla_version", "sparse_mla_decode_static", "sparse_mla_static_read_status",
    "STATIC_SCRATCH_BYTES",
    "smla_decode_opts", "sparse_mla_decode_fwd_ex", "sparse_mla_combine_ex",
    "sparse_mla_plan_has_splits", "smla_topk_dims", "sparse_mla_topk_page_table",
    "topk_page_table", "SMLA_SCORES_BF16", "SMLA_SCORES_FP32",
    "smla_indexer_dims", "sparse_mla_indexer_scores", "indexer_scores",
    "sparse_mla_indexer_topk_scratch_size", "sparse_mla_indexer_topk", "indexer_topk",
    "SELECT_SCRATCH_BUDGET", "SparseMLADecode", "dims_for",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libsparse_mla.so")
_lock = threading.Lock()
_lib = None

SMLA_OK = 0
SMLA_ERR_WORKSPACE = 4
SMLA_ERR_TIMEOUT = 6
SMLA_DEV_TIMEOUT, SMLA_DEV_Q_RANGE, SMLA_DEV_SCALE_RANGE, SMLA_DEV_TOPK_TABLE = 0x1, 0x2, 0x4, 0x8
SMLA_DEV_NAN_INPUT = 0x10
# cache formats of smla_dims.kv_format / extra_kv_format
SMLA_KV_V32, SMLA_KV_V4, SMLA_KV_V41, SMLA_KV_V41_FP4 = 0, 1, 2, 3
_KV_FORMATS = {"v32": SMLA_KV_V32, "v4": SMLA_KV_V4, "v41": SMLA_KV_V41}
SMLA_SCORES_BF16, SMLA_SCORES_FP32 = 0, 1
EXPORTED = ["sparse_mla_workspace_size", "sparse_mla_sched_meta", "sparse_mla_decode_fwd",
            "sparse_mla_combine", "sparse_mla_status_string", "sparse_mla_read_device_status",
            "sparse_mla_version", "sparse_mla_decode_static", "sparse_mla_decode_fwd_ex",
            "sparse_mla_combine_ex", "sparse_mla_plan_has_splits", "sparse_mla_topk_page_table",
            "sparse_mla_indexer_scores", "sparse_mla_indexer_topk_scratch_size",
            "sparse_mla_indexer_topk", "sparse_mla_static_read_status"]
# Scratch budget of the chained selection (SMLA_SELECT_SCRATCH_BUDGET): scores kept in L2.
SELECT_SCRATCH_BUDGET = 48 << 20
# Size of the library-owned scratch of sparse_mla_decode_static (SMLA_STATIC_SCRATCH_BYTES).
STATIC_SCRATCH_BYTES = 48 << 20


class SparseMLAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {sparse_mla_status_string(code)} (status {code})")


class smla_dims(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int32), ("s_q", ctypes.c_int32), ("h_q", ctypes.c_int32),
                ("d_qk", ctypes.c_int32), ("d_v", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("page_block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int64),
                ("extra_topk", ctypes.c_int32), ("extra_num_blocks", ctypes.c_int64),
                ("kv_format", ctypes.c_int32), ("extra_kv_format", ctypes.c_int32)]


class smla_decode_opts(ctypes.Structure):
    """Optional decode inputs: device pointers (0 = variant off) to fp32 attn_sink [h_q] and
    int32 topk_length [b, s_q]; partials_bf16 != 0 keeps split partials in bf16; the extra
    cache (uint8 [extra_num_blocks, 64, 1, 656]), its indices (int32 [b, s_q, extra_topk]) and
    optional lengths (int32 [b, s_q])."""
    _fields_ = [("attn_sink", ctypes.c_void_p), ("topk_length", ctypes.c_void_p),
                ("partials_bf16", ctypes.c_int32), ("extra_kv_cache", ctypes.c_void_p),
                ("extra_indices", ctypes.c_void_p), ("extra_topk_length", ctypes.c_void_p),
                ("test_stall", ctypes.c_int32)]


class smla_topk_dims(ctypes.Structure):
    _fields_ = [("n_tok", ctypes.c_int32), ("s_q", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("ld", ctypes.c_int32), ("max_pages", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class smla_indexer_dims(ctypes.Structure):
    _fields_ = [("n_tok", ctypes.c_int32), ("s_q", ctypes.c_int32), ("heads", ctypes.c_int32),
                ("dim", ctypes.c_int32), ("max_pages", ctypes.c_int32), ("ld", ctypes.c_int32),
                ("num_pages", ctypes.c_int64), ("test_stall", ctypes.c_int32)]


def library_path() -> str:
    return _LIB_PATH


def build(force: bool = False) -> str:
    from . import _build
    return _build.build(force=force)


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"{_LIB_PATH} is missing: build it first (sparse_mla_attention_decode_gb300."
                    "build() or __graft_entry__.build()); there is no fallback path")
            L = ctypes.CDLL(_LIB_PATH)
            P = ctypes.POINTER
            vp, sz = ctypes.c_void_p, ctypes.c_size_t
            L.sparse_mla_workspace_size.argtypes = [P(smla_dims), ctypes.c_int, P(sz), P(sz)]
            L.sparse_mla_sched_meta.argtypes = [P(smla_dims), ctypes.c_int, vp, sz, vp]
            L.sparse_mla_decode_fwd.argtypes = [P(smla_dims), ctypes.c_int, vp, vp, vp,
                                                ctypes.c_float, vp, vp, sz, vp, vp, vp]
            L.sparse_mla_combine.argtypes = [P(smla_dims), ctypes.c_int, vp, vp, sz, vp, vp, vp]
            L.sparse_mla_decode_fwd_ex.argtypes = [P(smla_dims), ctypes.c_int, vp, vp, vp,
                                                   ctypes.c_float, P(smla_decode_opts), vp, vp,
                                                   sz, vp, vp, vp]
            L.sparse_mla_combine_ex.argtypes = [P(smla_dims), ctypes.c_int, P(smla_decode_opts),
                                                vp, vp, sz, vp, vp, vp]
            L.sparse_mla_plan_has_splits.argtypes = [P(smla_dims), ctypes.c_int, P(ctypes.c_int)]
            L.sparse_mla_topk_page_table.argtypes = [P(smla_topk_dims), vp, vp, vp, vp, vp, vp]
            L.sparse_mla_indexer_scores.argtypes = [P(smla_indexer_dims), ctypes.c_int, vp, vp, vp,
                                                    vp, vp, vp, vp, vp]
            L.sparse_mla_indexer_topk_scratch_size.argtypes = [P(smla_indexer_dims), P(sz)]
            L.sparse_mla_indexer_topk.argtypes = [P(smla_indexer_dims), ctypes.c_int32, ctypes.c_int,
                                                  vp, vp, vp, vp, vp, vp, sz, vp, vp, vp]
            L.sparse_mla_status_string.argtypes = [ctypes.c_int]
            L.sparse_mla_status_string.restype = ctypes.c_char_p
            L.sparse_mla_read_device_status.argtypes = [P(smla_dims), ctypes.c_int, vp,
                                                        P(ctypes.c_int), vp]
            L.sparse_mla_version.restype = ctypes.c_char_p
            L.sparse_mla_decode_static.argtypes = [P(smla_dims), ctypes.c_int, vp, vp, vp,
                                                   ctypes.c_float, vp, vp, vp]
            L.sparse_mla_static_read_status.argtypes = [P(smla_dims), ctypes.c_int,
                                                        P(ctypes.c_int), vp]
            for f in EXPORTED:
                if f not in ("sparse_mla_status_string", "sparse_mla_version"):
                    getattr(L, f).restype = ctypes.c_int
            _lib = L
    return _lib


def _check(rc: int, where: str) -> None:
    if rc != SMLA_OK:
        raise SparseMLAError(rc, where)


def sparse_mla_status_string(code: int) -> str:
    return lib().sparse_mla_status_string(int(code)).decode()


def sparse_mla_version() -> str:
    return lib().sparse_mla_version().decode()


def sparse_mla_workspace_size(dims: smla_dims, num_sms: int = 0) -> tuple[int, int]:
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().sparse_mla_workspace_size(ctypes.byref(dims), int(num_sms), ctypes.byref(a),
                                           ctypes.byref(b)), "sparse_mla_workspace_size")
    return a.value, b.value


def sparse_mla_sched_meta(dims: smla_dims, num_sms: int, sched_meta: int, sched_bytes: int,
                          stream: int = 0) -> None:
    _check(lib().sparse_mla_sched_meta(ctypes.byref(dims), int(num_sms), sched_meta,
                                       int(sched_bytes), stream), "sparse_mla_sched_meta")


def sparse_mla_decode_fwd(dims: smla_dims, num_sms: int, q: int, kv_cache: int, indices: int,
                          sm_scale: float, sched_meta: int, workspace: int, workspace_bytes: int,
                          out: int, lse: int, stream: int = 0) -> None:
    _check(lib().sparse_mla_decode_fwd(ctypes.byref(dims), int(num_sms), q, kv_cache, indices,
                                       float(sm_scale), sched_meta, workspace,
                                       int(workspace_bytes), out, lse, stream),
           "sparse_mla_decode_fwd")


def sparse_mla_combine(dims: smla_dims, num_sms: int, sched_meta: int, workspace: int,
                       workspace_bytes: int, out: int, lse: int, stream: int = 0) -> None:
    _check(lib().sparse_mla_combine(ctypes.byref(dims), int(num_sms), sched_meta, workspace,
                                    int(workspace_bytes), out, lse, stream),
           "sparse_mla_combine")


def sparse_mla_decode_fwd_ex(dims: smla_dims, num_sms: int, q: int, kv_cache: int, indices: int,
                             sm_scale: float, opts, sched_meta: int, workspace: int,
                             workspace_bytes: int, out: int, lse: int, stream: int = 0) -> None:
    _check(lib().sparse_mla_decode_fwd_ex(ctypes.byref(dims), int(num_sms), q, kv_cache, indices,
                                          float(sm_scale),
                                          None if opts is None else ctypes.byref(opts),
                                          sched_meta, workspace, int(workspace_bytes), out, lse,
                                          stream),
           "sparse_mla_decode_fwd_ex")


def sparse_mla_combine_ex(dims: smla_dims, num_sms: int, opts, sched_meta: int, workspace: int,
                          workspace_bytes: int, out: int, lse: int, stream: int = 0) -> None:
    _check(lib().sparse_mla_combine_ex(ctypes.byref(dims), int(num_sms),
                                       None if opts is None else ctypes.byref(opts), sched_meta,
                                       workspace, int(workspace_bytes), out, lse, stream),
           "sparse_mla_combine_ex")


def sparse_mla_decode_static(dims: smla_dims, num_sms: int, q: int, kv_cache: int,
                             indices: int, sm_scale: float, out: int, lse: int,
                             stream: int = 0) -> None:
    """Plan + decode + combine on the library's own fixed scratch (no caller buffers).

    For callers that cannot allocate device memory.  Calls on one device share the scratch,
    so their executions must not overlap; the first call on a device should come before
    any stream capture.  Problems above STATIC_SCRATCH_BYTES are rejected.
    """
    rc = lib().sparse_mla_decode_static(ctypes.byref(dims), int(num_sms), q, kv_cache, indices,
                                        float(sm_scale), out, lse, stream)
    if rc == SMLA_ERR_WORKSPACE:
        sb, ab = sparse_mla_workspace_size(dims, num_sms)
        need = ((ab + 255) // 256) * 256 + sb
        raise SparseMLAError(rc, f"sparse_mla_decode_static: the problem needs {need} bytes of "
                                 f"scratch, the fixed scratch holds {STATIC_SCRATCH_BYTES}")
    _check(rc, "sparse_mla_decode_static")


def sparse_mla_static_read_status(dims: smla_dims, num_sms: int, stream: int = 0) -> tuple[int, int]:
    """(status code of the call, device status word) of the last sparse_mla_decode_static call
    with these sizes on the current device."""
    code = ctypes.c_int()
    rc = lib().sparse_mla_static_read_status(ctypes.byref(dims), int(num_sms), ctypes.byref(code),
                                             stream)
    return rc, code.value


def sparse_mla_plan_has_splits(dims: smla_dims, num_sms: int) -> bool:
    """Whether the plan splits any request (host-only; then sparse_mla_combine has work)."""
    v = ctypes.c_int()
    _check(lib().sparse_mla_plan_has_splits(ctypes.byref(dims), int(num_sms), ctypes.byref(v)),
           "sparse_mla_plan_has_splits")
    return bool(v.value)


def sparse_mla_topk_page_table(dims: smla_topk_dims, scores: int, valid_len: int,
                               block_table: int, out_indices: int, status: int = 0,
                               stream: int = 0) -> None:
    _check(lib().sparse_mla_topk_page_table(ctypes.byref(dims), scores, valid_len, block_table,
                                            out_indices, status or None, stream),
           "sparse_mla_topk_page_table")


def topk_page_table(scores, valid_len, block_table, s_q: int, k: int, out=None, status=None,
                    stream=None):
    """Exact top-k of each row of ``scores`` (bf16 or fp32 [n_tok, ld] device tensor) over its
    first valid_len[t] positions, as physical ids through ``block_table`` (int32 [b, pages];
    row t uses request t // s_q): int32 [n_tok, k], -1 after the selected ids."""
    import torch
    if scores.dim() != 2 or scores.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("scores must be a 2-D bf16 or fp32 tensor")
    if scores.stride(1) != 1:
        raise ValueError("scores rows must be contiguous")
    for name, t in (("valid_len", valid_len), ("block_table", block_table)):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 tensor")
    n_tok = scores.shape[0]
    if out is None:
        out = torch.empty(n_tok, k, dtype=torch.int32, device=scores.device)
    d = smla_topk_dims(n_tok, s_q, k, scores.stride(0), block_table.shape[1],
                       SMLA_SCORES_FP32 if scores.dtype == torch.float32 else SMLA_SCORES_BF16)
    st = (stream if stream is not None else torch.cuda.current_stream(scores.device)).cuda_stream
    sparse_mla_topk_page_table(d, scores.data_ptr(), valid_len.data_ptr(), block_table.data_ptr(),
                               out.data_ptr(), status.data_ptr() if status is not None else 0, st)
    return out


def sparse_mla_indexer_scores(dims: smla_indexer_dims, num_sms: int, q8: int, weights: int,
                              k_cache: int, block_table: int, valid_len: int, scores: int,
                              status: int = 0, stream: int = 0) -> None:
    _check(lib().sparse_mla_indexer_scores(ctypes.byref(dims), int(num_sms), q8, weights, k_cache,
                                           block_table, valid_len, scores, status or None,
                                           stream),
           "sparse_mla_indexer_scores")


def indexer_scores(q8, weights, k_cache, block_table, valid_len, s_q: int, ld: int, out=None,
                   status=None, num_sms: int = 0, stream=None):
    """Indexer scores fp32 [n_tok, ld] (written for s < valid_len[t]) from e4m3 codes q8
    (uint8 [n_tok, 64, 128]), fp32 weights [n_tok, 64], the paged key cache (uint8
    [num_pages, 8448]) and the page table (int32 [n_tok / s_q, max_pages])."""
    import torch
    for name, t, dt in (("q8", q8, torch.uint8), ("weights", weights, torch.float32),
                        ("k_cache", k_cache, torch.uint8), ("block_table", block_table, torch.int32),
                        ("valid_len", valid_len, torch.int32)):
        if t.dtype != dt or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {dt} tensor")
    n_tok = q8.shape[0]
    if out is None:
        out = torch.empty(n_tok, ld, dtype=torch.float32, device=q8.device)
    d = smla_indexer_dims(n_tok, s_q, 64, 128, block_table.shape[1], ld, k_cache.shape[0])
    st = (stream if stream is not None else torch.cuda.current_stream(q8.device)).cuda_stream
    sparse_mla_indexer_scores(d, num_sms, q8.data_ptr(), weights.data_ptr(), k_cache.data_ptr(),
                              block_table.data_ptr(), valid_len.data_ptr(), out.data_ptr(),
                              status.data_ptr() if status is not None else 0, st)
    return out


def sparse_mla_indexer_topk_scratch_size(dims: smla_indexer_dims) -> int:
    n = ctypes.c_size_t()
    _check(lib().sparse_mla_indexer_topk_scratch_size(ctypes.byref(dims), ctypes.byref(n)),
           "sparse_mla_indexer_topk_scratch_size")
    return n.value


def sparse_mla_indexer_topk(dims: smla_indexer_dims, topk: int, num_sms: int, q8: int,
                            weights: int, k_cache: int, block_table: int, valid_len: int,
                            scratch: int, scratch_bytes: int, out_indices: int, status: int = 0,
                            stream: int = 0) -> None:
    _check(lib().sparse_mla_indexer_topk(ctypes.byref(dims), int(topk), int(num_sms), q8, weights,
                                         k_cache, block_table, valid_len, scratch,
                                         int(scratch_bytes), out_indices, status or None, stream),
           "sparse_mla_indexer_topk")


def indexer_topk(q8, weights, k_cache, block_table, valid_len, s_q: int, ld: int, k: int,
                 out=None, scratch=None, status=None, num_sms: int = 0, stream=None):
    """The indexer scores and their exact top-k chained (int32 ids [n_tok, k], -1 padding)
    without the [n_tok, ld] score matrix: the scores of one run of tokens at a time live in
    ``scratch`` (a contiguous device tensor; by default uint8 of the size the library asks
    for)."""
    import torch
    for name, t, dt in (("q8", q8, torch.uint8), ("weights", weights, torch.float32),
                        ("k_cache", k_cache, torch.uint8), ("block_table", block_table, torch.int32),
                        ("valid_len", valid_len, torch.int32)):
        if t.dtype != dt or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {dt} tensor")
    n_tok = q8.shape[0]
    d = smla_indexer_dims(n_tok, s_q, 64, 128, block_table.shape[1], ld, k_cache.shape[0])
    if scratch is None:
        scratch = torch.empty(sparse_mla_indexer_topk_scratch_size(d), dtype=torch.uint8,
                              device=q8.device)
    elif not scratch.is_contiguous():
        raise ValueError("scratch must be contiguous")
    if out is None:
        out = torch.empty(n_tok, k, dtype=torch.int32, device=q8.device)
    if status is None:  # the chained call needs a status word; this one is not read back
        status = torch.zeros(1, dtype=torch.int32, device=q8.device)
    st = (stream if stream is not None else torch.cuda.current_stream(q8.device)).cuda_stream
    sparse_mla_indexer_topk(d, k, num_sms, q8.data_ptr(), weights.data_ptr(), k_cache.data_ptr(),
                            block_table.data_ptr(), valid_len.data_ptr(), scratch.data_ptr(),
                            scratch.numel() * scratch.element_size(), out.data_ptr(),
                            status.data_ptr(), st)
    return out


def sparse_mla_read_device_status(dims: smla_dims, num_sms: int, sched_meta: int,
                                  stream: int = 0) -> tuple[int, int]:
    """(status code of the call, device status word)."""
    code = ctypes.c_int()
    rc = lib().sparse_mla_read_device_status(ctypes.byref(dims), int(num_sms), sched_meta,
                                             ctypes.byref(code), stream)
    return rc, code.value


def dims_for(b: int, s_q: int, h_q: int, topk: int, num_blocks: int, extra_topk: int = 0,
             extra_num_blocks: int = 0, kv_format: str = "v32") -> smla_dims:
    """Problem sizes; kv_format "v32" (656-byte rows, d_qk 576), "v4" or "v41" (d_qk 512; the
    extra cache of a "v41" cache is FP4)."""
    f = _KV_FORMATS[kv_format]
    return smla_dims(b, s_q, h_q, 576 if f == SMLA_KV_V32 else 512, 512, topk, 64, num_blocks,
                     extra_topk, extra_num_blocks, f,
                     SMLA_KV_V41_FP4 if f == SMLA_KV_V41 else SMLA_KV_V32)


class SparseMLADecode:
    """Owns the plan and workspace buffers of one problem shape and runs the three calls.

    q: bf16 [b, s_q, h_q, d_qk]; kv_cache: uint8 pages (656-byte rows, [num_blocks, 64, 1,
    656], or ``kv_format`` "v4" / "v41": [num_blocks, 64 * 584] / [num_blocks, 64 * 528], data
    rows then scale rows); indices: int32 [b, s_q, topk]; returns (out bf16 [b, s_q, h_q,
    512], lse fp32 [b, h_q, s_q]).
    Optional ``attn_sink`` (fp32 [h_q]) and ``topk_length`` (int32 [b, s_q]) device tensors
    and ``partials_bf16`` select the decode variants of ``smla_decode_opts``; a problem built
    with ``extra_topk`` > 0 takes ``extra_kv`` (uint8 [extra_num_blocks, 64, 1, 656]),
    ``extra_indices`` (int32 [b, s_q, extra_topk]) and optionally ``extra_topk_length``.
    """

    def __init__(self, b: int, s_q: int, h_q: int, topk: int, num_blocks: int, device=None,
                 num_sms: int = 0, extra_topk: int = 0, extra_num_blocks: int = 0,
                 kv_format: str = "v32"):
        import torch
        self.device = torch.device(device if device is not None else "cuda")
        if num_sms <= 0:
            num_sms = torch.cuda.get_device_properties(self.device).multi_processor_count
        self.num_sms = int(num_sms)
        self.dims = dims_for(b, s_q, h_q, topk, num_blocks, extra_topk, extra_num_blocks,
                             kv_format)
        sb, ab = sparse_mla_workspace_size(self.dims, self.num_sms)
        self.sched_bytes, self.accum_bytes = sb, ab
        self.sched = torch.empty(max(sb, 16), dtype=torch.uint8, device=self.device)
        self.workspace = torch.empty(max(ab, 16), dtype=torch.uint8, device=self.device)

    def run(self, q, kv_cache, indices, sm_scale: float, out=None, lse=None, stream=None,
            attn_sink=None, topk_length=None, partials_bf16: bool = False, extra_kv=None,
            extra_indices=None, extra_topk_length=None):
        import torch
        d = self.dims
        if out is None:
            out = torch.empty(d.b, d.s_q, d.h_q, 512, dtype=torch.bfloat16, device=self.device)
        if lse is None:
            lse = torch.empty(d.b, d.h_q, d.s_q, dtype=torch.float32, device=self.device)
        st = (stream if stream is not None else torch.cuda.current_stream(self.device)).cuda_stream
        for name, t in (("q", q), ("kv_cache", kv_cache), ("indices", indices), ("out", out),
                        ("lse", lse)):
            if not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous")
        opts = None
        if d.extra_topk > 0 and extra_indices is None:
            raise ValueError("this problem has an extra list: pass extra_kv and extra_indices")
        for name, t in (("extra_kv", extra_kv), ("extra_indices", extra_indices),
                        ("extra_topk_length", extra_topk_length)):
            if t is not None and not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous")
        if (attn_sink is not None or topk_length is not None or partials_bf16
                or extra_indices is not None):
            if attn_sink is not None and (attn_sink.dtype != torch.float32
                                          or attn_sink.numel() != d.h_q
                                          or not attn_sink.is_contiguous()):
                raise ValueError("attn_sink must be a contiguous fp32 tensor of h_q values")
            if topk_length is not None and (topk_length.dtype != torch.int32
                                            or topk_length.numel() != d.b * d.s_q
                                            or not topk_length.is_contiguous()):
                raise ValueError("topk_length must be a contiguous int32 tensor [b, s_q]")
            opts = smla_decode_opts(
                attn_sink.data_ptr() if attn_sink is not None else None,
                topk_length.data_ptr() if topk_length is not None else None,
                1 if partials_bf16 else 0,
                extra_kv.data_ptr() if extra_kv is not None else None,
                extra_indices.data_ptr() if extra_indices is not None else None,
                extra_topk_length.data_ptr() if extra_topk_length is not None else None)
        sparse_mla_sched_meta(d, self.num_sms, self.sched.data_ptr(), self.sched_bytes, st)
        sparse_mla_decode_fwd_ex(d, self.num_sms, q.data_ptr(), kv_cache.data_ptr(),
                                 indices.data_ptr(), sm_scale, opts, self.sched.data_ptr(),
                                 self.workspace.data_ptr(), self.accum_bytes, out.data_ptr(),
                                 lse.data_ptr(), st)
        sparse_mla_combine_ex(d, self.num_sms, opts, self.sched.data_ptr(),
                              self.workspace.data_ptr(), self.accum_bytes, out.data_ptr(),
                              lse.data_ptr(), st)
        return out, lse

    def device_status(self, stream=None) -> int:
        import torch
        st = (stream if stream is not None else torch.cuda.current_stream(self.device)).cuda_stream
        rc, word = sparse_mla_read_device_status(self.dims, self.num_sms, self.sched.data_ptr(), st)
        return word

    def plan(self):
        """(meta int32 [parts, 8], num_splits prefix int32 [b + 1]) copied to the host."""
        parts = max(self.num_sms // max(self.dims.s_q, 1) // 2, 1)
        raw = self.sched.cpu()
        meta = raw[: parts * 32].view(dtype=__import__("torch").int32).view(parts, 8)
        pre = raw[parts * 32: parts * 32 + (self.dims.b + 1) * 4].view(
            dtype=__import__("torch").int32)
        return meta, pre
