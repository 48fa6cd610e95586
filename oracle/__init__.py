"""Plain CPU oracle for sparse MLA decode attention (fp64).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference legs may import this package.  The CUDA library and
its Python binding never import it, and it imports nothing from them: the two share no
code, header, table or constant.

* ``sparse_mla_oracle.c`` -- e4m3 / bf16 field decoders, the 656-byte row decoder and the
  sparse attention definition in fp64 (C with OpenMP, built by :func:`build`).
* ``sched.py`` -- the greedy split-KV partition planner.
* ``combine.py`` -- the LSE-weighted merge of split partials.
* ``online.py`` -- the base-2 online softmax recurrence, step by step.
* ``variants.py`` -- per-token top-k length masking and the attention-sink output factor.
* ``formats.py`` -- the later cache formats (V4, V4.1, FP4 extra: structure-of-arrays pages,
  e8m0 / e4m3 group scales, d_qk = d_v = 512) decoded and attended in numpy.

Parity status: every function here is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle*.py`` (worked-example values from the pages, closed forms, brute force
against an independent numpy path, invariants).  No function is "parity unpinned".
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import combine, online, sched, variants  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sparse_mla_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

D_QK, D_V, ROW_BYTES = 576, 512, 656


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (portable flags only; no -march=native)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O3", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o",
                               tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.smla_oracle_e4m3.restype = ctypes.c_double
            lib.smla_oracle_e4m3.argtypes = [ctypes.c_uint8]
            lib.smla_oracle_bf16.restype = ctypes.c_double
            lib.smla_oracle_bf16.argtypes = [ctypes.c_uint16]
            lib.smla_oracle_e4m3_array.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                                                   ctypes.c_int64]
            lib.smla_oracle_bf16_array.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                                                   ctypes.c_int64]
            lib.smla_oracle_decode_row.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
            lib.smla_oracle_max_threads.restype = ctypes.c_int
            lib.smla_oracle_sparse_decode.restype = ctypes.c_int
            lib.smla_oracle_sparse_decode.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_double, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def max_threads() -> int:
    return int(_load().smla_oracle_max_threads())


def e4m3_decode(codes) -> np.ndarray:
    """Decode e4m3 codes (uint8 array) to fp64 from their integer fields."""
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.empty(c.shape, dtype=np.float64)
    _load().smla_oracle_e4m3_array(_ptr(c), _ptr(out), c.size)
    return out


def bf16_decode(bits) -> np.ndarray:
    """Decode bf16 bit patterns (uint16 array) to fp64 from their fields."""
    c = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    out = np.empty(c.shape, dtype=np.float64)
    _load().smla_oracle_bf16_array(_ptr(c), _ptr(out), c.size)
    return out


def decode_row(row: np.ndarray) -> np.ndarray:
    """The 576 key dims of one 656-byte row (the first 512 are also the value)."""
    r = np.ascontiguousarray(np.asarray(row, dtype=np.uint8))
    assert r.size == ROW_BYTES
    out = np.empty(D_QK, dtype=np.float64)
    _load().smla_oracle_decode_row(_ptr(r), _ptr(out))
    return out


def sparse_mla_decode(q_bits: np.ndarray, kv: np.ndarray, indices: np.ndarray, sm_scale: float,
                      tokens=None, slot_range=None, threads: int = 0, attn_sink=None,
                      topk_length=None, extra_kv=None, extra_indices=None,
                      extra_topk_length=None):
    """Sparse MLA decode in fp64.

    q_bits:  uint16 bf16 bit patterns [b, s_q, h_q, 576]
    kv:      uint8 [num_blocks, page_block_size, 656] (an h_kv = 1 axis may be present)
    indices: int32 [b, s_q, topk]
    tokens:  optional list of flattened query-token ids (bi * s_q + si); default all
    slot_range: optional (begin, end) sub-range of the top-k slots (one split's share)
    attn_sink:   optional per-head sink values [h_q] (``variants``); whole rows only
    topk_length: optional per-token valid prefix lengths [b, s_q] (``variants``)
    extra_kv, extra_indices, extra_topk_length: optional second cache and slot list, joined
                 after the main list (``variants.join_extra``); slot_range then indexes the
                 joined list

    Returns (out fp64 [n_tok, h_q, 512], lse fp64 [n_tok, h_q], n_valid int32 [n_tok])
    where n_tok runs over ``tokens`` in order.
    """
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    b, s_q, h_q, d = q_bits.shape
    assert d == D_QK
    kv = np.ascontiguousarray(kv, dtype=np.uint8)
    assert kv.shape[-1] == ROW_BYTES
    num_blocks, page = kv.shape[0], kv.shape[1]
    if topk_length is not None:
        indices = variants.mask_beyond_length(indices, topk_length)
    if extra_indices is not None:
        kv, indices = variants.join_extra(kv, indices, extra_kv, extra_indices, extra_topk_length)
        num_blocks, page = kv.shape[0], kv.shape[1]
    indices = np.ascontiguousarray(indices, dtype=np.int32)
    assert indices.shape[:2] == (b, s_q)
    topk = indices.shape[2]
    if tokens is None:
        tokens = np.arange(b * s_q, dtype=np.int32)
    tokens = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    lo, hi = (0, topk) if slot_range is None else slot_range
    n = tokens.size
    out = np.empty((n, h_q, D_V), dtype=np.float64)
    lse = np.empty((n, h_q), dtype=np.float64)
    nv = np.empty(n, dtype=np.int32)
    rc = _load().smla_oracle_sparse_decode(b, s_q, h_q, topk, num_blocks, page, _ptr(q_bits),
                                           _ptr(kv), _ptr(indices), float(sm_scale),
                                           _ptr(tokens), n, int(lo), int(hi), _ptr(out),
                                           _ptr(lse), _ptr(nv), int(threads))
    if rc != 0:
        raise MemoryError("oracle allocation failed")
    if attn_sink is not None:
        assert slot_range is None, "the sink scales whole rows, not one split's share"
        sink = np.asarray(attn_sink, dtype=np.float64).reshape(1, h_q)
        out *= variants.sink_factor(lse, sink)[:, :, None]
    return out, lse, nv


def sparse_mla_decode_full(q_bits, kv, indices, sm_scale, threads: int = 0, attn_sink=None,
                           topk_length=None, extra_kv=None, extra_indices=None,
                           extra_topk_length=None):
    """Whole-problem form with the library's output layouts: out [b, s_q, h_q, 512],
    lse [b, h_q, s_q]."""
    b, s_q, h_q, _ = q_bits.shape
    out, lse, _ = sparse_mla_decode(q_bits, kv, indices, sm_scale, threads=threads,
                                    attn_sink=attn_sink, topk_length=topk_length,
                                    extra_kv=extra_kv, extra_indices=extra_indices,
                                    extra_topk_length=extra_topk_length)
    return out.reshape(b, s_q, h_q, D_V), lse.reshape(b, s_q, h_q).transpose(0, 2, 1).copy()
