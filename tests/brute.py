"""Independent textbook attention used to pin the oracle (tests only).

Nothing here is shared with ``oracle/``: rows are decoded with torch's float8_e4m3fn and
bfloat16 views and numpy byte views (library routines), and attention is plain
``softmax(Q K^T * scale) V`` with numpy matmuls in float64.
"""

from __future__ import annotations

import numpy as np
import torch

PAGE = 64


def decode_rows_lib(rows_u8: np.ndarray) -> np.ndarray:
    """[n, 656] bytes -> [n, 576] float64 keys using torch/numpy views only."""
    rows_u8 = np.ascontiguousarray(rows_u8, dtype=np.uint8)
    n = rows_u8.shape[0]
    codes = torch.from_numpy(rows_u8[:, :512].copy()).view(torch.float8_e4m3fn)
    nope = codes.to(torch.float64).numpy().reshape(n, 4, 128)
    scales = rows_u8[:, 512:528].copy().view("<f4").astype(np.float64)  # [n, 4]
    rope = torch.from_numpy(rows_u8[:, 528:656].copy().view("<i2").copy()).view(
        torch.bfloat16).to(torch.float64).numpy()
    k = np.empty((n, 576), dtype=np.float64)
    k[:, :512] = (nope * scales[:, :, None]).reshape(n, 512)
    k[:, 512:] = rope
    return k


def q_lib(q_bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(q_bits).view(np.int16)).view(
        torch.bfloat16).to(torch.float64).numpy()


def sparse_attention(q_bits, kv, indices, sm_scale):
    """out [b, s_q, h, 512], lse [b, h, s_q] straight from the definition."""
    q = q_lib(q_bits)
    b, s_q, h, _ = q.shape
    kv = kv.reshape(-1, 656)
    nrows = kv.shape[0]
    out = np.zeros((b, s_q, h, 512))
    lse = np.full((b, h, s_q), np.inf)
    for bi in range(b):
        for si in range(s_q):
            idx = indices[bi, si]
            sel = idx[(idx >= 0) & (idx < nrows)]
            if sel.size == 0:
                continue
            k = decode_rows_lib(kv[sel])
            s = q[bi, si] @ k.T * sm_scale  # [h, n]
            m = s.max(axis=1, keepdims=True)
            e = np.exp(s - m)
            tot = e.sum(axis=1, keepdims=True)
            out[bi, si] = (e / tot) @ k[:, :512]
            lse[bi, :, si] = (m + np.log(tot))[:, 0]
    return out, lse


def dense_attention(q_bits, kv, block_table, ctx, sm_scale, seq):
    """Dense MLA over all ``ctx`` positions of sequence ``seq``, walking its page table:
    position p lives in physical page block_table[seq, p // 64], slot p % 64."""
    q = q_lib(q_bits)
    kv = kv.reshape(kv.shape[0], PAGE, 656)
    rows = np.stack([kv[block_table[seq, p // PAGE], p % PAGE] for p in range(ctx)])
    k = decode_rows_lib(rows)
    s = q[seq] @ k.T * sm_scale  # [s_q, h, ctx]
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    tot = e.sum(axis=-1, keepdims=True)
    return (e / tot) @ k[:, :512], (m + np.log(tot))[..., 0]
