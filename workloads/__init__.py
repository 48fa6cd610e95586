"""Seeded synthetic inputs for sparse MLA decode over a paged FP8 KV cache.

This module builds INPUTS only.  It holds none of the attention arithmetic; the CUDA
library and the CPU oracle both consume what it makes, and neither is imported here.

Row format ("FlashMLA 与 DSA：内核、流水线和正确性边界", section 3.1; "FlashMLA Sparse
Decode 完整计算过程详解", steps 2.2, 4.2 and 4.3): 656 bytes per token = 512 e4m3 codes of
the NoPE part, 4 little-endian fp32 scales (one per 128-dim group; the stored value is
the dequant multiplier), 64 bf16 RoPE values stored as is.

Quantiser (input preparation, step 4.2 of the second page): per 128-dim group,
``scale = amax / 448`` in fp32, or the power of two ``2^ceil(log2(amax / 448))`` for
ue8m0-style scales; ``code = rn_e4m3(x / scale)`` with the quotient in fp32, saturated to
+-448; an all-zero group gets scale 1.

Indices are physical token ids ``page * 64 + offset`` reached through a per-sequence page
table whose pages are scattered at random over a shared pool.

Later formats ("FlashMLA 与 DSA", sections 3.1 and 6.4; d_qk = 512): a page of 64 tokens holds
the 64 data rows, then the 64 scale rows.  V4: 448 e4m3 NoPE codes + 64 bf16 RoPE values, then
7 e8m0 scales (per 64 NoPE dims) + 1 zero pad byte (584 bytes a token).  V4.1: 512 e4m3 codes,
then 16 e8m0 scales (per 32 dims) (528).  FP4 (extra cache only): 512 e2m1 values, two per
byte with the even element in the low nibble, then 32 e4m3 scales (per 16 dims) (288).
Quantisers: e8m0 scale = the power of two 2^ceil(log2(amax / 448)) (1 for an all-zero group),
code = rn_e4m3(x / scale); FP4 scale = rn_e4m3(amax / 6) (1 for an all-zero group), code =
the nearest e2m1 value of x / scale (ties to the even code, saturating at 6).

The five benchmark workloads (``CONFIGS``) follow the configuration list this project is
measured on; ``seed`` is the config's position 0..4.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

D_NOPE, D_ROPE, D_QK, D_V = 512, 64, 576, 512
GROUP = 128
ROW_BYTES = 656
PAGE = 64
E4M3_MAX = 448.0


@dataclass
class Spec:
    name: str
    b: int
    s_q: int
    h_q: int
    topk: int
    ctx: int  # tokens per sequence
    ue8m0: bool = False
    masked_per_row: int = 0  # exactly this many slots per row set to -1
    causal_base: int | None = None  # query token i sees positions [0, causal_base + i]
    sort_indices: bool = False  # sort each row ascending by physical id
    extra_pool_pages: int = 0
    seed: int = 0
    kv_format: str = "v32"  # "v32" (656-byte rows, d_qk 576), "v4" or "v41" (d_qk 512)

    @property
    def d_qk(self) -> int:
        return D_QK if self.kv_format == "v32" else 512

    @property
    def pages_per_seq(self) -> int:
        return -(-self.ctx // PAGE)

    @property
    def num_blocks(self) -> int:
        return self.b * self.pages_per_seq + self.extra_pool_pages


CONFIGS: dict[str, Spec] = {
    # b=2, s_q=1, h=128, topk=128, 4096-token context per sequence.
    "c1_b2_h128_k128": Spec("c1_b2_h128_k128", b=2, s_q=1, h_q=128, topk=128, ctx=4096, seed=0),
    # b=64, h=128, topk=2048, 32768-token context, 5% (102) slots per row masked.
    "c2_b64_h128_k2048_mask5": Spec("c2_b64_h128_k2048_mask5", b=64, s_q=1, h_q=128,
                                    topk=2048, ctx=32768, masked_per_row=102, seed=1),
    # h=64, b=128, s_q=2 (multi-token decode), 65536-token context, causal prefix.
    "c3_b128_sq2_h64_k2048": Spec("c3_b128_sq2_h64_k2048", b=128, s_q=2, h_q=64, topk=2048,
                                  ctx=65536, causal_base=65534, seed=2),
    # ue8m0 power-of-two scales, b=32, 131072-token context; sorted and permuted indices.
    "c4_b32_h128_k2048_ue8m0_sorted": Spec("c4_b32_h128_k2048_ue8m0_sorted", b=32, s_q=1,
                                           h_q=128, topk=2048, ctx=131072, ue8m0=True,
                                           sort_indices=True, seed=3),
    "c4_b32_h128_k2048_ue8m0_perm": Spec("c4_b32_h128_k2048_ue8m0_perm", b=32, s_q=1,
                                         h_q=128, topk=2048, ctx=131072, ue8m0=True, seed=3),
    # prefill-shaped: b=1, s_q=4096, h=128, topk=2048 from a 65536-token context, causal
    # (query i sees [0, 61440 + i]).
    "c5_b1_sq4096_h128_k2048": Spec("c5_b1_sq4096_h128_k2048", b=1, s_q=4096, h_q=128,
                                    topk=2048, ctx=65536, causal_base=61440, seed=4),
}


# The decode-shaped workload in the later cache formats (d_qk = 512): measured beside the five
# configurations above, not part of their list.
FORMAT_CONFIGS: dict[str, Spec] = {
    "c2fmt_b64_h128_k2048_mask5_v41": Spec("c2fmt_b64_h128_k2048_mask5_v41", b=64, s_q=1,
                                           h_q=128, topk=2048, ctx=32768, masked_per_row=102,
                                           seed=1, kv_format="v41"),
    "c2fmt_b64_h128_k2048_mask5_v4": Spec("c2fmt_b64_h128_k2048_mask5_v4", b=64, s_q=1,
                                          h_q=128, topk=2048, ctx=32768, masked_per_row=102,
                                          seed=1, kv_format="v4"),
}


@dataclass
class Workload:
    spec: Spec
    q: torch.Tensor  # bf16 [b, s_q, h_q, 576]
    kv: torch.Tensor  # uint8 [num_blocks, 64, 1, 656]
    indices: torch.Tensor  # int32 [b, s_q, topk]
    block_table: torch.Tensor  # int32 [b, pages_per_seq]
    sm_scale: float
    extras: dict = field(default_factory=dict)

    @property
    def num_valid(self) -> int:
        nb = self.kv.shape[0] * PAGE
        i = self.indices
        return int(((i >= 0) & (i < nb)).sum().item())


def ue8m0_scale(amax_over_max: torch.Tensor) -> torch.Tensor:
    """2^ceil(log2(v)) for positive fp32 v, exactly (via frexp)."""
    m, e = torch.frexp(amax_over_max)
    e = torch.where(m == 0.5, e - 1, e)
    return torch.ldexp(torch.ones_like(amax_over_max), e)


def quantize_rows(x: torch.Tensor, ue8m0: bool = False) -> torch.Tensor:
    """bf16 [N, 576] -> uint8 [N, 656] in the FP8 row format."""
    assert x.dtype == torch.bfloat16 and x.shape[-1] == D_QK
    n = x.shape[0]
    nope = x[:, :D_NOPE].float().view(n, D_NOPE // GROUP, GROUP)
    amax = nope.abs().amax(dim=-1)
    ratio = amax / E4M3_MAX
    scale = ue8m0_scale(ratio) if ue8m0 else ratio
    scale = torch.where(amax == 0, torch.ones_like(scale), scale).float()
    q = (nope / scale[..., None]).clamp_(-E4M3_MAX, E4M3_MAX)
    codes = q.to(torch.float8_e4m3fn).view(torch.uint8).view(n, D_NOPE)
    out = torch.empty(n, ROW_BYTES, dtype=torch.uint8, device=x.device)
    out[:, :D_NOPE] = codes
    out[:, D_NOPE:D_NOPE + 16] = scale.contiguous().view(torch.uint8).view(n, 16)
    out[:, D_NOPE + 16:] = x[:, D_NOPE:].contiguous().view(torch.uint8).view(n, 2 * D_ROPE)
    return out


# bytes of one token's data row and scale row in the later formats
FMT_BYTES = {"v4": (448 + 2 * D_ROPE, 8), "v41": (512, 16), "v41_fp4": (256, 32)}


def _e8m0_codes(amax: torch.Tensor) -> tuple[torch.Tensor, torch.Tensor]:
    """(scale fp32, e8m0 byte) per group: the power of two 2^ceil(log2(amax / 448))."""
    scale = ue8m0_scale(amax / E4M3_MAX)
    scale = torch.where(amax == 0, torch.ones_like(scale), scale).float()
    code = ((scale.view(torch.int32) >> 23) & 0xFF).to(torch.uint8)
    return scale, code


def _e4m3(x: torch.Tensor) -> torch.Tensor:
    return x.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)


def _e2m1(v: torch.Tensor) -> torch.Tensor:
    """Nearest e2m1 code of each value (ties to the even code, saturating at 6)."""
    a = v.abs()
    c = ((a > 0.25).int() + (a >= 0.75).int() + (a > 1.25).int() + (a >= 1.75).int()
         + (a > 2.5).int() + (a >= 3.5).int() + (a > 5.0).int())
    return (c + torch.where(v < 0, 8, 0)).to(torch.uint8)


def quantize_fmt(x: torch.Tensor, fmt: str) -> tuple[torch.Tensor, torch.Tensor]:
    """bf16 [N, 512] -> (data rows uint8 [N, data_bytes], scale rows uint8 [N, scale_bytes])."""
    assert x.dtype == torch.bfloat16 and x.shape[-1] == 512
    n = x.shape[0]
    xf = x.float()
    if fmt == "v4":
        g = xf[:, :448].view(n, 7, 64)
        scale, code = _e8m0_codes(g.abs().amax(-1))
        data = torch.empty(n, 576, dtype=torch.uint8, device=x.device)
        data[:, :448] = _e4m3(g / scale[..., None]).view(n, 448)
        data[:, 448:] = x[:, 448:].contiguous().view(torch.uint8).view(n, 128)
        sc = torch.zeros(n, 8, dtype=torch.uint8, device=x.device)
        sc[:, :7] = code
        return data, sc
    if fmt == "v41":
        g = xf.view(n, 16, 32)
        scale, code = _e8m0_codes(g.abs().amax(-1))
        return _e4m3(g / scale[..., None]).view(n, 512), code.contiguous()
    if fmt == "v41_fp4":
        g = xf.view(n, 32, 16)
        amax = g.abs().amax(-1)
        s8 = torch.where(amax == 0, torch.ones_like(amax), amax / 6.0).to(torch.float8_e4m3fn)
        s = s8.float()
        codes = _e2m1(g / s[..., None]).view(n, 512)
        data = codes[:, 0::2] | (codes[:, 1::2] << 4)
        return data.contiguous(), s8.view(torch.uint8).contiguous()
    raise ValueError(fmt)


def make_pool_fmt(num_blocks: int, fmt: str, gen: torch.Generator, device,
                  chunk_pages: int = 1 << 14) -> torch.Tensor:
    """uint8 [num_blocks, 64 * (data + scale bytes)]: each page's data rows, then scale rows."""
    db, sb = FMT_BYTES[fmt]
    pool = torch.empty(num_blocks, PAGE * (db + sb), dtype=torch.uint8, device=device)
    for lo in range(0, num_blocks, chunk_pages):
        hi = min(num_blocks, lo + chunk_pages)
        x = torch.randn((hi - lo) * PAGE, 512, generator=gen, device=device).to(torch.bfloat16)
        data, sc = quantize_fmt(x, fmt)
        pool[lo:hi, :PAGE * db] = data.view(hi - lo, PAGE * db)
        pool[lo:hi, PAGE * db:] = sc.view(hi - lo, PAGE * sb)
    return pool


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_pool(num_blocks: int, ue8m0: bool, gen: torch.Generator, device,
              chunk_rows: int = 1 << 20) -> torch.Tensor:
    rows = num_blocks * PAGE
    kv = torch.empty(rows, ROW_BYTES, dtype=torch.uint8, device=device)
    for lo in range(0, rows, chunk_rows):
        hi = min(rows, lo + chunk_rows)
        x = torch.randn(hi - lo, D_QK, generator=gen, device=device).to(torch.bfloat16)
        kv[lo:hi] = quantize_rows(x, ue8m0)
    return kv.view(num_blocks, PAGE, 1, ROW_BYTES)


def sample_distinct(rows: int, limits: torch.Tensor, k: int, gen: torch.Generator,
                    device) -> torch.Tensor:
    """k distinct positions per row, uniform over [0, limits[row]) (in random order)."""
    maxlim = int(limits.max().item())
    out = torch.empty(rows, k, dtype=torch.int64, device=device)
    step = max(1, (1 << 27) // max(maxlim, 1))
    for lo in range(0, rows, step):
        hi = min(rows, lo + step)
        keys = torch.rand(hi - lo, maxlim, generator=gen, device=device)
        pos = torch.arange(maxlim, device=device)[None, :]
        keys = torch.where(pos < limits[lo:hi, None], keys, torch.full_like(keys, 2.0))
        out[lo:hi] = torch.topk(keys, k, dim=1, largest=False, sorted=True).indices
    return out


def logical_to_physical(pos: torch.Tensor, block_table: torch.Tensor,
                        seq_of_row: torch.Tensor) -> torch.Tensor:
    page = block_table[seq_of_row[:, None], pos // PAGE].long()
    return page * PAGE + pos % PAGE


def make(spec: Spec, device="cpu", gen_device=None) -> Workload:
    """Build the workload for ``spec`` deterministically from ``spec.seed``."""
    device = torch.device(device)
    gd = torch.device(gen_device) if gen_device is not None else device
    gen = _gen(gd, spec.seed)
    b, s_q, h, k = spec.b, spec.s_q, spec.h_q, spec.topk
    q = torch.randn(b, s_q, h, spec.d_qk, generator=gen, device=gd).to(torch.bfloat16)
    if spec.kv_format == "v32":
        kv = make_pool(spec.num_blocks, spec.ue8m0, gen, gd)
    else:
        kv = make_pool_fmt(spec.num_blocks, spec.kv_format, gen, gd)
    perm = torch.randperm(spec.num_blocks, generator=gen, device=gd)
    block_table = perm[: b * spec.pages_per_seq].view(b, spec.pages_per_seq).to(torch.int32)
    rows = b * s_q
    seq_of_row = torch.arange(b, device=gd).repeat_interleave(s_q)
    if spec.causal_base is not None:
        qi = torch.arange(s_q, device=gd).repeat(b)
        limits = torch.clamp(spec.causal_base + qi + 1, max=spec.ctx)
    else:
        limits = torch.full((rows,), spec.ctx, dtype=torch.int64, device=gd)
    kk = min(k, int(limits.min().item()))
    pos = sample_distinct(rows, limits, kk, gen, gd)
    phys = logical_to_physical(pos, block_table, seq_of_row)
    if kk < k:  # a row shorter than topk is padded with -1 at the end
        pad = torch.full((rows, k - kk), -1, dtype=phys.dtype, device=gd)
        phys = torch.cat([phys, pad], dim=1)
    if spec.sort_indices:
        phys = torch.sort(phys, dim=1).values
    if spec.masked_per_row:
        which = torch.topk(torch.rand(rows, k, generator=gen, device=gd), spec.masked_per_row,
                           dim=1).indices
        phys = phys.scatter(1, which, -1)
    indices = phys.to(torch.int32).view(b, s_q, k)
    wl = Workload(spec, q.to(device), kv.to(device), indices.to(device),
                  block_table.to(device), 1.0 / math.sqrt(spec.d_qk))
    return wl


def small(b=2, s_q=1, h_q=128, topk=128, ctx=512, ue8m0=False, masked_per_row=0,
          causal_base=None, sort_indices=False, extra_pool_pages=0, seed=0,
          device="cpu", kv_format="v32") -> Workload:
    """A scaled-down workload with the same structure (for parity tests)."""
    spec = Spec(f"small_b{b}_sq{s_q}_h{h_q}_k{topk}_ctx{ctx}_{kv_format}", b=b, s_q=s_q,
                h_q=h_q, topk=topk, ctx=ctx, ue8m0=ue8m0, masked_per_row=masked_per_row,
                causal_base=causal_base, sort_indices=sort_indices,
                extra_pool_pages=extra_pool_pages, seed=seed, kv_format=kv_format)
    return make(spec, device=device)


def attn_sink(h_q: int, seed: int, device="cpu") -> torch.Tensor:
    """fp32 [h_q] per-head sink values: head 0 takes -2.5 (the worked example's value), the
    others are uniform on [-4, 10], a range that straddles the log-sum-exp of a few hundred
    to a few thousand keys with unit-variance scores, so the sink visibly changes some rows
    and barely touches others."""
    g = _gen(torch.device("cpu"), seed)
    s = torch.rand(h_q, generator=g, dtype=torch.float64) * 14.0 - 4.0
    s[0] = -2.5
    return s.float().to(device)


def topk_lengths(b: int, s_q: int, topk: int, seed: int, device="cpu") -> torch.Tensor:
    """int32 [b, s_q] per-token valid prefix lengths: uniform on [0, topk], with the edge
    values 0, 1, 63, 64, 65, topk and topk + 7 (beyond the list) placed on the first tokens
    when they fit."""
    g = _gen(torch.device("cpu"), seed)
    n = b * s_q
    lens = torch.randint(0, topk + 1, (n,), generator=g, dtype=torch.int64)
    edges = [v for v in (0, 1, 63, 64, 65, topk, topk + 7) if v <= topk + 7]
    k = min(n, len(edges))
    lens[:k] = torch.tensor(edges[:k], dtype=torch.int64)
    return lens.to(torch.int32).view(b, s_q).to(device)


def index_scores(n_tok: int, ld: int, dtype=torch.bfloat16, seed: int = 0, device="cpu",
                 levels: int = 0) -> torch.Tensor:
    """[n_tok, ld] synthetic index scores, N(0, 1) rounded to ``dtype`` (bf16 rounding makes
    ties common at any threshold); levels > 0 draws from that many integer values instead (a
    tie-heavy row)."""
    g = _gen(torch.device("cpu"), seed)
    if levels > 0:
        x = torch.randint(0, levels, (n_tok, ld), generator=g).float()
    else:
        x = torch.randn(n_tok, ld, generator=g)
    return x.to(dtype).to(device)


def e4m3_codes(shape, seed: int, device="cpu", scale: float = 1.0) -> torch.Tensor:
    """uint8 e4m3 codes of N(0, scale^2) values (saturated at +-448; never the NaN codes)."""
    g = _gen(torch.device("cpu"), seed)
    x = (torch.randn(shape, generator=g) * scale).clamp_(-E4M3_MAX, E4M3_MAX)
    return x.to(torch.float8_e4m3fn).view(torch.uint8).to(device)


def indexer_cache(num_pages: int, seed: int, device="cpu") -> torch.Tensor:
    """uint8 [num_pages, 8448] indexer key pages: 64 x 128 e4m3 codes of N(0, 1) keys, then 64
    fp32 per-token scales uniform on [0.5, 1.5] / 16."""
    g = _gen(torch.device("cpu"), seed)
    codes = e4m3_codes((num_pages, 64 * 128), seed + 1)
    scales = (torch.rand(num_pages, 64, generator=g) + 0.5) / 16.0
    page = torch.empty(num_pages, 64 * 128 + 256, dtype=torch.uint8)
    page[:, : 64 * 128] = codes
    page[:, 64 * 128:] = scales.float().contiguous().view(torch.uint8).view(num_pages, 256)
    return page.to(device)


def indexer_queries(n_tok: int, seed: int, device="cpu"):
    """(q8 uint8 [n_tok, 64, 128] e4m3 codes of N(0, 1) queries, weights fp32 [n_tok, 64]
    uniform on [-1, 1] / 8: signed, as the head weights are not a softmax)."""
    g = _gen(torch.device("cpu"), seed)
    q8 = e4m3_codes((n_tok, 64, 128), seed + 2)
    w = (torch.rand(n_tok, 64, generator=g) * 2 - 1) / 8
    return q8.to(device), w.float().to(device)


def to_numpy_inputs(wl: Workload):
    """(q as uint16 bf16 bits, kv uint8, indices int32) numpy arrays on the host."""
    q = wl.q.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
    kv = wl.kv.detach().cpu().contiguous().numpy()
    kv = kv.reshape(kv.shape[0], kv.shape[1], ROW_BYTES)
    idx = wl.indices.detach().cpu().contiguous().numpy()
    return q, kv, idx


def row_bytes(spec: Spec) -> int:
    """Bytes of one cached token in the spec's format (data + scales)."""
    return ROW_BYTES if spec.kv_format == "v32" else sum(FMT_BYTES[spec.kv_format])


def flops_valid(wl: Workload) -> float:
    """Algorithmic FLOPs: 2 * h * (d_qk + 512) per valid slot (an FMA counts 2)."""
    return 2.0 * wl.spec.h_q * (wl.spec.d_qk + D_V) * wl.num_valid


def alg_bytes(wl: Workload) -> float:
    """Algorithmic HBM bytes: gathered rows + Q + O + indices + LSE per query token."""
    tok = wl.spec.b * wl.spec.s_q
    h = wl.spec.h_q
    return (wl.num_valid * row_bytes(wl.spec)
            + tok * (h * wl.spec.d_qk * 2 + h * D_V * 2 + wl.spec.topk * 4 + h * 4))
