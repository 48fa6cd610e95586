"""Greedy split-KV partition planner, written as a plain Python loop.

TEST INFRASTRUCTURE ONLY (the oracle): the product path never imports this module.

Source: "FlashMLA Sparse Decode 完整计算过程详解", step 3 (Tile Scheduler), sections 3.1,
3.3, 3.4 and 3.5, and "FlashMLA 与 DSA：内核、流水线和正确性边界", section 3.2.

What it computes, in the pages' terms:

* The top-k list of each request is cut into blocks of 64 slots (these are blocks of the
  index list, not KV pages): ``num_blocks[i] = ceil(topk_i / 64)``.
* Each request also costs a fixed overhead of 5 block-units (Q load, softmax state,
  write-back): ``total = sum_i (num_blocks[i] + 5)``.
* ``payload = ceil(total / num_sm_parts) + 5`` is the capacity of every partition.
* Partitions are filled left to right.  The rest of the current request goes in whole
  when ``blocks_left + 5 <= remain``; otherwise the partition takes ``remain - 5``
  blocks of it, the request is split there, and the partition is closed.  A partition
  that has taken a whole request and has no room left is closed too.
* ``num_splits`` is the prefix sum over requests of the number of partitions that touch
  each request.

Readings where the pages are silent:

* ``end_block`` is exclusive and ``end_req`` is the last request the partition touches.
* A partition stops as soon as ``remain - 5 <= 0`` would leave it nothing to take.
* ``begin_split_idx`` is the slot, in the split-partial buffers, of the partition's first
  (request, split) pair; it equals ``num_splits[begin_req]`` plus the number of earlier
  partitions that already worked on ``begin_req``.
* ``num_sm_parts = max(num_sms // s_q // 2, 1)``: one partition is one pair of SMs, as in
  the pages' section 3.3 formula for 128 heads on two CTAs.
"""

from __future__ import annotations

from dataclasses import dataclass

TOPK_BLOCK = 64
FIXED_OVERHEAD = 5


@dataclass(frozen=True)
class Partition:
    begin_req: int
    end_req: int
    begin_block: int
    end_block: int
    begin_split_idx: int
    is_first_req_splitted: bool
    is_last_req_splitted: bool

    def empty(self, batch: int) -> bool:
        return self.begin_req >= batch


def num_sm_parts(num_sms: int, s_q: int) -> int:
    return max(num_sms // s_q // 2, 1)


def plan(topk_per_req: list[int], parts: int) -> tuple[list[Partition], list[int]]:
    """Return (partitions, num_splits_prefix) for the given per-request top-k lengths."""
    b = len(topk_per_req)
    nblocks = [(t + TOPK_BLOCK - 1) // TOPK_BLOCK for t in topk_per_req]
    total = sum(n + FIXED_OVERHEAD for n in nblocks)
    payload = -(-total // parts) + FIXED_OVERHEAD
    splits_per_req = [0] * b
    out: list[Partition] = []
    now_req, now_block = 0, 0
    for _ in range(parts):
        if now_req >= b:
            out.append(Partition(b, b, 0, 0, 0, False, False))
            continue
        remain = payload
        begin_req, begin_block = now_req, now_block
        first_split = now_block > 0
        end_req, end_block, last_split = now_req, now_block, False
        while now_req < b:
            left = nblocks[now_req] - now_block
            if left + FIXED_OVERHEAD <= remain:
                remain -= left + FIXED_OVERHEAD
                splits_per_req[now_req] += 1
                end_req, end_block, last_split = now_req, nblocks[now_req], False
                now_req, now_block = now_req + 1, 0
                if remain - FIXED_OVERHEAD <= 0:
                    break
            else:
                take = remain - FIXED_OVERHEAD
                if take > 0:
                    splits_per_req[now_req] += 1
                    now_block += take
                    end_req, end_block, last_split = now_req, now_block, True
                break
        out.append(Partition(begin_req, end_req, begin_block, end_block, -1, first_split,
                             last_split))
    prefix = [0]
    for n in splits_per_req:
        prefix.append(prefix[-1] + n)
    # begin_split_idx: slot of the partition's first (request, split) pair.
    seen = [0] * b
    fixed: list[Partition] = []
    for p in out:
        if p.empty(b):
            fixed.append(Partition(p.begin_req, p.end_req, 0, 0, prefix[b], False, False))
            continue
        first = prefix[p.begin_req] + seen[p.begin_req]
        for r in range(p.begin_req, p.end_req + 1):
            seen[r] += 1
        fixed.append(Partition(p.begin_req, p.end_req, p.begin_block, p.end_block, first,
                               p.is_first_req_splitted, p.is_last_req_splitted))
    return fixed, prefix


def block_range(p: Partition, req: int, nblocks_req: int) -> tuple[int, int]:
    """Blocks [begin, end) of request ``req`` that partition ``p`` processes."""
    begin = p.begin_block if req == p.begin_req else 0
    end = p.end_block if req == p.end_req else nblocks_req
    return begin, end
