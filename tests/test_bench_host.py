"""Host logic of bench.py that needs no GPU: the rotated index sets of the end-to-end loop."""

import torch

import bench
import workloads


def test_rotated_index_sets_keep_the_workload_structure():
    wl = workloads.small(b=3, s_q=2, h_q=64, topk=200, ctx=4096, masked_per_row=9, seed=5)
    sets = bench.rotated_index_sets(wl.indices, wl.block_table, wl.kv.shape[0], 4, shift_pages=16)
    assert len(sets) == 4 and torch.equal(sets[0], wl.indices.to(torch.int32))
    base = wl.indices
    first = set(base[base >= 0].tolist())
    for s in sets[1:]:
        assert s.shape == base.shape and s.dtype == torch.int32
        assert torch.equal(s < 0, base < 0)  # the same masked slots
        for r in range(base.shape[0]):
            pages = set(wl.block_table[r].tolist())
            for t in range(base.shape[1]):
                v = s[r, t][s[r, t] >= 0]
                assert v.unique().numel() == v.numel()  # still distinct within a row
                assert set((v // 64).tolist()) <= pages  # still the sequence's own pages
        moved = set(s[s >= 0].tolist())
        assert len(first & moved) < 0.3 * len(first)  # mostly other rows


def test_rotation_is_a_shift_of_logical_positions():
    # one sequence whose pages are in order: a shift by p pages adds p * 64 to the position
    bt = torch.arange(8, dtype=torch.int32).view(1, 8)
    idx = torch.tensor([[[0, 5, 64, 130, -1, 511]]], dtype=torch.int32)
    s = bench.rotated_index_sets(idx, bt, 8, 2, shift_pages=2)[1]
    assert s.tolist() == [[[128, 133, 192, 258, -1, (511 + 128) % 512]]]
