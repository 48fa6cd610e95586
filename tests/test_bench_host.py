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


def test_code_hash_ignores_comments_and_whitespace_only(tmp_path):
    a = tmp_path / "a.cu"
    a.write_text("// header\nint f(int x) {  /* a\\nblock */ return x + 1; }  // tail\n")
    b = tmp_path / "b.cu"
    b.write_text("// another header\n\nint f(int x) {\n  return x + 1;\n}\n")
    c = tmp_path / "c.cu"
    c.write_text("int f(int x) { return x + 2; }\n")
    assert bench.code_sha256(str(a)) == bench.code_sha256(str(b))
    assert bench.code_sha256(str(a)) != bench.code_sha256(str(c))


def test_committed_profiles_match_the_current_kernels():
    # each kernel's ncu summary was taken on the code that is in the tree now
    import os
    csrc = os.path.join(bench.ROOT, "sparse_mla_attention_decode_gb300", "csrc")
    for src, prof in (("decode_fwd.cu", "decode_kernel_c2_b64_h128_k2048_mask5.md"),
                      ("decode_fwd.cu", "decode_kernel_c5_b1_sq4096_h128_k2048.md"),
                      ("decode_fwd.cu", "decode_kernel_c4_b32_h128_k2048_ue8m0_sorted.md"),
                      ("topk.cu", "topk_kernel_prefill_1024x65536_k2048.md"),
                      ("indexer.cu", "indexer_kernel_decode_b64_ctx32768.md"),
                      ("indexer.cu", "indexer_kernel_prefill_sq4096_ctx65536.md")):
        assert bench.traffic_from_profiles(os.path.join(csrc, src), prof) is not None, prof
    # the selection chain's two kernels share one summary
    assert bench.traffic_from_pair_profile(
        [os.path.join(csrc, "indexer.cu"), os.path.join(csrc, "topk.cu")],
        "select_kernels_decode_b64_ctx32768_k2048.md") is not None
