"""The C-ABI library loads, exports every entry point its header declares, and rejects bad
arguments before launching anything (no GPU needed)."""

import ctypes
import os
import re

import pytest

import sparse_mla_attention_decode_gb300 as smla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    smla.build()
    return smla.lib()


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", f)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(sparse_mla_\w+)\s*\(", txt))
    return names


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert {"sparse_mla_sched_meta", "sparse_mla_decode_fwd", "sparse_mla_combine"} <= names
    for n in names:
        assert hasattr(L, n), n
    assert set(smla.EXPORTED) == names


def test_status_strings(L):
    assert smla.sparse_mla_status_string(0) == "ok"
    assert "unsupported" in smla.sparse_mla_status_string(2)
    assert smla.sparse_mla_status_string(99) == "unknown status"
    assert "sm_103a" in smla.sparse_mla_version()


def test_workspace_sizes(L):
    d = smla.dims_for(64, 1, 128, 2048, 32768)
    sb, ab = smla.sparse_mla_workspace_size(d, 152)
    parts = 152 // 1 // 2
    assert sb >= parts * 32 + 65 * 4 + 4
    assert ab == 0  # this plan splits no request: no split-partial workspace at all
    # the prefill-shaped problem needs none either (it used to ask for 2 GiB)
    assert smla.sparse_mla_workspace_size(smla.dims_for(1, 4096, 128, 2048, 1024), 152)[1] == 0


def _expected_accum_bytes(b, s_q, h_q, topk, num_sms):
    """The split-partial workspace as the header documents it, from the oracle's planner:
    slots = num_splits[r + 1] for the last split request r, fp32 O [slots][s_q][h_q][512],
    then the base-2 lse [slots][s_q][h_q] at the next 256-byte boundary."""
    from oracle import sched as osched
    _, prefix = osched.plan([topk] * b, osched.num_sm_parts(num_sms, s_q))
    split = [r for r in range(b) if prefix[r + 1] - prefix[r] > 1]
    if not split:
        return 0
    slots = prefix[split[-1] + 1]
    lse_off = (slots * s_q * h_q * 512 * 4 + 255) // 256 * 256
    return lse_off + slots * s_q * h_q * 4


def test_workspace_size_follows_the_plan(L):
    """accum_bytes covers exactly the split slots the oracle's planner numbers."""
    rng = __import__("random").Random(17)
    cases = [(2, 1, 128, 128, 132), (64, 1, 128, 2048, 152), (32, 1, 128, 2048, 152),
             (128, 2, 64, 2048, 152), (1, 4096, 128, 2048, 152), (3, 2, 64, 2048, 40),
             (2, 3, 128, 2048, 60), (1, 1, 128, 2048, 152), (4, 1, 128, 512, 120),
             (77, 1, 128, 2048, 152), (5, 1, 64, 0, 16), (64, 8, 128, 2048, 152)]
    cases += [(rng.randint(1, 300), rng.choice([1, 1, 2, 3, 8]), rng.choice([64, 128]),
               rng.randint(0, 5000), rng.randint(2, 300)) for _ in range(300)]
    for b, s_q, h_q, topk, num_sms in cases:
        d = smla.dims_for(b, s_q, h_q, topk, 64)
        _, ab = smla.sparse_mla_workspace_size(d, num_sms)
        assert ab == _expected_accum_bytes(b, s_q, h_q, topk, num_sms), (b, s_q, h_q, topk, num_sms)


@pytest.mark.parametrize("field,value,code", [("h_q", 96, 2), ("d_qk", 512, 2), ("d_v", 256, 2),
                                              ("page_block_size", 32, 2), ("b", -1, 1),
                                              ("topk", -5, 1), ("num_blocks", 1 << 26, 2),
                                              ("extra_topk", -1, 1),
                                              ("extra_num_blocks", 1 << 26, 2)])
def test_bad_dims_rejected(L, field, value, code):
    d = smla.dims_for(2, 1, 128, 128, 64)
    setattr(d, field, value)
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    assert L.sparse_mla_workspace_size(ctypes.byref(d), 152, ctypes.byref(a), ctypes.byref(b)) == code


@pytest.mark.parametrize("fmt,d_qk,extra_topk,extra_fmt,code", [
    ("v41", 512, 0, 3, 0), ("v41", 512, 64, 3, 0), ("v4", 512, 0, 0, 0),
    ("v4", 512, 64, 0, 2),      # no extra cache beside a V4 cache
    ("v41", 512, 64, 0, 2),     # the extra cache of a V4.1 cache is FP4
    ("v32", 512, 0, 0, 2), ("v41", 576, 0, 3, 2), ("v4", 576, 0, 0, 2),
    ("v32", 576, 64, 3, 2)])
def test_kv_formats_checked(L, fmt, d_qk, extra_topk, extra_fmt, code):
    d = smla.dims_for(2, 1, 128, 128, 64, extra_topk=extra_topk,
                      extra_num_blocks=8 if extra_topk else 0, kv_format=fmt)
    d.d_qk, d.extra_kv_format = d_qk, extra_fmt
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    assert L.sparse_mla_workspace_size(ctypes.byref(d), 152, ctypes.byref(a), ctypes.byref(b)) == code
    d.kv_format = 7
    assert L.sparse_mla_workspace_size(ctypes.byref(d), 152, ctypes.byref(a), ctypes.byref(b)) == 2


def test_pointer_checks_before_launch(L):
    d = smla.dims_for(2, 1, 128, 128, 64)
    sb, ab = smla.sparse_mla_workspace_size(d, 152)
    fake = 0x10000
    # null plan
    assert L.sparse_mla_sched_meta(ctypes.byref(d), 152, None, sb, None) == 1
    # misaligned plan
    assert L.sparse_mla_sched_meta(ctypes.byref(d), 152, fake + 4, sb, None) == 3
    # plan buffer too small
    assert L.sparse_mla_sched_meta(ctypes.byref(d), 152, fake, sb - 1, None) == 4
    args = dict(q=fake, kv=fake, idx=fake, plan=fake, ws=fake, out=fake, lse=fake)

    def call(**kw):
        a = {**args, **kw}
        return L.sparse_mla_decode_fwd(ctypes.byref(d), 152, a["q"], a["kv"], a["idx"],
                                       ctypes.c_float(0.0417), a["plan"], a["ws"],
                                       kw.get("wsb", ab), a["out"], a["lse"], None)

    assert call(q=None) == 1
    assert call(out=fake + 8) == 3
    assert call(kv=fake + 8) == 3
    assert call(wsb=ab - 1) == 4
    assert L.sparse_mla_decode_fwd(ctypes.byref(d), 152, fake, fake, fake, ctypes.c_float(float("nan")),
                                   fake, fake, ab, fake, fake, None) == 1
    assert L.sparse_mla_combine(ctypes.byref(d), 152, fake, fake, ab - 1, fake, fake, None) == 4
    code = ctypes.c_int()
    assert L.sparse_mla_read_device_status(ctypes.byref(d), 152, None, ctypes.byref(code), None) == 1


def test_decode_option_checks_before_launch(L):
    d = smla.dims_for(2, 1, 128, 128, 64)
    sb, ab = smla.sparse_mla_workspace_size(d, 152)
    fake = 0x10000

    def fwd(opts):
        return L.sparse_mla_decode_fwd_ex(ctypes.byref(d), 152, fake, fake, fake,
                                          ctypes.c_float(0.0417), opts, fake, fake, ab, fake,
                                          fake, None)

    def comb(opts):
        return L.sparse_mla_combine_ex(ctypes.byref(d), 152, opts, fake, fake, ab, fake, fake,
                                       None)

    for bad in (smla.smla_decode_opts(fake + 2, None), smla.smla_decode_opts(None, fake + 1),
                smla.smla_decode_opts(None, None, 0, fake + 8, fake),
                smla.smla_decode_opts(None, None, 0, fake, fake + 2)):
        assert fwd(ctypes.byref(bad)) == 3
        assert comb(ctypes.byref(bad)) == 3
    # other argument errors still come first or alongside: a null q with options set
    ok = smla.smla_decode_opts(fake, fake)
    assert L.sparse_mla_decode_fwd_ex(ctypes.byref(d), 152, None, fake, fake,
                                      ctypes.c_float(0.0417), ctypes.byref(ok), fake, fake, ab,
                                      fake, fake, None) == 1
    assert L.sparse_mla_combine_ex(ctypes.byref(d), 152, ctypes.byref(ok), fake, fake, ab - 1,
                                   fake, fake, None) == 4


def test_no_device_is_a_cuda_error_not_a_crash(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    d = smla.dims_for(2, 1, 128, 128, 64)
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    # num_sms <= 0 asks the library to query the device: on a machine without one -> CUDA error
    assert L.sparse_mla_workspace_size(ctypes.byref(d), 0, ctypes.byref(a), ctypes.byref(b)) == 5


def test_product_path_does_not_touch_the_oracle():
    """The package and its kernels never import, link or read anything under oracle/."""
    pkg = os.path.join(ROOT, "sparse_mla_attention_decode_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                txt = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "oracle" not in txt.lower(), f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c")):
            txt = open(os.path.join(ROOT, "oracle", f), encoding="utf-8").read()
            assert "sparse_mla_attention_decode_gb300" not in txt and "sparse_mla.h" not in txt, f


def test_plan_has_splits_matches_oracle_planner(L):
    """The host-side walk of the plan agrees with the oracle's greedy planner (any request
    split)."""
    from oracle import sched as osched
    rng = __import__("random").Random(5)
    cases = [(2, 1, 128, 132), (64, 1, 2048, 152), (32, 1, 2048, 152), (128, 2, 2048, 152),
             (1, 4096, 2048, 152), (76, 1, 2048, 152), (77, 1, 2048, 152), (1, 1, 1, 152),
             (300, 1, 2048, 152), (64, 1, 4096, 152), (5, 1, 64, 16), (200, 1, 64, 6)]
    cases += [(rng.randint(1, 400), rng.choice([1, 1, 2, 3, 4]), rng.randint(1, 5000),
               rng.randint(2, 300)) for _ in range(400)]
    for b, s_q, topk, num_sms in cases:
        d = smla.dims_for(b, s_q, 128, topk, 64)
        got = smla.sparse_mla_plan_has_splits(d, num_sms)
        parts = osched.num_sm_parts(num_sms, s_q)
        _, prefix = osched.plan([topk] * b, parts)
        want = any(prefix[i + 1] - prefix[i] > 1 for i in range(b))
        assert got == want, (b, s_q, topk, num_sms)


def test_extra_list_needs_its_pointers(L):
    d = smla.dims_for(2, 1, 128, 128, 64, extra_topk=64, extra_num_blocks=8)
    sb, ab = smla.sparse_mla_workspace_size(d, 152)
    fake = 0x10000
    # the plain call has no extra pointers: rejected before launch
    assert L.sparse_mla_decode_fwd(ctypes.byref(d), 152, fake, fake, fake, ctypes.c_float(0.04),
                                   fake, fake, ab, fake, fake, None) == 1
    no_cache = smla.smla_decode_opts(None, None, 0, None, fake)
    assert L.sparse_mla_decode_fwd_ex(ctypes.byref(d), 152, fake, fake, fake, ctypes.c_float(0.04),
                                      ctypes.byref(no_cache), fake, fake, ab, fake, fake, None) == 1
    # the plan counts both lists: 2 + 1 blocks per request
    d0 = smla.dims_for(2, 1, 128, 128, 64)
    d3 = smla.dims_for(2, 1, 128, 192, 64)
    assert smla.sparse_mla_plan_has_splits(d, 152) == smla.sparse_mla_plan_has_splits(d3, 152)
    assert smla.sparse_mla_workspace_size(d, 152) == smla.sparse_mla_workspace_size(d3, 152)
    assert smla.sparse_mla_workspace_size(d0, 152)[0] == smla.sparse_mla_workspace_size(d, 152)[0]


def test_topk_argument_checks(L):
    fake = 0x10000
    d = smla.smla_topk_dims(4, 1, 64, 128, 2, smla.SMLA_SCORES_BF16)
    call = lambda dd, sc=fake: L.sparse_mla_topk_page_table(ctypes.byref(dd), sc, fake, fake,
                                                            fake, None, None)
    assert call(smla.smla_topk_dims(4, 1, 0, 128, 2, 0)) == 1      # k = 0
    assert call(smla.smla_topk_dims(4, 0, 64, 128, 2, 0)) == 1     # s_q = 0
    assert call(smla.smla_topk_dims(4, 1, 64, 128, 2, 7)) == 2     # dtype
    assert call(smla.smla_topk_dims(4, 1, 64, 100, 2, 0)) == 3     # row stride not 16 bytes
    assert call(d, fake + 8) == 3                                  # misaligned scores
    assert L.sparse_mla_topk_page_table(ctypes.byref(d), fake, None, fake, fake, None, None) == 1
    assert call(smla.smla_topk_dims(0, 1, 64, 128, 2, 0)) == 0     # no rows: nothing to do


def test_indexer_argument_checks(L):
    fake = 0x10000
    call = lambda d, q=fake: L.sparse_mla_indexer_scores(ctypes.byref(d), 152, q, fake, fake,
                                                         fake, fake, fake, None, None)
    assert call(smla.smla_indexer_dims(4, 1, 32, 128, 8, 512, 16)) == 2   # heads
    assert call(smla.smla_indexer_dims(4, 1, 64, 64, 8, 512, 16)) == 2    # dim
    assert call(smla.smla_indexer_dims(5, 2, 64, 128, 8, 512, 16)) == 1   # n_tok % s_q
    assert call(smla.smla_indexer_dims(4, 1, 64, 128, 8, 512, 16), fake + 4) == 3  # q8 alignment
    assert call(smla.smla_indexer_dims(0, 1, 64, 128, 8, 512, 16)) == 0   # nothing to do


def test_indexer_topk_argument_checks(L):
    fake = 0x10000

    def call(d, topk=16, scratch=fake, nbytes=1 << 20, status=fake):
        return L.sparse_mla_indexer_topk(ctypes.byref(d), topk, 152, fake, fake, fake, fake, fake,
                                         scratch, nbytes, fake, status, None)
    ok = smla.smla_indexer_dims(4, 2, 64, 128, 8, 512, 16)
    assert call(ok, topk=0) == 1                                             # topk
    assert call(ok, status=None) == 1                                         # status required
    assert call(smla.smla_indexer_dims(4, 1, 32, 128, 8, 512, 16)) == 2       # heads
    assert call(smla.smla_indexer_dims(5, 2, 64, 128, 8, 512, 16)) == 1       # n_tok % s_q
    assert call(ok, scratch=None) == 1                                        # no scratch
    assert call(smla.smla_indexer_dims(4, 2, 64, 128, 8, 510, 16)) == 3       # ld % 4
    assert call(ok, scratch=fake + 8) == 3                                    # scratch alignment
    assert call(ok, nbytes=512 * 4 - 16) == 4                                 # below one token
    assert call(smla.smla_indexer_dims(0, 1, 64, 128, 8, 512, 16)) == 0       # nothing to do


def test_indexer_topk_scratch_size(L):
    def size(d):
        n = ctypes.c_size_t()
        assert L.sparse_mla_indexer_topk_scratch_size(ctypes.byref(d), ctypes.byref(n)) == 0
        return n.value
    # positions = min(ld, max_pages * 64); rows = min(n_tok, budget // (positions * 4))
    assert size(smla.smla_indexer_dims(64, 1, 64, 128, 512, 32768, 1)) == 64 * 32768 * 4
    assert size(smla.smla_indexer_dims(64, 1, 64, 128, 100, 32768, 1)) == 64 * 6400 * 4
    big = smla.smla_indexer_dims(4096, 4096, 64, 128, 1024, 65536, 1)
    assert size(big) == (smla.SELECT_SCRATCH_BUDGET // (65536 * 4)) * 65536 * 4
    assert size(smla.smla_indexer_dims(3, 1, 64, 128, 1 << 20, 1 << 26, 1)) == (1 << 26) * 4
