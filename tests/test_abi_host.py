"""The C-ABI library loads and exports every entry point include/specdec.h
declares; argument checks that run on the host return their error codes
without enqueuing anything.  No GPU needed."""
import ctypes
import os
import re

import pytest

import speculative_decoding_draft_select_gb300 as sd
from speculative_decoding_draft_select_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "specdec.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|int64_t|size_t)\s+(\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    build()
    return sd.lib()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n
    assert set(sd._SIGS) >= set(names)


def test_binding_exports_exist_and_refuse_host_tensors():
    """Every name the binding exports exists, and the calls refuse host
    (CPU) tensors before touching the library: there is no CPU path."""
    import torch
    for n in sd.__all__:
        assert hasattr(sd, n), n
    x = torch.zeros((2, 8))
    with pytest.raises(ValueError):
        sd.spec_softmax_topk(x, 1.0, 2)
    ids = torch.zeros(8, dtype=torch.int32)
    with pytest.raises(ValueError):
        sd.tli_constrain_map_qlogits(x, ids, ids, 1.0)
    tgt = torch.zeros((1, 2, 8))
    tok = torch.zeros((1, 2), dtype=torch.int32)
    with pytest.raises(ValueError):
        sd.spec_verify_sample(tgt, 1.0, torch.zeros((1, 2, 8)), tok, tok, tok, torch.zeros((1, 2)), torch.zeros(1),
                              without_replacement=True)


def test_host_side_argument_checks_null_pointers(lib):
    """Checks reached with null pointers only: nothing here can launch."""
    null = None
    # k > V, T <= 0, T_score <= 0, null pointers
    assert lib.spec_softmax_topk(null, 1, 4, 3, 1.0, 1.0, 4, null, null, null, null, null, null) == -1
    assert lib.spec_softmax_topk(null, 1, 4, 8, 0.0, 1.0, 2, null, null, null, null, null, null) == -1
    assert lib.spec_softmax_topk(null, 1, 4, 8, 1.0, 0.0, 2, null, null, null, null, null, null) == -1
    assert lib.spec_softmax_topk(null, 1, 4, 8, 1.0, 1.0, 2, null, null, null, null, null, null) == -1
    assert lib.spec_softmax_topk(null, 1, 0, 8, 1.0, 1.0, 2, null, null, null, null, null, null) == 0
    assert lib.spec_softmax_sample(null, 1, 0, 8, 1.0, null, null, null, null, null, null, null) == 0
    assert lib.spec_tree_expand(0, 2, 4, 0, null, null, null, null, null, null, null, null, null) == -1
    assert lib.spec_tree_expand(2, 2, 4, 2, null, null, null, null, null, null, null, null, null) == -1
    assert lib.spec_build_tree(1, 2, 2, 8, *([null] * 15)) == -1  # N > P = 7
    assert lib.spec_verify_greedy(2, 4, 10, 1, *([null] * 5), -1, *([null] * 8), 0, null) == -1
    assert lib.spec_verify_sample(2, 4, 10, 1, null, 0.0, *([null] * 8), -1, *([null] * 8), 0, null) == -1
    assert lib.spec_verify_sample_qlogits(2, 4, 10, 1, null, 1.0, null, 1, null, 0.0, *([null] * 7), -1,
                                          *([null] * 8), 0, null) == -1
    assert lib.spec_compact_slots(2, 4, 0, *([null] * 4), 16, *([null] * 4), 0, *([null] * 3), 0, 0, null,
                                  null) == -1
    assert lib.spec_verify_sample_flags(0, 4, 10, 1, *([null] * 1), 1.0, *([null] * 8), -1, *([null] * 8), 0, 1,
                                        null) == 0
    assert lib.tli_constrain_map(4, 10, 10, null, 1, null, null, 1.0, null, null, null, null, null, null) == -1
    assert lib.tli_map_ids(null, null, -1, null, 0, 0, null) == -1
    assert lib.tli_plan_build(10, 10, null, null, null, null) == -1
    assert lib.tli_constrain_map_planned(0, 10, 10, null, 1, null, null, null, 1.0, null, null, null, null, null,
                                         null) == 0
    assert lib.tli_constrain_map_qlogits(0, 10, 10, null, 1, null, null, null, 1.0, null, null, null, null, null,
                                         null, null, null) == 0
    # filtering: negative rows, V < 1, T <= 0, NaN top_p, bad dtype; nothing to filter; null logits
    assert lib.spec_filter_logits(null, 1, -1, 8, 1.0, 2, 0.5, null, null) == -1
    assert lib.spec_filter_logits(null, 1, 4, 0, 1.0, 2, 0.5, null, null) == -1
    assert lib.spec_filter_logits(null, 1, 4, 8, 0.0, 2, 0.5, null, null) == -1
    assert lib.spec_filter_logits(null, 1, 4, 8, 1.0, 2, float("nan"), null, null) == -1
    assert lib.spec_filter_logits(null, 7, 4, 8, 1.0, 2, 0.5, null, null) == -2
    assert lib.spec_filter_logits(null, 1, 4, 8, 1.0, 0, 1.0, null, null) == 0   # top_k off, top_p 1: no work
    assert lib.spec_filter_logits(null, 1, 4, 8, 1.0, 8, 1.0, null, null) == 0   # top_k >= V: no work
    assert lib.spec_filter_logits(null, 1, 4, 8, 1.0, 2, 1.0, null, null) == -1  # work, but no logits
    # pruned head: bad sizes and temperature, empty batch, null pointers
    ph = lambda M, H, K, Vd, T: lib.tli_pruned_head(M, H, K, null, null, null, null, Vd, T, *([null] * 8), 0, null)
    assert ph(-1, 64, 8, 16, 1.0) == -1
    assert ph(4, 0, 8, 16, 1.0) == -1
    assert ph(4, 64, 0, 16, 1.0) == -1
    assert ph(4, 64, 8, 0, 1.0) == -1
    assert ph(4, 64, 8, 16, 0.0) == -1
    assert ph(0, 64, 8, 16, 1.0) == 0
    assert ph(4, 64, 8, 16, 1.0) == -1
    # the mapped stochastic verify needs its map
    assert lib.spec_verify_sample_qlogits_mapped(2, 4, 10, 1, null, 1.0, null, 1, null, 1.0, *([null] * 7), -1,
                                                 *([null] * 8), 0, 0, null, null) == -1


def _cuda_present():
    import torch
    return torch.cuda.is_available()


@pytest.mark.skipif(_cuda_present(), reason="made-up addresses are passed only where no GPU could run a kernel")
def test_host_side_argument_checks(lib):
    """Checks that need non-null (made-up) addresses to get past the null
    tests.  Each must return before any launch; run only without a GPU, so
    that a check that regressed gives a wrong return code, never a kernel
    reading a made-up address."""
    null = None
    p16 = ctypes.c_void_p(16)
    # bad dtype, k above the limit
    assert lib.spec_softmax_topk(p16, 7, 4, 8, 1.0, 1.0, 2, p16, p16, null, null, null, null) == -2
    assert lib.spec_softmax_topk(p16, 1, 4, 100, 1.0, 1.0, 33, p16, p16, null, null, null, null) == -2
    # fused softmax + draw: T <= 0, bad dtype, a vocabulary beyond its shared-memory tiles
    assert lib.spec_softmax_sample(p16, 1, 4, 8, 0.0, p16, p16, null, null, null, null, null) == -1
    assert lib.spec_softmax_sample(p16, 5, 4, 8, 1.0, p16, p16, null, null, null, null, null) == -2
    assert lib.spec_softmax_sample(p16, 1, 4, 524289, 1.0, p16, p16, null, null, null, null, null) == -2
    assert lib.spec_softmax_sample(p16, 0, 4, 262145, 1.0, p16, p16, null, null, null, null, null) == -2
    # verify flags: unknown bits are rejected before anything else is looked at
    assert lib.spec_verify_sample_flags(2, 4, 10, 1, p16, 1.0, *([p16] * 8), -1, *([p16] * 6), null, p16, 1 << 20,
                                        2, null) == -1
    assert lib.spec_verify_sample_qlogits_flags(2, 4, 10, 1, p16, 1.0, p16, 1, p16, 1.0, *([p16] * 7), -1,
                                                *([p16] * 6), null, p16, 1 << 20, 6, null) == -1
    # plan: misaligned buffers, planned constrain without a plan
    assert lib.tli_plan_build(10, 10, p16, p16, ctypes.c_void_p(24), null) == -1
    assert lib.tli_plan_build(1 << 23, 10, p16, p16, p16, null) == -2
    assert lib.tli_constrain_map_planned(4, 10, 10, p16, 1, p16, p16, null, 1.0, p16, p16, p16, null, null,
                                         null) == -1
    # q in logit form: t2d and both outputs required, element-aligned logits, T > 0; R = 0 is a no-op
    p17 = ctypes.c_void_p(17)
    assert lib.tli_constrain_map_qlogits(4, 10, 10, p16, 1, p16, null, null, 1.0, p16, p16, p16, p16, p16, null,
                                         null, null) == -1
    assert lib.tli_constrain_map_qlogits(4, 10, 10, p16, 1, p16, p16, null, 1.0, p16, p16, p16, null, p16, null,
                                         null, null) == -1
    assert lib.tli_constrain_map_qlogits(4, 10, 10, p16, 1, p16, p16, null, 1.0, p16, p16, p16, p16, null, null,
                                         null, null) == -1
    assert lib.tli_constrain_map_qlogits(4, 10, 10, p16, 1, p16, p16, null, 1.0, p16, p16, p16, p17, p16, null,
                                         null, null) == -1
    assert lib.tli_constrain_map_qlogits(4, 10, 10, p16, 1, p16, p16, p16, 0.0, p16, p16, p16, p16, p16, null,
                                         null, null) == -1
    # fused expansion: no expansion struct, or one whose k or row count does not match the launch
    assert lib.spec_softmax_topk_expand(p16, 1, 8, 100, 1.0, 1.0, 4, p16, p16, null, null, null, null, null) == -1
    assert lib.spec_softmax_sample_expand(p16, 1, 8, 100, 1.0, p16, p16, p16, null, null, null, null, null) == -1
    pool = sd.new_pool(2, 4, 3, device="cpu")
    ex = sd._expand((pool, 1))
    assert lib.spec_softmax_topk_expand(p16, 1, 8, 100, 1.0, 1.0, 2, p16, p16, null, null, null, ex, null) == -1  # k
    assert lib.spec_softmax_topk_expand(p16, 1, 7, 100, 1.0, 1.0, 4, p16, p16, null, null, null, ex, null) == -1  # R
    assert lib.spec_softmax_sample_expand(p16, 1, 2, 100, 1.0, p16, p16, p16, null, null, null, ex, null) == -1
    for plan in (null, p16):  # k = 4 is not a chain
        assert lib.tli_constrain_map_qlogits(2, 10, 10, p16, 1, p16, p16, plan, 1.0, p16, p16, p16, p16, p16, null,
                                             ex, null) == -1


def test_sizes_and_config_check(lib):
    assert sd.spec_tree_pool_size(8, 6) == 1 + 8 + 5 * 64
    assert sd.spec_tree_pool_size(4, 3) == 37
    assert sd.spec_verify_ws_size(128, 64) >= 128 * 64 * 12
    assert sd.spec_compact_freed_capacity(128, 64, 16) == 128 * 5
    assert sd.spec_compact_freed_capacity(4, 16, 1) == 60
    # plan: 16-byte header, 8 bytes per bitmap word (count rounded up to even), 4 per target (to 4)
    assert sd.tli_plan_bytes(151936, 128256) == 16 + 8 * 4748 + 4 * 128256
    assert sd.tli_plan_bytes(33, 5) == 16 + 8 * 2 + 4 * 8
    assert sd.tli_check_config(1, 4, 5)
    assert not sd.tli_check_config(2, 4, 5)
    assert not sd.tli_check_config(1, 4, 4)
