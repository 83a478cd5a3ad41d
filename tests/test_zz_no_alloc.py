"""spec_verify_greedy_noalloc: greedy verify for callers that cannot allocate
device memory (a plugin handed only its input and output buffers by a host
framework that owns all device memory, or a path that must not call
cudaMalloc).  Its scratch is a fixed array inside the library, so its output
must equal spec_verify_greedy's (with caller scratch) exactly, call after
call, even though every call reuses the same array -- and both must equal the
CPU oracle's greedy commit."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_draft_select_gb300 as sd
from oracle.pipeline import np_logits

pytestmark = pytest.mark.gpu

OUTPUTS = ("committed", "num_committed", "accept_length", "accept_path", "next_root", "walk_info")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_draft_select_gb300.build import build
    build()
    sd.lib()


def random_tree_inputs(seed, B, k, steps, N, V, dtype):
    """A tree from the library's own draft kernels on random draft logits, and
    random target logits whose argmax often matches the drafts."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    pool = sd.new_pool(B, k, steps)
    for s in range(steps):
        rows = B * (1 if s == 0 else k)
        d = (torch.randn((rows, V), generator=g, device="cuda") * 3).to(dtype)
        tp, ti, _ = sd.spec_softmax_topk(d, 1.0, k)
        sd.spec_tree_expand(pool, s, tp, ti)
    root = torch.randint(0, V, (B,), generator=g, device="cuda", dtype=torch.int32)
    seq = torch.randint(16, 2048, (B,), generator=g, device="cuda", dtype=torch.int32)
    tree = sd.spec_build_tree(pool, N, root, seq)
    target = (torch.randn((B, N, V), generator=g, device="cuda") * 3)
    # plant each node's first child token as that row's argmax half of the time
    first = tree["retrieve_next_token"].long().clamp(min=0)
    tok = torch.gather(tree["draft_token"].long(), 1, first)
    plant = (torch.rand((B, N), generator=g, device="cuda") < 0.5) & (tree["retrieve_next_token"] >= 0)
    target.scatter_add_(2, tok.unsqueeze(-1), (plant.float() * 40).unsqueeze(-1))
    budget = torch.randint(1, 12, (B,), generator=g, device="cuda", dtype=torch.int32)
    return tree, target.to(dtype).contiguous(), budget


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_noalloc_matches_scratch_entry_point_on_consecutive_calls(dtype):
    cases = [random_tree_inputs(11, 64, 4, 5, 16, 4097, dtype), random_tree_inputs(12, 37, 3, 4, 10, 1000, dtype)]
    for tree, target, budget in cases:  # two calls in a row, different inputs each time
        ref = sd.spec_verify_greedy(target, tree["draft_token"], tree["retrieve_next_token"],
                                    tree["retrieve_next_sibling"], budget=budget, eos_id=7)
        got = sd.spec_verify_greedy_noalloc(target, tree["draft_token"], tree["retrieve_next_token"],
                                            tree["retrieve_next_sibling"], budget=budget, eos_id=7)
        torch.cuda.synchronize()
        for name in OUTPUTS:
            assert torch.equal(got[name], ref[name]), name
        assert int(ref["accept_length"].max()) >= 2
        o = oracle.verify_greedy(np_logits(target), tree["draft_token"].cpu().numpy(),
                                 tree["retrieve_next_token"].cpu().numpy(), tree["retrieve_next_sibling"].cpu().numpy(),
                                 budget=budget.cpu().numpy(), eos=7)
        for name in OUTPUTS:
            np.testing.assert_array_equal(got[name].cpu().numpy(), o[name], err_msg=name)


def test_noalloc_rejects_batches_above_its_array():
    B, N, V = (1 << 18) // 16 + 1, 16, 2
    target = torch.zeros((B, N, V), dtype=torch.float32, device="cuda")
    ids = torch.zeros((B, N), dtype=torch.int32, device="cuda")
    with pytest.raises(sd.SpecError) as e:
        sd.spec_verify_greedy_noalloc(target, ids, ids, ids)
    assert e.value.rc == -2
