"""CUDA path vs the CPU oracle on the same seeded inputs, through the C ABI.

Bars: integer outputs (indices, tokens, tree fields, accept lengths and
paths, compacted slots) bit-exact; probabilities within 1e-5 absolute; a
sampled token or acceptance decision may differ only where the oracle's
uniform lies within 1e-5 of the decision boundary (counted)."""
import math
import time

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_draft_select_gb300 as sd
from speculative_decoding_draft_select_gb300.pipeline import StepBuffers, run_draft, run_verify
from workloads import CONFIGS, assemble_target, generate

from oracle.pipeline import fetch_request, np_logits, run_request

pytestmark = pytest.mark.gpu

PROB_TOL = 1e-5
BOUNDARY = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_draft_select_gb300.build import build
    build()
    sd.lib()


def dev(x, dtype=None):
    t = torch.as_tensor(x)
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda().contiguous()


def make_logits(rng, R, V, dtype, std=3.0):
    x = rng.normal(0, std, (R, V)).astype(np.float32)
    t = torch.from_numpy(x).to(dtype)
    return t


# ------------------------------------------------------------ softmax/top-k

CASES = [(7, 1, 1), (5, 7, 3), (9, 33, 4), (4, 4095, 8), (3, 4097, 8), (6, 32000, 4), (2, 128256, 8),
         (3, 1000, 16), (2, 3000, 32), (300, 200, 2)]


@pytest.mark.parametrize("R,V,k", CASES)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_softmax_topk_parity(R, V, k, dtype, T):
    rng = np.random.default_rng(R * 1000 + V + k)
    x = make_logits(rng, R, V, dtype)
    if V >= 8:
        x[0, 3] = x[0, 5] = x[0].max() + 1  # tie at the max: lower index first
        x[min(1, R - 1), 2] = float("-inf")
    if R > 2 and V >= 4:
        x[2, 1] = float("nan")
    topk_p, topk_idx, probs = sd.spec_softmax_topk(dev(x), T, k, want_probs=True)
    torch.cuda.synchronize()
    op, oi, oprobs, oflag = oracle.softmax_topk(np_logits(x), T, k, want_probs=True)
    np.testing.assert_array_equal(topk_idx.cpu().numpy(), oi)
    np.testing.assert_allclose(topk_p.cpu().numpy(), op, rtol=0, atol=PROB_TOL)
    np.testing.assert_allclose(probs.cpu().numpy(), oprobs, rtol=0, atol=PROB_TOL)
    # tree scores at a plain softmax (score_T = 1) beside q at T: one pass
    # with two normalisers when q is written, one normaliser when it is not
    rs = torch.empty((R, 2), device="cuda")
    tp1, ti1, pr1 = sd.spec_softmax_topk(dev(x), T, k, want_probs=True, row_stats=rs, score_T=1.0)
    tp2, ti2, _ = sd.spec_softmax_topk(dev(x), T, k, score_T=1.0)
    torch.cuda.synchronize()
    op1, oi1, _, _ = oracle.softmax_topk(np_logits(x), T, k, score_T=1.0)
    np.testing.assert_array_equal(ti1.cpu().numpy(), oi1)
    np.testing.assert_array_equal(ti2.cpu().numpy(), oi1)
    np.testing.assert_allclose(tp1.cpu().numpy(), op1, rtol=0, atol=PROB_TOL)
    np.testing.assert_allclose(tp2.cpu().numpy(), op1, rtol=0, atol=PROB_TOL)
    np.testing.assert_allclose(pr1.cpu().numpy(), oprobs, rtol=0, atol=PROB_TOL)
    if T == 1.0:
        assert torch.equal(tp1, topk_p) and torch.equal(pr1, probs)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_softmax_topk_row_edges(dtype):
    """Rows with equal maxima far apart (lower index first), a long NaN run,
    fewer than k finite keys, a +inf element, and ties at the end of the
    row, against the oracle; topk_p does not depend on whether the
    probabilities are written."""
    rng = np.random.default_rng(17)
    R, V, k, run = 6, 40000, 8, 10048
    x = make_logits(rng, R, V, torch.float32).numpy()
    top = x.max() + 2
    x[0, [25000, 10, 31000, 9]] = [top, top, top - 1, top - 1]
    x[1, run:2 * run] = np.nan
    x[1, 5] = np.nan
    x[2, :] = -np.inf
    x[2, [3, 20000, 39999]] = [1.0, 2.0, 1.0]
    x[3, 12345] = np.inf
    x[4, [run - 1, run, 2 * run - 1, 2 * run]] = [top, top, top - 0.5, top - 0.5]
    x[5, V - 8:] = top
    xt = torch.from_numpy(x).to(dtype)
    stats = sd.new_stats()
    tp, ti, pr = sd.spec_softmax_topk(dev(xt), 0.7, k, want_probs=True, stats=stats)
    rs = torch.empty((R, 2), device="cuda")
    tp2, ti2, _ = sd.spec_softmax_topk(dev(xt), 0.7, k, row_stats=rs)
    torch.cuda.synchronize()
    op, oi, oprobs, _ = oracle.softmax_topk(np_logits(xt), 0.7, k, want_probs=True)
    np.testing.assert_array_equal(ti.cpu().numpy(), oi)
    np.testing.assert_array_equal(ti2.cpu().numpy(), oi)
    np.testing.assert_allclose(tp.cpu().numpy(), op, rtol=0, atol=PROB_TOL)
    assert torch.equal(tp, tp2)
    np.testing.assert_allclose(pr.cpu().numpy(), oprobs, rtol=0, atol=PROB_TOL)
    assert int(stats[sd.STATS["nonfinite_row"]]) == 1
    assert not torch.isfinite(rs[3, 0])
    # the same rows with the scores at T = 1 beside q at 0.7 (two normalisers,
    # both repaired on the NaN rows)
    rs1 = torch.empty((R, 2), device="cuda")
    tp3, ti3, pr3 = sd.spec_softmax_topk(dev(xt), 0.7, k, want_probs=True, row_stats=rs1, score_T=1.0)
    torch.cuda.synchronize()
    op3, oi3, _, _ = oracle.softmax_topk(np_logits(xt), 0.7, k, score_T=1.0)
    np.testing.assert_array_equal(ti3.cpu().numpy(), oi3)
    np.testing.assert_allclose(tp3.cpu().numpy(), op3, rtol=0, atol=PROB_TOL)
    np.testing.assert_allclose(pr3.cpu().numpy(), oprobs, rtol=0, atol=PROB_TOL)
    fin = torch.isfinite(rs[:, 0])
    assert torch.equal(rs1[fin, 0], rs[fin, 0])  # the max does not depend on the temperature
    torch.testing.assert_close(rs1[fin, 1], rs[fin, 1], rtol=1e-5, atol=0)  # Z: another summation order


@pytest.mark.parametrize("k", [8, 32])
def test_softmax_topk_long_equal_runs(k):
    """More equal keys than the candidate buffer holds (the whole-row rank
    fallback) and rows with fewer than k non-NaN keys."""
    R, V = 3, 5000
    x = torch.zeros((R, V))
    x[1, ::3] = float("nan")
    x[2, :] = float("nan")
    x[2, [7, 4000]] = 1.0
    tp, ti, _ = sd.spec_softmax_topk(dev(x), 1.0, k)
    torch.cuda.synchronize()
    op, oi, _, _ = oracle.softmax_topk(np_logits(x), 1.0, k)
    np.testing.assert_array_equal(ti.cpu().numpy(), oi)
    np.testing.assert_allclose(tp.cpu().numpy(), op, rtol=0, atol=PROB_TOL)


def test_softmax_topk_nonfinite_rows_flagged():
    x = torch.full((3, 50), float("-inf"))
    x[1, 7] = float("inf")
    x[2] = torch.randn(50)
    stats = sd.new_stats()
    tp, ti, pr = sd.spec_softmax_topk(dev(x), 1.0, 2, want_probs=True, stats=stats)
    torch.cuda.synchronize()
    assert int(stats[sd.STATS["nonfinite_row"]]) == 2
    assert torch.all(pr[:2] == 0) and torch.all(tp[:2] == 0)
    _, oi, _, _ = oracle.softmax_topk(np_logits(x), 1.0, 2)
    np.testing.assert_array_equal(ti.cpu().numpy(), oi)


# ---------------------------------------------------------------- sampling

@pytest.mark.parametrize("V", [1, 7, 33, 4097, 32000])
@pytest.mark.parametrize("use_probs", [True, False])
def test_sample_parity(V, use_probs):
    rng = np.random.default_rng(V)
    R = 64
    x = make_logits(rng, R, V, torch.bfloat16)
    u = rng.random(R).astype(np.float32)
    u[:3] = [0.0, 0.5, np.nextafter(np.float32(1), np.float32(0))]
    if use_probs:
        _, _, probs, _ = oracle.softmax_topk(np_logits(x), 0.8, 1, want_probs=True)
        probs = probs.astype(np.float32)
        tok, prob = sd.spec_sample(dev(u), probs=dev(probs))
        otok, oprob, margin, _ = oracle.sample(u, probs=probs)
    else:
        tok, prob = sd.spec_sample(dev(u), logits=dev(x), T=0.8)
        otok, oprob, margin, _ = oracle.sample(u, logits=np_logits(x), T=0.8)
    torch.cuda.synchronize()
    tok, prob = tok.cpu().numpy(), prob.cpu().numpy()
    # a token may differ only where u is within 1e-5 of a CDF boundary, and
    # such differences are rare (fp32 vs fp64 rounding of the prefix sums)
    diff = tok != otok
    assert not (diff & (margin >= BOUNDARY)).any()
    assert diff.sum() <= 1
    same = ~diff
    np.testing.assert_allclose(prob[same], oprob[same], atol=PROB_TOL)


@pytest.mark.parametrize("V", [7, 4097, 129280])
def test_sample_with_row_stats_equals_sample_alone(V):
    """Given the row statistics of spec_softmax_topk, spec_sample reads each
    row once and draws exactly what it draws on its own."""
    rng = np.random.default_rng(V + 3)
    R = 48
    x = dev(make_logits(rng, R, V, torch.bfloat16))
    x[5] = float("-inf")  # a row without a finite max
    u = dev(rng.random(R).astype(np.float32))
    rs = torch.empty((R, 2), device="cuda")
    sd.spec_softmax_topk(x, 0.8, 1, row_stats=rs)
    s1, s2 = sd.new_stats(), sd.new_stats()
    a = sd.spec_sample(u, logits=x, T=0.8, stats=s1)
    b = sd.spec_sample(u, logits=x, T=0.8, row_stats=rs, stats=s2)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert torch.equal(s1, s2) and int(s1[sd.STATS["nonfinite_row"]]) == 1


@pytest.mark.parametrize("V", [7, 33, 4097, 32000, 129280])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_softmax_sample_parity(V, dtype):
    """One pass gives the draw of spec_sample, the probabilities of
    spec_softmax_topk and the row maximum; against the oracle (a token may
    differ only within 1e-5 of a CDF boundary)."""
    rng = np.random.default_rng(V + 11)
    R = 40
    x = make_logits(rng, R, V, dtype)
    x[3] = float("-inf")
    x[4, 1] = float("inf")
    if V >= 8:
        x[5, 2] = float("nan")
    u = rng.random(R).astype(np.float32)
    u[:3] = [0.0, 0.5, np.nextafter(np.float32(1), np.float32(0))]
    rs = torch.empty((R, 2), device="cuda")
    stats = sd.new_stats()
    tok, prob, probs = sd.spec_softmax_sample(dev(x), 0.8, dev(u), row_stats=rs, want_probs=True, stats=stats)
    torch.cuda.synchronize()
    xl = np_logits(x)
    otok, oprob, margin, _ = oracle.sample(u, logits=xl, T=0.8)
    _, _, oprobs, _ = oracle.softmax_topk(xl, 0.8, 1, want_probs=True)
    tok, prob = tok.cpu().numpy(), prob.cpu().numpy()
    keys = x.float().numpy()
    keys = np.where(np.isnan(keys), -np.inf, keys)  # NaN counts as -inf
    finite = np.isfinite(keys.max(axis=1))
    diff = (tok != otok) & finite
    assert not (diff & (margin >= BOUNDARY)).any()
    assert diff.sum() <= 1
    same = ~diff & finite
    np.testing.assert_allclose(prob[same], oprob[same], atol=PROB_TOL)
    assert (tok[~finite] == 0).all() and (prob[~finite] == 0).all()
    assert int(stats[sd.STATS["nonfinite_row"]]) == int((~finite).sum()) == 2
    np.testing.assert_allclose(probs.cpu().numpy(), oprobs, rtol=0, atol=PROB_TOL)
    np.testing.assert_array_equal(rs[torch.from_numpy(finite).cuda(), 0].cpu().numpy(),
                                  keys[finite].max(axis=1).astype(np.float32))


# -------------------------------------------------------------------- tree

def oracle_topk_inputs(rng, B, k, steps, ties=False):
    out = []
    for s in range(steps):
        rows = B * (1 if s == 0 else k)
        p = np.sort(rng.uniform(0.001, 1.0, (rows, k)).astype(np.float32), axis=1)[:, ::-1].copy()
        p /= np.float32(k)
        if ties:
            p[::3, 1:] = p[::3, :1]  # equal probabilities inside a row
            p = np.round(p * 64) / 64  # many equal products across rows
        idx = np.stack([rng.choice(50000, k, replace=False) for _ in range(rows)]).astype(np.int32)
        out.append((np.ascontiguousarray(p, np.float32), idx))
    return out


@pytest.mark.parametrize("B,k,steps,N,ties", [(4, 1, 6, 7, False), (64, 4, 5, 16, False), (16, 8, 6, 64, False),
                                              (8, 3, 4, 2, True), (8, 4, 5, 16, True), (3, 2, 3, 11, True),
                                              (2, 16, 3, 200, False), (2, 16, 3, 300, True),
                                              (2, 32, 3, 100, True)])
def test_tree_parity(B, k, steps, N, ties):
    rng = np.random.default_rng(B * 7 + k + N)
    inputs = oracle_topk_inputs(rng, B, k, steps, ties)
    opool = oracle.Pool(B, k, steps)
    gpool = sd.new_pool(B, k, steps)
    for s, (p, idx) in enumerate(inputs):
        oracle.tree_expand(opool, s, p, idx)
        sd.spec_tree_expand(gpool, s, dev(p), dev(idx))
        torch.cuda.synchronize()
        np.testing.assert_array_equal(gpool["frontier_id"].cpu().numpy(), opool.frontier_id)
        np.testing.assert_array_equal(gpool["frontier_score"].cpu().numpy(), opool.frontier_score)
    for name, arr in (("score", opool.score), ("token", opool.token), ("parent", opool.parent),
                      ("qrow", opool.qrow)):
        np.testing.assert_array_equal(gpool[name].cpu().numpy(), arr, err_msg=name)
    root = rng.integers(0, 1000, B).astype(np.int32)
    seq = rng.integers(16, 2048, B).astype(np.int32)
    gt = sd.spec_build_tree(gpool, N, dev(root), dev(seq))
    ot = oracle.build_tree(opool, N, root, seq)
    torch.cuda.synchronize()
    for name in ot:
        np.testing.assert_array_equal(gt[name].cpu().numpy(), ot[name], err_msg=name)


def test_tree_build_detaches_invalid_parents():
    """Pool parents that are not a tree (out of range, negative, a candidate
    outside the selection, the node itself, a later node) must not derail
    the build: the selection (tokens, draft rows) is the oracle's, every
    valid parent is the oracle's, and a node with an invalid parent is
    detached (parent -1, a mask row and depth of its own chain), so that no
    link from the root reaches it."""
    B, k, steps, N = 6, 4, 4, 16
    rng = np.random.default_rng(777)
    inputs = oracle_topk_inputs(rng, B, k, steps, False)
    opool = oracle.Pool(B, k, steps)
    for s, (p, idx) in enumerate(inputs):
        oracle.tree_expand(opool, s, p, idx)
    root = rng.integers(0, 1000, B).astype(np.int32)
    seq = rng.integers(16, 2048, B).astype(np.int32)
    ot = oracle.build_tree(opool, N, root, seq)
    P = opool.score.shape[1]
    # the pool ids of the selected nodes (node n >= 1), from the oracle's tree
    bad = opool.parent.copy()
    planted = {}
    for b in range(B):
        # selected candidates: nodes 1..N-1 in ascending pool-id order
        order = np.argsort(-opool.score[b, 1:], kind="stable")[: N - 1] + 1
        sel = np.sort(order)
        unselected = np.setdiff1d(np.arange(1, P), sel)
        picks = rng.choice(np.arange(1, N - 1), size=5, replace=False)  # node N-1 is "later" than each
        for n, kind in zip(picks, ("range", "negative", "unselected", "self", "later")):
            pid = sel[n - 1]
            if kind == "range":
                bad[b, pid] = P + 3
            elif kind == "negative":
                bad[b, pid] = -5
            elif kind == "unselected":
                bad[b, pid] = unselected[0]
            elif kind == "self":
                bad[b, pid] = pid
            else:
                bad[b, pid] = sel[-1]
            planted[(b, int(n))] = kind
    gpool = sd.new_pool(B, k, steps)
    for name, arr in (("score", opool.score), ("token", opool.token), ("parent", bad), ("qrow", opool.qrow)):
        gpool[name].copy_(torch.from_numpy(np.ascontiguousarray(arr)))
    gt = sd.spec_build_tree(gpool, N, dev(root), dev(seq))
    torch.cuda.synchronize()
    g = {name: t.cpu().numpy() for name, t in gt.items()}
    for name in ("draft_token", "q_row", "retrieve_index"):
        np.testing.assert_array_equal(g[name], ot[name], err_msg=name)
    for b in range(B):
        par = g["parent"][b]
        assert par[0] == -1
        for n in range(1, N):
            if (b, n) in planted:
                assert par[n] == -1, (b, n, planted[(b, n)])
            else:
                assert par[n] == ot["parent"][b, n], (b, n)
            # the node's chain, depth and mask row from the kernel's own parents
            chain, a = [], n
            while a >= 0:
                chain.append(a)
                a = par[a]
            assert g["positions"][b, n] == seq[b] + (len(chain) - 1 if chain[-1] == 0 else len(chain))
            row = np.zeros(N, np.uint8)
            row[chain] = 1
            np.testing.assert_array_equal(g["tree_mask"][b, n], row)
        # the nodes the root's links reach: exactly those whose chain ends at the root
        seen, stack = set(), [0]
        while stack:
            a = stack.pop()
            seen.add(a)
            c = g["retrieve_next_token"][b, a]
            while c > 0:
                stack.append(c)
                c = g["retrieve_next_sibling"][b, c]
        reach = set()
        for n in range(N):
            a = n
            while a > 0:
                a = par[a]
            if a == 0:
                reach.add(n)
        assert seen == reach
        assert not any((b, n) in planted for n in seen)


# ------------------------------------------------------------------ verify

def verify_compare(g, o, b_g, b_o=0, mode="greedy"):
    """True when every output matches the oracle; False for a difference the
    tolerance allows (stochastic mode, the oracle's uniform within 1e-5 of a
    decision boundary); raises otherwise."""
    names = ("committed", "num_committed", "accept_length", "accept_path", "next_root", "walk_info")
    if all(np.array_equal(g[n][b_g].cpu().numpy(), o[n][b_o]) for n in names):
        return True
    if mode == "sample" and o["margin"][b_o] < BOUNDARY:
        return False
    for n in names:
        np.testing.assert_array_equal(g[n][b_g].cpu().numpy(), o[n][b_o], err_msg=f"{n} request {b_g}")
    return True


def chain_meta(B, N):
    nt = np.tile(np.array([n + 1 if n + 1 < N else -1 for n in range(N)], np.int32), (B, 1))
    return nt, np.full((B, N), -1, np.int32)


@pytest.mark.parametrize("V,dtype", [(1000, torch.bfloat16), (4097, torch.bfloat16), (33, torch.float32)])
def test_verify_greedy_chain_eos_budget(V, dtype):
    rng = np.random.default_rng(V)
    B, N = 96, 16
    target = make_logits(rng, B * N, V, dtype).view(B, N, V)
    eos = 5
    # make drafts agree with the target argmax often, plant EOS rows
    am = target.float().argmax(-1).numpy()
    draft = np.where(rng.random((B, N)) < 0.8, np.roll(am, 1, axis=1), rng.integers(0, V, (B, N))).astype(np.int32)
    plant = torch.from_numpy(rng.random((B, N)) < 1 / 8)
    tf = target.float()
    tf[plant, eos] = 50.0
    target = tf.to(dtype)
    budget = rng.integers(0, 20, B).astype(np.int32)
    budget[0] = 0
    nt, ns = chain_meta(B, N)
    g = sd.spec_verify_greedy(dev(target), dev(draft), dev(nt), dev(ns), budget=dev(budget), eos_id=eos)
    o = oracle.verify_greedy(np_logits(target), draft, nt, ns, budget=budget, eos=eos)
    torch.cuda.synchronize()
    for b in range(B):
        for name in ("committed", "num_committed", "accept_length", "accept_path", "next_root", "walk_info"):
            np.testing.assert_array_equal(g[name][b].cpu().numpy(), o[name][b], err_msg=f"{name} {b}")
    assert (o["accept_length"] > 2).any()


def small(cfg_name, **kw):
    return CONFIGS[cfg_name].scaled(**kw)


def run_gpu_pipeline(cfg, work, mode, q_mode="probs"):
    buf = StepBuffers(cfg.kind, cfg.B, cfg.topk, cfg.steps, cfg.N, cfg.V, "cuda", want_q=(mode == "sample"),
                      sampled=(cfg.kind == "chain" and mode == "sample"), V_t=cfg.V_t or None, q_mode=q_mode,
                      q_logit_dtype=cfg.dtype)
    tree = run_draft(buf, work["draft_table"], cfg.T, work["root_token"], work["seq_lens"],
                     draft_u=work["draft_u"], d2t=work.get("d2t"), t2d=work.get("t2d"))
    target = assemble_target(work, tree["q_row"])
    out = run_verify(buf, target, mode, cfg.T, work["coins"], work["u_final"], work.get("budget"),
                     int(work["eos_id"]))
    torch.cuda.synchronize()
    return buf, tree, out


def _oracle_requests(cfg, work, mode, reqs, chunk=64):
    """The oracle's step for each request of reqs, in order, computed on
    every host core: inputs are fetched here a chunk of requests at a time,
    the oracle runs in threads (its C routines release the interpreter lock
    while they compute)."""
    import concurrent.futures
    import os
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1)) as ex:
        for i in range(0, len(reqs), chunk):
            fetched = [fetch_request(cfg, work, b) for b in reqs[i:i + chunk]]
            yield from ex.map(lambda d: run_request(cfg, d, mode), fetched)


def compare_pipeline(cfg, work, mode, reqs, q_mode="probs"):
    buf, tree, out = run_gpu_pipeline(cfg, work, mode, q_mode)
    reqs = list(reqs)
    exact = boundary = 0
    host_tree = {name: tree[name].cpu().numpy() for name in tree}
    names = ("draft_token", "parent", "positions", "tree_mask", "retrieve_index", "retrieve_next_token",
             "retrieve_next_sibling", "q_row")
    for b, (ot, q, target, o, _) in zip(reqs, _oracle_requests(cfg, work, mode, reqs)):
        ov = {name: ot[name][0] + (b * cfg.N if name == "retrieve_index" else 0) for name in names}
        if not all(np.array_equal(host_tree[name][b], ov[name]) for name in names) and o["draft_margin"] < BOUNDARY:
            boundary += 1  # a draft drawn within the tolerance of a CDF boundary: the tree may differ
            continue
        for name in names:
            np.testing.assert_array_equal(host_tree[name][b], ov[name], err_msg=f"{cfg.name} {name} request {b}")
        if verify_compare(out, o, b, 0, mode):
            exact += 1
        else:
            boundary += 1
    return exact, boundary, out


SMALL = {
    "c1": dict(),
    "c2": dict(B=12, V=4097),
    "c3": dict(B=6, V=4097, page_size=0, bytes_per_slot=0),
    "c4": dict(B=16, V=6001, V_t=5003, K=2500),
    "c5": dict(B=48, V=3001),
}


@pytest.mark.parametrize("name,mode,q_mode", [("c1", "greedy", "probs"), ("c1", "sample", "probs"),
                                              ("c1", "sample", "logits"), ("c2", "greedy", "probs"),
                                              ("c3", "sample", "probs"), ("c3", "sample", "logits"),
                                              ("c4", "sample", "probs"), ("c4", "sample", "logits"),
                                              ("c5", "greedy", "probs"), ("c5", "sample", "probs"),
                                              ("c5", "sample", "logits")])
def test_pipeline_small(name, mode, q_mode, boundary_report):
    cfg = small(name, **SMALL[name])
    work = generate(cfg, "cuda")
    exact, boundary, _ = compare_pipeline(cfg, work, mode, range(cfg.B), q_mode)
    if mode == "sample":
        boundary_report(f"{name} small {mode} q={q_mode}", boundary, cfg.B)
    assert exact >= cfg.B - 1, (exact, boundary)


@pytest.mark.parametrize("name,mode,q_mode", [("c1", "greedy", "probs"), ("c1", "sample", "logits"),
                                              ("c2", "greedy", "probs"), ("c3", "sample", "logits"),
                                              ("c3", "sample", "probs"), ("c4", "sample", "logits"),
                                              ("c5", "greedy", "probs"), ("c5", "sample", "logits")])
def test_pipeline_full_size_every_request(name, mode, q_mode, boundary_report):
    """Full-size workloads in the bench's launch configuration (the
    persistent verify at full occupancy, every queue position), compared
    with the oracle request by request for every request of the batch.
    Integer results must be bit-exact; a stochastic request may differ only
    where the oracle's uniform lies within 1e-5 of a decision boundary, and
    such requests are counted and reported."""
    cfg = CONFIGS[name].scaled(page_size=0, bytes_per_slot=0)
    work = generate(cfg, "cuda")
    exact, boundary, out = compare_pipeline(cfg, work, mode, range(cfg.B), q_mode)
    if mode == "sample":
        boundary_report(f"{name} full size {mode} q={q_mode}", boundary, cfg.B)
    assert exact + boundary == cfg.B
    # c5's sampled chain draws 15 drafts per request from 129280-token rows:
    # about two requests in three have a draw within 1e-5 of a CDF boundary,
    # and fp32 sums flip a few percent of those; everything else is exact
    assert exact >= 0.9 * cfg.B, (exact, boundary)
    al = out["accept_length"].float().mean().item()
    assert 0.0 <= al < cfg.N


@pytest.mark.parametrize("B", [24, 200, 400])
def test_verify_sample_tree_given_q_node_order(B):
    """Stochastic tree verify with q in node order (q_row = NULL) on oracle
    trees, including q[y] == 0 children and zero-mass target entries.  The
    batch sizes take each walk layout: 4 CTAs per request while the GPU
    holds all the clusters at once, then 2, then 1."""
    rng = np.random.default_rng(77 + B)
    k, steps, N, V = 3, 4, 12, 257
    opool = oracle.Pool(B, k, steps)
    for s, (p, idx) in enumerate(oracle_topk_inputs(rng, B, k, steps)):
        oracle.tree_expand(opool, s, p, np.ascontiguousarray(idx % V, np.int32))
    t = oracle.build_tree(opool, N, rng.integers(0, V, B).astype(np.int32), np.zeros(B, np.int32))
    target = make_logits(rng, B * N, V, torch.float32, std=2.0).view(B, N, V)
    target[:, :, :5] = float("-inf")
    _, _, q, _ = oracle.softmax_topk(np_logits(target + torch.randn(B, N, V) * 0.7), 1.0, 1, want_probs=True)
    q = q.astype(np.float32).reshape(B, N, V)
    dt = t["draft_token"]
    q[np.arange(B)[:, None], t["parent"].clip(0), dt] *= (rng.random((B, N)) > 0.1)  # some q[y] = 0
    coins = rng.random((B, N)).astype(np.float32)
    uf = rng.random(B).astype(np.float32)
    stats = sd.new_stats()
    g = sd.spec_verify_sample(dev(target), 1.0, dev(q), dev(dt), dev(t["retrieve_next_token"]),
                              dev(t["retrieve_next_sibling"]), dev(coins), dev(uf), stats=stats)
    o = oracle.verify_sample(np_logits(target), 1.0, q, dt, t["retrieve_next_token"], t["retrieve_next_sibling"],
                             coins, uf)
    torch.cuda.synchronize()
    exact = sum(verify_compare(g, o, b, b, "sample") for b in range(B))
    assert exact >= B - 1
    assert int(stats[sd.STATS["q_zero"]]) == o["q_zero"]


def _softmax64(x, T):
    x = x.astype(np.float64) / T
    x = np.where(np.isnan(x), -np.inf, x)
    m = x.max(-1, keepdims=True)
    e = np.where(np.isfinite(m), np.exp(x - np.where(np.isfinite(m), m, 0.0)), 0.0)
    z = e.sum(-1, keepdims=True)
    return np.where(z > 0, e / np.where(z > 0, z, 1.0), 0.0)


def _check_walk_outputs(out, B, N, V):
    """Well-formed verify outputs: 1..N tokens in [0, V) then -1 padding, an
    accepted path from the root of at most num_committed nodes in [1, N)."""
    com = out["committed"].cpu().numpy()
    nc = out["num_committed"].cpu().numpy()
    acc = out["accept_length"].cpu().numpy()
    path = out["accept_path"].cpu().numpy()
    for b in range(B):
        n = int(nc[b])
        assert 1 <= n <= N
        assert ((com[b, :n] >= 0) & (com[b, :n] < V)).all() and (com[b, n:] == -1).all()
        a = int(acc[b])
        assert 0 <= a <= n and a < N
        assert path[b, 0] == 0 and ((path[b, 1:a + 1] >= 1) & (path[b, 1:a + 1] < N)).all()
        assert (path[b, a + 1:] == -1).all()


@pytest.mark.parametrize("mode", ["greedy", "sample"])
def test_verify_links_that_loop_stay_in_bounds(mode):
    """Retrieve links that are not a tree (a sibling cycle among the root's
    children, a child that points back to an earlier node, a node that is
    its own first child and sibling): the walks bound every link chain by N
    hops and every path by N entries, so the launch ends with well-formed
    outputs (the parity suite's adversarial case for the bounds checks)."""
    rng = np.random.default_rng(4242)
    B, N, V, T = 16, 6, 257, 1.0
    nt = np.tile(np.array([1, 3, 1, 3, -1, -1], np.int32), (B, 1))
    ns = np.tile(np.array([-1, 2, 1, 3, -1, -1], np.int32), (B, 1))
    target = rng.normal(0, 2, (B, N, V)).astype(np.float32)
    am = target.argmax(-1)
    # drafts mostly agree with the argmax of the row they are tested on
    draft = rng.integers(0, V, (B, N)).astype(np.int32)
    for n, par in ((1, 0), (2, 0), (3, 1)):
        agree = rng.random(B) < 0.7
        draft[agree, n] = am[agree, par]
    tgt = dev(torch.from_numpy(target))
    if mode == "greedy":
        out = sd.spec_verify_greedy(tgt, dev(draft), dev(nt), dev(ns))
    else:
        q = _softmax64(target + rng.normal(0, 0.3, target.shape), T).astype(np.float32)
        coins = rng.random((B, N)).astype(np.float32)
        u_final = rng.random(B).astype(np.float32)
        out = sd.spec_verify_sample(tgt, T, dev(q), dev(draft), dev(nt), dev(ns), dev(coins), dev(u_final))
    torch.cuda.synchronize()
    _check_walk_outputs(out, B, N, V)


@pytest.mark.parametrize("B", [8, 200])
def test_verify_sample_fallbacks_and_counters(B):
    """zero-to-sglang ch.10 5.1 asks for numerical validity checks in finite
    precision.  Inputs that force each of them, compared with the oracle
    output by output and counter by counter:
      - a residual with no positive mass (q = 2p, above p everywhere): the
        rejection leaves p_cur as it is (residual fallback), twice at a node
        with two rejected children;
      - a target row with no finite logit at a leaf (the bonus draw finds no
        mass: CDF fallback) and at the root (p = 0: every child rejected,
        each residual empty, and the draw finds no mass);
      - q[y] = 0 where p[y] > 0 (accepted, counted);
      - a zero budget on a tree (nothing committed).
    Tree of every request: root -> 1, 2; node 1 -> 3, 4.  At B = 200 the
    walk runs 2 CTAs per request instead of 4."""
    rng = np.random.default_rng(9090 + B)
    N, V, T = 5, 4097, 0.9
    nt = np.tile(np.array([1, 3, -1, -1, -1], np.int32), (B, 1))
    ns = np.tile(np.array([-1, 2, -1, 4, -1], np.int32), (B, 1))
    parent = np.array([-1, 0, 0, 1, 1])
    target = rng.normal(0, 2, (B, N, V)).astype(np.float32)
    q = _softmax64(target + rng.normal(0, 0.6, (B, N, V)).astype(np.float32), T).astype(np.float32)
    p = _softmax64(target, T).astype(np.float32)
    # drafts: each child drawn from its parent's q row (distinct siblings)
    dt = np.zeros((B, N), np.int32)
    for b in range(B):
        for n in (1, 3):
            w = q[b, parent[n]].astype(np.float64)
            a = rng.choice(V, 2, replace=False, p=w / w.sum())
            dt[b, n], dt[b, n + 1] = a
    coins = rng.random((B, N)).astype(np.float32)
    uf = rng.random(B).astype(np.float32)
    budget = np.full(B, 100, np.int32)
    # request 1: q = 2p at the root, both children rejected -> 2 residual fallbacks
    q[1, 0] = 2 * p[1, 0]
    coins[1, 1] = coins[1, 2] = 0.9
    # request 2: path 0 -> 1 -> 3 accepted (q = p, coins 0), leaf row with no finite logit
    q[2, 0], q[2, 1] = p[2, 0], p[2, 1]
    coins[2, 1] = coins[2, 3] = 0.0
    target[2, 3] = -np.inf
    # request 3: a root row of NaN only -> p = 0
    target[3, 0] = np.nan
    # request 4: budget 0 on the tree
    budget[4] = 0
    # request 5: q[y] = 0 for the first child (p[y] > 0): accepted, counted
    q[5, 0, dt[5, 1]] = 0.0
    # request 6: q = 2p at the root; the first child rejected, the second accepted
    q[6, 0] = 2 * p[6, 0]
    coins[6, 1], coins[6, 2] = 0.9, 0.0
    stats = sd.new_stats()
    g = sd.spec_verify_sample(dev(target), T, dev(q), dev(dt), dev(nt), dev(ns), dev(coins), dev(uf),
                              budget=dev(budget), stats=stats)
    o = oracle.verify_sample(target, T, q, dt, nt, ns, coins, uf, budget=budget)
    torch.cuda.synchronize()
    exact = sum(verify_compare(g, o, b, b, "sample") for b in range(B))
    assert exact >= B - 1
    # the forced cases, as the oracle states them
    assert list(o["committed"][1][:1]) != [-1] and o["accept_length"][1] == 0 and o["walk_info"][1][1] == 2
    assert o["accept_length"][2] == 2 and o["walk_info"][2][2] == 2 and o["committed"][2][2] == 0
    assert o["accept_length"][3] == 0 and o["committed"][3][0] == 0
    assert o["num_committed"][4] == 0
    assert o["accept_length"][5] >= 1 and o["accept_length"][6] == 1
    assert o["residual_fallback"] >= 2 + 2 + 1 and o["cdf_fallback"] >= 2 and o["q_zero"] >= 1
    assert o["nonfinite_rows"] == 2
    st = stats.cpu().numpy()
    assert st[sd.STATS["q_zero"]] == o["q_zero"]
    assert st[sd.STATS["residual_fallback"]] == o["residual_fallback"]
    assert st[sd.STATS["cdf_fallback"]] == o["cdf_fallback"]
    # the batched pass sees every row; here the only non-finite rows are on walks
    assert st[sd.STATS["nonfinite_row"]] == o["nonfinite_rows"] == 2
    assert st[sd.STATS["wait_timeout"]] == 0


@pytest.mark.parametrize("B,N,V,q_form", [(8, 4, 33, "probs"), (96, 5, 4097, "probs"), (300, 16, 2053, "logits"),
                                          (1100, 3, 777, "probs"), (40, 5, 128256, "logits"),
                                          (64, 16, 30001, "logits")])
def test_chain_verify_parity(B, N, V, q_form, boundary_report):
    """The chain verify launch (SPEC_VERIFY_CHAIN: every node's test right
    after its row, the draw cut into chunk items) against the oracle on
    chains: drafts drawn from q, EOS planted in the target, budgets (zero
    included), q[y] = 0 children, a non-finite row, and q = 2p rows (no
    residual mass).  Every output and every counter is compared; a request
    may differ only within 1e-5 of a decision boundary."""
    rng = np.random.default_rng(B * 31 + N + V)
    T = 0.8
    eos = 5
    nt, ns = chain_meta(B, N)
    target = rng.normal(0, 2.5, (B, N, V)).astype(np.float32)
    target[rng.random((B, N)) < 0.05, eos] = 30.0  # EOS rows
    dl = target + rng.normal(0, 0.7, (B, N, V)).astype(np.float32)
    q = _softmax64(dl, T).astype(np.float32)
    p = _softmax64(target, T).astype(np.float32)
    dt = np.zeros((B, N), np.int32)
    for b in range(B):
        for n in range(1, N):
            w = q[b, n - 1].astype(np.float64)
            dt[b, n] = rng.choice(V, p=w / w.sum())
    coins = rng.random((B, N)).astype(np.float32)
    uf = rng.random(B).astype(np.float32)
    budget = rng.integers(0, N + 2, B).astype(np.int32)
    budget[1] = 0
    q[2, 0, dt[2, 1]] = 0.0  # q[y] = 0 with p[y] > 0
    budget[2] = N
    coins[3, 1:] = 0.0       # request 3 accepts everything it can
    target[3, N - 1] = -np.inf  # ... up to a leaf row without a finite logit
    budget[3] = N + 5
    q[4, 0] = 2 * p[4, 0]    # no residual mass at request 4's root
    coins[4, 1] = 0.9
    budget[4] = N
    stats = sd.new_stats()
    if q_form == "probs":
        out = sd.spec_verify_sample(dev(target), T, dev(q), dev(dt), dev(nt), dev(ns), dev(coins), dev(uf),
                                    budget=dev(budget), eos_id=eos, stats=stats, chain=True)
    else:
        # q in logit form: the draft logits with their (max, normaliser) at T
        dlt = dev(dl.reshape(B * N, V))
        rs = torch.empty((B * N, 2), device="cuda")
        sd.spec_softmax_topk(dlt, T, 1, row_stats=rs)
        out = sd.spec_verify_sample_qlogits(dev(target), T, dlt, rs, T, dev(dt), dev(nt), dev(ns), dev(coins),
                                            dev(uf), budget=dev(budget), eos_id=eos, stats=stats, chain=True)
        # the oracle reads the same q values the logit form gives (the GPU's
        # own written probabilities would equal them bit for bit)
        qprobs = torch.empty((B * N, V), device="cuda")
        sd.spec_softmax_topk(dlt, T, 1, probs=qprobs)
        q = qprobs.view(B, N, V).cpu().numpy()
    o = oracle.verify_sample(target, T, q, dt, nt, ns, coins, uf, budget=budget, eos=eos)
    torch.cuda.synchronize()
    exact = sum(verify_compare(out, o, b, b, "sample") for b in range(B))
    boundary_report(f"chain verify B={B} N={N} V={V} q={q_form}", B - exact, B)
    assert exact >= B - max(1, B // 100)
    if q_form == "logits":
        # the same launch with the committed ids mapped back through a table
        # (TLI's target-to-draft map, fused): identical outputs plus the map
        table = rng.integers(-1, 3 * V, V + 7).astype(np.int32)
        out2 = sd.spec_verify_sample_qlogits(dev(target), T, dlt, rs, T, dev(dt), dev(nt), dev(ns), dev(coins),
                                             dev(uf), budget=dev(budget), eos_id=eos, chain=True,
                                             id_map=(dev(table), 77))
        torch.cuda.synchronize()
        for name in ("committed", "num_committed", "accept_length", "accept_path", "next_root", "walk_info"):
            assert torch.equal(out2[name], out[name]), name
        com = out2["committed"].cpu().numpy()
        want = np.where(com >= 0, oracle.map_ids(com, table, 77), -1)
        np.testing.assert_array_equal(out2["committed_mapped"].cpu().numpy(), want)
    st = stats.cpu().numpy()
    for name in ("q_zero", "residual_fallback", "cdf_fallback"):
        assert st[sd.STATS[name]] == o[name], name
    assert st[sd.STATS["nonfinite_row"]] == int((~np.isfinite(np.where(np.isnan(target), -np.inf, target).max(-1))).sum())
    assert st[sd.STATS["wait_timeout"]] == 0 and st[sd.STATS["bad_request"]] == 0
    assert int(out["num_committed"][1]) == 0
    if q_form == "probs":
        assert o["q_zero"] >= 1 and o["residual_fallback"] >= 1


@pytest.mark.parametrize("B,q_form", [(24, "probs"), (200, "probs"), (400, "probs"), (24, "logits"),
                                      (400, "logits")])
def test_verify_sample_without_replacement(B, q_form):
    """The without-replacement sibling update (q loses each rejected token
    and is renormalised) against the oracle's, on oracle trees whose
    siblings sometimes repeat a token (V is small), in each walk layout (4,
    2 and 1 CTAs per request) and with q written or in logit form."""
    rng = np.random.default_rng(177 + B)
    k, steps, N, V = 3, 4, 12, 257
    opool = oracle.Pool(B, k, steps)
    for s, (p, idx) in enumerate(oracle_topk_inputs(rng, B, k, steps)):
        oracle.tree_expand(opool, s, p, np.ascontiguousarray(idx % V, np.int32))
    t = oracle.build_tree(opool, N, rng.integers(0, V, B).astype(np.int32), np.zeros(B, np.int32))
    target = make_logits(rng, B * N, V, torch.float32, std=2.0).view(B, N, V)
    target[:, :, :5] = float("-inf")
    dl = (target.view(B * N, V) + torch.from_numpy(rng.normal(0, 0.7, (B * N, V)).astype(np.float32)))
    dl[:, :5] = 0.0
    dt, par = t["draft_token"], t["parent"]
    # the draft puts much of its mass on the children it proposed (so that
    # removing a rejected child's q matters), the target somewhat less
    for b in range(B):
        for n in range(1, N):
            dl[b * N + par[b, n], dt[b, n]] += 3.0
            target[b, par[b, n], dt[b, n]] += 2.0
    _, _, q, _ = oracle.softmax_topk(np_logits(dl), 1.0, 1, want_probs=True)
    q = q.astype(np.float32).reshape(B, N, V)
    coins = rng.random((B, N)).astype(np.float32)
    uf = rng.random(B).astype(np.float32)
    stats = sd.new_stats()
    args = (dev(dt), dev(t["retrieve_next_token"]), dev(t["retrieve_next_sibling"]), dev(coins), dev(uf))
    if q_form == "probs":
        g = sd.spec_verify_sample(dev(target), 1.0, dev(q), *args, stats=stats, without_replacement=True)
    else:
        st = torch.empty((B * N, 2), dtype=torch.float32, device="cuda")
        sd.spec_softmax_topk(dev(dl), 1.0, 1, row_stats=st)
        g = sd.spec_verify_sample_qlogits(dev(target), 1.0, dev(dl), st, 1.0, *args, stats=stats,
                                          without_replacement=True)
    o = oracle.verify_sample(np_logits(target), 1.0, q, dt, t["retrieve_next_token"], t["retrieve_next_sibling"],
                             coins, uf, without_replacement=True)
    torch.cuda.synchronize()
    exact = sum(verify_compare(g, o, b, b, "sample") for b in range(B))
    assert exact >= B - max(1, B // 100)
    if exact == B:
        assert int(stats[sd.STATS["q_zero"]]) == o["q_zero"]
    # the inputs tell the two updates apart
    o_r = oracle.verify_sample(np_logits(target), 1.0, q, dt, t["retrieve_next_token"], t["retrieve_next_sibling"],
                               coins, uf)
    assert any(not np.array_equal(o["committed"][b], o_r["committed"][b]) for b in range(B))
    # and the default call still follows the fixed-q rule
    g_r = sd.spec_verify_sample(dev(target), 1.0, dev(q), *args)
    torch.cuda.synchronize()
    assert sum(verify_compare(g_r, o_r, b, b, "sample") for b in range(B)) >= B - max(1, B // 100)


@pytest.mark.parametrize("q_mode", ["probs", "logits"])
def test_pipeline_verify_without_replacement(q_mode):
    """run_verify(without_replacement=True) is the flagged verify call on
    the step's buffers."""
    cfg = small("c3", **SMALL["c3"])
    work = generate(cfg, "cuda")
    buf = StepBuffers(cfg.kind, cfg.B, cfg.topk, cfg.steps, cfg.N, cfg.V, "cuda", want_q=True, q_mode=q_mode,
                      q_logit_dtype=cfg.dtype)
    tree = run_draft(buf, work["draft_table"], cfg.T, work["root_token"], work["seq_lens"])
    target = assemble_target(work, tree["q_row"])
    vargs = (cfg.T, work["coins"], work["u_final"], work.get("budget"), int(work["eos_id"]))
    got = {n: v.clone() for n, v in run_verify(buf, target, "sample", *vargs, without_replacement=True).items()}
    t = buf.tree
    tree_args = (t["draft_token"], t["retrieve_next_token"], t["retrieve_next_sibling"], work["coins"],
                 work["u_final"])
    kw = dict(q_row=t["q_row"], budget=work.get("budget"), eos_id=int(work["eos_id"]), without_replacement=True)
    if q_mode == "logits":
        want = sd.spec_verify_sample_qlogits(target, cfg.T, buf.draft_table, buf.q_stats, buf.T_draft, *tree_args,
                                             **kw)
    else:
        want = sd.spec_verify_sample(target, cfg.T, buf.q, *tree_args, **kw)
    torch.cuda.synchronize()
    for n in got:
        assert torch.equal(got[n], want[n]), n
    assert int(got["num_committed"].sum()) > 0


@pytest.mark.parametrize("qdtype", [torch.bfloat16, torch.float32])
def test_q_in_logit_form_equals_written_q(qdtype):
    """spec_verify_sample_qlogits on (draft logits, row max/normaliser) gives
    exactly spec_verify_sample's result on the probabilities the draft kernel
    writes for the same rows."""
    rng = np.random.default_rng(5)
    B, k, steps, N, V = 16, 4, 4, 14, 3001
    cfg = CONFIGS["c3"].scaled(B=B, topk=k, steps=steps, N=N, V=V, dtype=qdtype, page_size=0, bytes_per_slot=0)
    work = generate(cfg, "cuda")
    outs = []
    for q_mode in ("probs", "logits"):
        buf, tree, out = run_gpu_pipeline(cfg, work, "sample", q_mode)
        outs.append({n: v.clone() for n, v in out.items()})
    for n in outs[0]:
        assert torch.equal(outs[0][n], outs[1][n]), n
    assert int(outs[0]["accept_length"].sum()) > 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_tli_q_in_logit_form_equals_written_q(dtype):
    """The TLI step with q in logit form (the partners' logits in target
    order and each row's max and normaliser, read by
    spec_verify_sample_qlogits) verifies exactly as with the fp32 q rows."""
    cfg = small("c4", **SMALL["c4"]).scaled(dtype=dtype)
    work = generate(cfg, "cuda")
    outs = []
    for q_mode in ("probs", "logits"):
        buf, tree, out = run_gpu_pipeline(cfg, work, "sample", q_mode)
        outs.append(({n: v.clone() for n, v in out.items()}, {n: v.clone() for n, v in tree.items()}))
    for n in outs[0][1]:
        assert torch.equal(outs[0][1][n], outs[1][1][n]), n
    for n in outs[0][0]:
        assert torch.equal(outs[0][0][n], outs[1][0][n]), n
    assert int(outs[0][0]["accept_length"].sum()) > 0


def test_tli_plan_follows_the_maps():
    """The pipeline builds the map plan once per pair of maps and builds it
    again when they change (here in place): after the change, the plan and
    the draft outputs equal those of fresh buffers."""
    cfg = small("c4", **SMALL["c4"])
    work = generate(cfg, "cuda")
    d2t, t2d = work["d2t"], work["t2d"]

    def fresh():
        return StepBuffers(cfg.kind, cfg.B, cfg.topk, cfg.steps, cfg.N, cfg.V, "cuda", want_q=True, V_t=cfg.V_t,
                           q_mode="logits", q_logit_dtype=cfg.dtype)

    def draft(buf):
        tree = run_draft(buf, work["draft_table"], cfg.T, work["root_token"], work["seq_lens"], d2t=d2t, t2d=t2d)
        torch.cuda.synchronize()
        return {n: v.clone() for n, v in tree.items()}, buf.tok.clone(), buf.q.clone()

    buf = fresh()
    draft(buf)
    key, plan0 = buf.tli_plan_key, buf.tli_plan.clone()
    draft(buf)
    assert buf.tli_plan_key == key  # same maps: not rebuilt
    # swap the target partners of two intersection ids, in place
    ids = torch.nonzero(d2t >= 0).flatten()[:2].tolist()
    ta, tb = int(d2t[ids[0]]), int(d2t[ids[1]])
    d2t[ids[0]], d2t[ids[1]] = tb, ta
    t2d[ta], t2d[tb] = ids[1], ids[0]
    got = draft(buf)
    assert buf.tli_plan_key != key
    assert not torch.equal(buf.tli_plan[16:], plan0[16:])
    ref_buf = fresh()
    want = draft(ref_buf)
    # every byte but the header's three pad words (bytes 4..15, never written)
    assert torch.equal(buf.tli_plan[:4], ref_buf.tli_plan[:4])
    assert torch.equal(buf.tli_plan[16:], ref_buf.tli_plan[16:])
    for n in got[0]:
        assert torch.equal(got[0][n], want[0][n]), n
    assert torch.equal(got[1], want[1]) and torch.equal(got[2], want[2])


def tli_check_qlogits(x, d2t, t2d, T, o, plan):
    """tli_constrain_map_qlogits against the oracle: the same top-1 outputs,
    the partners' logits bit for bit (-inf without a partner), m the top-1
    logit and Z = 1 / its probability, and the q they define."""
    Vd, Vt = x.shape[1], len(t2d)
    td, tt, tp, ql, qs = sd.tli_constrain_map_qlogits(dev(x), dev(d2t), dev(t2d), T, plan=plan)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(td.cpu().numpy(), o["top1_draft"])
    np.testing.assert_array_equal(tt.cpu().numpy(), o["top1_target"])
    np.testing.assert_allclose(tp.cpu().numpy(), o["top1_p"], atol=PROB_TOL)
    ok_t = (t2d >= 0) & (t2d < Vd)
    want = torch.full((x.shape[0], Vt), float("-inf"), dtype=x.dtype)
    want[:, torch.from_numpy(np.nonzero(ok_t)[0])] = x[:, torch.from_numpy(t2d[ok_t].astype(np.int64))]
    ibits = torch.int16 if x.dtype == torch.bfloat16 else torch.int32
    assert torch.equal(ql.cpu().view(ibits), want.view(ibits))
    qs = qs.cpu().numpy().astype(np.float64)
    full = o["top1_draft"] >= 0
    xf = x.float().numpy().astype(np.float64)
    np.testing.assert_array_equal(qs[full, 0], xf[np.nonzero(full)[0], o["top1_draft"][full]])
    np.testing.assert_allclose(qs[full, 1], 1.0 / o["top1_p"][full], rtol=1e-5)
    assert np.all(qs[~full, 0] == -np.inf)
    key = ql.cpu().float().numpy().astype(np.float64)
    key[np.isnan(key)] = -np.inf
    with np.errstate(invalid="ignore", over="ignore"):
        q = np.where(full[:, None], np.exp((key - qs[:, :1]) / T) / qs[:, 1:], 0.0)
    np.testing.assert_allclose(np.minimum(q, 1.0), o["q_target"], atol=PROB_TOL)


def test_worked_example_monte_carlo_gpu(golden):
    """p=[0.4,0.6], q=[0.8,0.2]: the committed token is 0 with probability
    exactly 0.4 (zero-to-sglang ch.10, section 5.1)."""
    g = golden("stochastic_worked_example.json")
    n = g["monte_carlo"]["trials"]
    gen = torch.Generator(device="cuda").manual_seed(31)
    B, N, V = n, 2, 2
    target = torch.log(torch.tensor([0.4, 0.6], device="cuda")).expand(B, N, V).contiguous()
    q = torch.tensor([0.8, 0.2], device="cuda").expand(B, N, V).contiguous()
    y = (torch.rand(B, generator=gen, device="cuda") >= 0.8).int()
    draft = torch.stack([torch.zeros_like(y), y], 1).contiguous()
    nt = torch.tensor([1, -1], dtype=torch.int32, device="cuda").expand(B, 2).contiguous()
    ns = torch.full((B, 2), -1, dtype=torch.int32, device="cuda")
    coins = torch.rand((B, N), generator=gen, device="cuda")
    uf = torch.rand((B,), generator=gen, device="cuda")
    out = sd.spec_verify_sample(target, 1.0, q, draft, nt, ns, coins, uf)
    f0 = (out["committed"][:, 0] == 0).float().mean().item()
    sigma = math.sqrt(0.4 * 0.6 / n)
    assert abs(f0 - 0.4) < g["monte_carlo"]["sigma_bound"] * sigma
    assert abs(f0 - 0.56) > 100 * sigma


# -------------------------------------------------------------- compaction

@pytest.mark.parametrize("ps,with_kv", [(1, False), (16, True), (16, False), (4, True)])
def test_compact_parity(ps, with_kv):
    cfg = CONFIGS["c3"].scaled(page_size=ps, bytes_per_slot=4096 if with_kv else 0)
    if ps != 16:
        cfg = cfg.scaled(B=40)
    work = generate(cfg, "cuda")
    rng = np.random.default_rng(ps)
    B, N = cfg.B, cfg.N
    acc = rng.integers(0, N, B).astype(np.int32)
    acc[:3] = [0, N - 1, 2]
    path = np.full((B, N), -1, np.int32)
    for b in range(B):
        path[b, :acc[b] + 1] = [0] + sorted(rng.choice(np.arange(1, N), acc[b], replace=False))
    path[2, :3] = [0, 2, 3]  # the race case
    path[1] = np.arange(N)
    seq = work["seq_lens"].cpu().numpy()
    rt_o = work["req_to_token"].cpu().numpy().copy()
    kv_o = work["kv_pool"].cpu().numpy().copy() if with_kv else None
    o = oracle.compact_slots(seq, path, acc, rt_o, ps, kv_pool=kv_o)
    rt_g = work["req_to_token"].clone()
    kv_g = work["kv_pool"] if with_kv else None
    stats = sd.new_stats()
    g = sd.spec_compact_slots(work["seq_lens"], dev(path), dev(acc), rt_g, ps, kv_pool=kv_g, stats=stats)
    torch.cuda.synchronize()
    for name in ("move_src", "move_dst", "num_moves", "new_kv_len"):
        np.testing.assert_array_equal(g[name].cpu().numpy(), o[name], err_msg=name)
    nf = int(g["num_freed"].item())
    assert nf == len(o["freed"])
    np.testing.assert_array_equal(g["freed"][:nf].cpu().numpy(), o["freed"])
    np.testing.assert_array_equal(rt_g.cpu().numpy(), rt_o)
    if with_kv:
        assert np.array_equal(kv_g.cpu().numpy(), kv_o)
    assert int(stats[sd.STATS["bad_request"]]) == int(o["bad"][0])


@pytest.mark.parametrize("ps", [1, 4])
def test_compact_many_requests_and_bad_ones(ps):
    """More requests than one round of the index kernel (128 lane groups),
    a path longer than a lane group, and requests the kernel must skip: an
    accept length out of range, a path that does not increase, a path that
    does not start at 0, a sequence that would overflow max_ctx."""
    rng = np.random.default_rng(40 + ps)
    B, N, max_ctx = 300, 21, 64
    seq = rng.integers(0, max_ctx - N, B).astype(np.int32)
    slots = rng.permutation(B * max_ctx).astype(np.int32).reshape(B, max_ctx)
    acc = rng.integers(0, N, B).astype(np.int32)
    acc[:4] = [N - 1, N - 1, 13, 0]
    path = np.full((B, N), -1, np.int32)
    for b in range(B):
        path[b, :acc[b] + 1] = [0] + sorted(rng.choice(np.arange(1, N), acc[b], replace=False))
    acc[5] = N          # out of range
    acc[6] = max(acc[6], 2)
    path[6, :3] = [0, 4, 4]  # not increasing
    path[7, 0] = 1      # does not start at 0
    seq[8] = max_ctx - N + 1  # overflows max_ctx
    rt_o = slots.copy()
    o = oracle.compact_slots(seq, path, acc, rt_o, ps)
    rt_g = dev(slots)
    stats = sd.new_stats()
    g = sd.spec_compact_slots(dev(seq), dev(path), dev(acc), rt_g, ps, stats=stats)
    torch.cuda.synchronize()
    for name in ("move_src", "move_dst", "num_moves", "new_kv_len"):
        np.testing.assert_array_equal(g[name].cpu().numpy(), o[name], err_msg=name)
    nf = int(g["num_freed"].item())
    assert nf == len(o["freed"])
    np.testing.assert_array_equal(g["freed"][:nf].cpu().numpy(), o["freed"])
    np.testing.assert_array_equal(rt_g.cpu().numpy(), rt_o)
    assert int(stats[sd.STATS["bad_request"]]) == int(o["bad"][0]) >= 4


def _pools_equal(a, b):
    for n in ("score", "token", "parent", "qrow", "frontier_score", "frontier_id", "counters"):
        assert torch.equal(a[n], b[n]), n


@pytest.mark.parametrize("B,k,steps,V", [(5, 8, 4, 3000), (9, 4, 3, 1000), (7, 1, 5, 777), (3, 32, 2, 4096),
                                         (400, 8, 2, 600)])
def test_fused_expansion_equals_separate_launches(B, k, steps, V):
    """A draft launch with the step's expansion fused writes the same pool
    and frontier as the draft launch followed by spec_tree_expand (the last
    CTA of a request's rows expands it; counters return to zero)."""
    rng = np.random.default_rng(B * 100 + k)
    pa, pb = sd.new_pool(B, k, steps), sd.new_pool(B, k, steps)
    for s in range(steps):
        R = B if s == 0 else B * k
        x = dev(make_logits(rng, R, V, torch.bfloat16))
        ta = sd.spec_softmax_topk(x, 0.8, k)
        sd.spec_tree_expand(pa, s, ta[0], ta[1])
        tb = sd.spec_softmax_topk(x, 0.8, k, expand=(pb, s))
        torch.cuda.synchronize()
        assert torch.equal(ta[0], tb[0]) and torch.equal(ta[1], tb[1])
        _pools_equal(pa, pb)


def test_fused_expansion_sampled_chain_and_tli():
    """The same for the fused sampler (chain, k = 1) and the planned TLI
    kernel."""
    rng = np.random.default_rng(12)
    B, steps, V = 33, 4, 5000
    pa, pb = sd.new_pool(B, 1, steps), sd.new_pool(B, 1, steps)
    for s in range(steps):
        x = dev(make_logits(rng, B, V, torch.bfloat16))
        u = dev(rng.random(B).astype(np.float32))
        ta = sd.spec_softmax_sample(x, 0.9, u)
        sd.spec_tree_expand(pa, s, ta[1], ta[0])
        tb = sd.spec_softmax_sample(x, 0.9, u, expand=(pb, s))
        torch.cuda.synchronize()
        assert torch.equal(ta[0], tb[0]) and torch.equal(ta[1], tb[1])
        _pools_equal(pa, pb)
    Vd, Vt, K = 4097, 3001, 1500
    dids = np.sort(rng.choice(Vd, K, replace=False))
    tids = rng.choice(Vt, K, replace=False)
    d2t = np.full(Vd, -1, np.int32)
    d2t[dids] = tids
    t2d = np.full(Vt, -1, np.int32)
    t2d[tids] = dids
    plan = sd.tli_plan_build(dev(d2t), dev(t2d))
    pa, pb = sd.new_pool(B, 1, steps), sd.new_pool(B, 1, steps)
    for s in range(steps):
        x = dev(make_logits(rng, B, Vd, torch.bfloat16))
        ta = sd.tli_constrain_map(x, dev(d2t), 1.0, t2d=dev(t2d), want_q=True, plan=plan)
        sd.spec_tree_expand(pa, s, ta[2], ta[1])
        tb = sd.tli_constrain_map(x, dev(d2t), 1.0, t2d=dev(t2d), want_q=True, plan=plan, expand=(pb, s))
        torch.cuda.synchronize()
        for u_, v_ in zip(ta, tb):
            assert torch.equal(u_, v_)
        _pools_equal(pa, pb)


def test_bounded_wait_runs_out_and_the_context_stays_usable():
    """The flag wait of the stochastic verify, on a flag that nothing sets:
    it gives up after its limit, counts the timeout, and the next launches
    run normally (a set flag is seen at once)."""
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    stats = sd.new_stats()
    t0 = time.perf_counter()
    seen = sd.spec_wait_probe(flag, 4_000_000, stats=stats)  # about 2 ms of SM clock
    torch.cuda.synchronize()
    assert int(seen.item()) == 0
    assert int(stats[sd.STATS["wait_timeout"]]) == 1
    assert time.perf_counter() - t0 < 5.0
    flag.fill_(1)
    seen = sd.spec_wait_probe(flag, 4_000_000, stats=stats)
    torch.cuda.synchronize()
    assert int(seen.item()) == 1
    assert int(stats[sd.STATS["wait_timeout"]]) == 1
    # the context is intact: a verify launch afterwards matches the oracle
    rng = np.random.default_rng(3)
    B, N, V = 8, 4, 300
    target = make_logits(rng, B * N, V, torch.float32).view(B, N, V)
    draft = rng.integers(0, V, (B, N)).astype(np.int32)
    nt, ns = chain_meta(B, N)
    g = sd.spec_verify_greedy(dev(target), dev(draft), dev(nt), dev(ns))
    o = oracle.verify_greedy(np_logits(target), draft, nt, ns)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(g["committed"].cpu().numpy(), o["committed"])


# --------------------------------------------------------------------- TLI

# Cases: the resident-bitmap kernel with the intersection logits in shared
# memory (bf16), with more rows than CTAs (each CTA walks several rows), with
# fp32 logits too many to hold (gathers from the row), and a draft
# vocabulary too large for the bitmap (one CTA per row, mask from d2t).
@pytest.mark.parametrize("Vd,Vt,K,dtype,R", [(4097, 3001, 1500, torch.bfloat16, 24),
                                             (151936, 128256, 60000, torch.bfloat16, 200),
                                             (37, 29, 11, torch.float32, 24),
                                             (4101, 999, 700, torch.bfloat16, 700),
                                             (151936, 128256, 60000, torch.float32, 24),
                                             (1000003, 50000, 30000, torch.bfloat16, 6)])
def test_tli_parity(Vd, Vt, K, dtype, R):
    rng = np.random.default_rng(Vd)
    dids = np.sort(rng.choice(Vd, K, replace=False))
    tids = rng.choice(Vt, K, replace=False)
    d2t = np.full(Vd, -1, np.int32)
    d2t[dids] = tids
    t2d = np.full(Vt, -1, np.int32)
    t2d[tids] = dids
    x = make_logits(rng, R, Vd, dtype)
    x[3, torch.from_numpy(dids)] = float("-inf")  # empty after masking
    x[4, int(dids[2])] = x[4, int(dids[5])] = 40.0  # tie inside the intersection
    o = oracle.tli_constrain_map(np_logits(x), d2t, t2d, 0.9, want_q=True)
    plan = sd.tli_plan_build(dev(d2t), dev(t2d))
    for p in (None, plan):
        stats = sd.new_stats()
        td, tt, tp, qt = sd.tli_constrain_map(dev(x), dev(d2t), 0.9, t2d=dev(t2d), want_q=True, stats=stats, plan=p)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(td.cpu().numpy(), o["top1_draft"])
        np.testing.assert_array_equal(tt.cpu().numpy(), o["top1_target"])
        np.testing.assert_allclose(tp.cpu().numpy(), o["top1_p"], atol=PROB_TOL)
        np.testing.assert_allclose(qt.cpu().numpy(), o["q_target"], atol=PROB_TOL)
        assert int(stats[sd.STATS["empty_intersection"]]) == int(o["row_flag"].sum()) == 1
        # without q the top-1 outputs are the same
        td2, tt2, tp2, _ = sd.tli_constrain_map(dev(x), dev(d2t), 0.9, t2d=dev(t2d), plan=p)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(td2.cpu().numpy(), o["top1_draft"])
        np.testing.assert_allclose(tp2.cpu().numpy(), o["top1_p"], atol=PROB_TOL)
        # q in logit form
        tli_check_qlogits(x, d2t, t2d, 0.9, o, p)
    ids = np.concatenate([dids[:100], np.setdiff1d(np.arange(Vd), dids)[:50], [-3, Vd, Vd + 9]]).astype(np.int32)
    g = sd.tli_map_ids(dev(ids), dev(d2t), 7)
    np.testing.assert_array_equal(g.cpu().numpy(), oracle.map_ids(ids, d2t, 7))
    back = sd.tli_map_ids(sd.tli_map_ids(dev(dids.astype(np.int32)), dev(d2t), -1), dev(t2d), -1)
    np.testing.assert_array_equal(back.cpu().numpy(), dids)


def test_tli_t2d_outside_intersection():
    """A target id whose t2d entry names a draft id outside the intersection
    reads that id's logit from the row (the map is taken as given); ids past
    the draft vocabulary give 0."""
    Vd, Vt, K, R = 5000, 3000, 1200, 8
    rng = np.random.default_rng(5)
    dids = np.sort(rng.choice(Vd, K, replace=False))
    tids = rng.choice(Vt, K, replace=False)
    d2t = np.full(Vd, -1, np.int32)
    d2t[dids] = tids
    t2d = np.full(Vt, -1, np.int32)
    t2d[tids] = dids
    outside = np.setdiff1d(np.arange(Vd), dids)[:5]
    free_t = np.setdiff1d(np.arange(Vt), tids)[:6]
    t2d[free_t[:5]] = outside
    x = make_logits(rng, R, Vd, torch.bfloat16)
    x[:, torch.from_numpy(outside)] = -2.0  # below the row's masked max: q stays below 1
    o = oracle.tli_constrain_map(np_logits(x), d2t, t2d, 0.8, want_q=True)
    t2d[free_t[5]] = Vd + 3  # past the vocabulary: 0 (the oracle row keeps 0 there)
    for p in (None, sd.tli_plan_build(dev(d2t), dev(t2d))):
        td, tt, tp, qt = sd.tli_constrain_map(dev(x), dev(d2t), 0.8, t2d=dev(t2d), want_q=True, plan=p)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(td.cpu().numpy(), o["top1_draft"])
        np.testing.assert_allclose(qt.cpu().numpy(), o["q_target"], atol=PROB_TOL)
        tli_check_qlogits(x, d2t, t2d, 0.8, o, p)
    assert (o["q_target"][:, free_t[:5]] > 0).all()


@pytest.mark.parametrize("Vd,Vt,K", [(151936, 128256, 60000), (33, 5, 3), (64, 64, 0), (100003, 7, 7)])
def test_tli_plan_parity(Vd, Vt, K):
    """The plan tli_plan_build writes equals the oracle's, word for word."""
    rng = np.random.default_rng(K + Vd)
    dids = np.sort(rng.choice(Vd, K, replace=False))
    tids = rng.choice(Vt, K, replace=False)
    d2t = np.full(Vd, -1, np.int32)
    d2t[dids] = tids
    t2d = np.full(Vt, -1, np.int32)
    t2d[tids] = dids
    free = np.setdiff1d(np.arange(Vt), tids)
    if len(free) >= 2:
        t2d[free[0]] = np.setdiff1d(np.arange(Vd), dids)[0]  # a partner outside the intersection
        t2d[free[1]] = Vd  # past the vocabulary
    o = oracle.tli_plan(d2t, t2d)
    g = sd.tli_plan_build(dev(d2t), dev(t2d)).cpu().numpy()
    words = len(o["bits"])
    assert g.size == sd.tli_plan_bytes(Vd, Vt) == 16 + 8 * words + 4 * len(o["t2r"])
    assert int(g[:4].view(np.int32)[0]) == int(o["K"][0])
    mw = g[16:16 + 8 * words].view(np.uint32).reshape(words, 2)
    np.testing.assert_array_equal(mw[:, 0], o["bits"])
    np.testing.assert_array_equal(mw[:, 1], o["before"])
    np.testing.assert_array_equal(g[16 + 8 * words:].view(np.int32), o["t2r"])


# ------------------------------------------------------- toy LM end to end

def test_greedy_spec_decoding_on_gpu_equals_argmax_decoding():
    """Rounds of draft tree -> verify on the GPU reproduce plain argmax
    decoding of the target (zero-to-sglang ch.10, 4.2: every committed token
    is the target's choice on the committed prefix)."""
    rng = np.random.default_rng(12)
    V, k, S, N = 40, 3, 3, 8
    tab = torch.from_numpy(rng.normal(0, 2, (V * V, V)).astype(np.float32))
    dtab = tab + torch.from_numpy(rng.normal(0, 0.8, tab.shape).astype(np.float32))
    tab_g, dtab_g = tab.cuda(), dtab.cuda()
    ctx = [3, 17]
    ref = list(ctx)
    for _ in range(50):
        ref.append(int(torch.argmax(tab[ref[-2] * V + ref[-1]])))
    out = list(ctx)
    while len(out) < len(ref):
        pool = sd.new_pool(1, k, S)
        pctx = {0: tuple(out)}
        rows = dtab_g[[pctx[0][-2] * V + pctx[0][-1]]]
        for s in range(S):
            tp, ti, _ = sd.spec_softmax_topk(rows.contiguous(), 1.0, k)
            sd.spec_tree_expand(pool, s, tp, ti)
            tok = pool["token"][0].cpu().numpy()
            par = pool["parent"][0].cpu().numpy()
            lo = 1 if s == 0 else 1 + k + (s - 1) * k * k
            hi = 1 + k if s == 0 else lo + k * k
            for pid in range(lo, hi):
                pctx[pid] = pctx[int(par[pid])] + (int(tok[pid]),)
            fr = pool["frontier_id"][0].cpu().numpy()
            rows = dtab_g[[pctx[int(f)][-2] * V + pctx[int(f)][-1] for f in fr]]
        t = sd.spec_build_tree(pool, N, dev(np.array([out[-1]], np.int32)), dev(np.array([len(out)], np.int32)))
        par = t["parent"][0].cpu().numpy()
        dtk = t["draft_token"][0].cpu().numpy()
        nctx = [tuple(out)]
        for n in range(1, N):
            nctx.append(nctx[par[n]] + (int(dtk[n]),))
        target = torch.stack([tab_g[c[-2] * V + c[-1]] for c in nctx])[None].contiguous()
        v = sd.spec_verify_greedy(target, t["draft_token"], t["retrieve_next_token"], t["retrieve_next_sibling"])
        nc = int(v["num_committed"][0])
        out += v["committed"][0, :nc].cpu().tolist()
    assert out[:len(ref)] == ref


@pytest.mark.parametrize("name,mode,q_mode", [("c3", "sample", "logits"), ("c5", "greedy", "probs"),
                                              ("c4", "sample", "probs")])
def test_captured_step_replays_the_eager_step(name, mode, q_mode):
    """A whole step (draft steps, tree build, verify, compaction) captured in
    a CUDA graph and replayed writes exactly what the eager step wrote."""
    from speculative_decoding_draft_select_gb300.pipeline import capture_step, run_compact
    cfg = small(name, **SMALL[name])
    if name == "c3":
        cfg = cfg.scaled(page_size=16, bytes_per_slot=64)
    work = generate(cfg, "cuda")
    buf = StepBuffers(cfg.kind, cfg.B, cfg.topk, cfg.steps, cfg.N, cfg.V, "cuda", want_q=(mode == "sample"),
                      sampled=(cfg.kind == "chain" and mode == "sample"), V_t=cfg.V_t or None,
                      page_size=cfg.page_size, q_mode=q_mode)
    tree = run_draft(buf, work["draft_table"], cfg.T, work["root_token"], work["seq_lens"],
                     draft_u=work["draft_u"], d2t=work.get("d2t"), t2d=work.get("t2d"))
    target = assemble_target(work, tree["q_row"]).contiguous()
    r2t0 = work["req_to_token"].clone() if cfg.page_size else None
    kv0 = work["kv_pool"].clone() if cfg.page_size else None

    def step():
        run_draft(buf, work["draft_table"], cfg.T, work["root_token"], work["seq_lens"], draft_u=work["draft_u"],
                  d2t=work.get("d2t"), t2d=work.get("t2d"))
        run_verify(buf, target, mode, cfg.T, work["coins"], work["u_final"], work.get("budget"),
                   int(work["eos_id"]))
        if cfg.page_size:
            run_compact(buf, work["seq_lens"], work["req_to_token"], cfg.page_size, kv_pool=work["kv_pool"])

    def outputs():
        o = {f"tree.{k}": v.clone() for k, v in buf.tree.items()}
        o.update({f"verify.{k}": v.clone() for k, v in buf.verify_out.items()})
        if cfg.page_size:
            o.update({f"compact.{k}": v.clone() for k, v in buf.compact_out.items()})
            o["req_to_token"] = work["req_to_token"].clone()
            o["kv_pool"] = work["kv_pool"].clone()
        return o

    def reset():
        for d in (buf.tree, buf.verify_out, buf.compact_out or {}):
            for v in d.values():
                v.fill_(-7)
        if cfg.page_size:  # compaction edits the slot table and pool in place
            work["req_to_token"].copy_(r2t0)
            work["kv_pool"].copy_(kv0)

    reset()
    step()
    torch.cuda.synchronize()
    eager = outputs()
    reset()
    graph = capture_step(step)
    reset()
    graph.replay()
    torch.cuda.synchronize()
    replayed = outputs()
    for k in eager:
        assert torch.equal(eager[k], replayed[k]), k


# ------------------------------------------------------ pruned draft LM head

def _head_inputs(rng, M, H, K, Vd, Vt):
    hidden = torch.from_numpy(rng.normal(0, 1, (M, H)).astype(np.float32)).to(torch.bfloat16)
    weight = torch.from_numpy(rng.normal(0, 3 / math.sqrt(H), (K, H)).astype(np.float32)).to(torch.bfloat16)
    ids = np.sort(rng.choice(Vd, K, replace=False)).astype(np.int32)
    d2t = np.full(Vd, -1, np.int32)
    d2t[ids] = rng.choice(Vt, K, replace=False)
    return hidden, weight, ids, d2t


def _head_compare(g, o, hidden, weight, rows, T):
    """GPU pruned-head outputs of `rows` against the oracle's.  Logits: within
    the fp32 accumulation bound H * 2^-24 * sum |hidden * weight| (any
    summation order); the top-1 may differ only where the oracle's two
    logits lie within that bound of each other (counted); the probability
    and normaliser within what that bound allows."""
    h64 = np.abs(hidden.float().numpy().astype(np.float64))[rows]
    w64 = np.abs(weight.float().numpy().astype(np.float64))
    H = hidden.shape[1]
    bound = H * 2.0 ** -24 * (h64 @ w64.T) + 1e-6
    if "logits" in g:
        gl = g["logits"].cpu().numpy().astype(np.float64)[rows]
        assert np.all(np.abs(gl - o["logits"]) <= bound), np.max(np.abs(gl - o["logits"]) / bound)
    near = 0
    gr = g["top1_rank"].cpu().numpy()[rows]
    for i in range(len(rows)):
        if gr[i] != o["top1_rank"][i]:
            a, b = gr[i], o["top1_rank"][i]
            assert abs(o["logits"][i, a] - o["logits"][i, b]) <= bound[i, a] + bound[i, b], (i, a, b)
            near += 1
            continue
        assert g["top1_draft"][rows[i]].item() == o["top1_draft"][i]
        assert g["top1_target"][rows[i]].item() == o["top1_target"][i]
        d = 2 * bound[i].max() / T
        np.testing.assert_allclose(g["top1_p"][rows[i]].item(), o["top1_p"][i], rtol=math.expm1(d) + 1e-6, atol=1e-7)
        st = g["row_stats"][rows[i]].cpu().numpy()
        assert abs(st[0] - o["row_max"][i]) <= bound[i].max()
        np.testing.assert_allclose(st[1], o["row_z"][i], rtol=math.expm1(d) + 1e-6)
    return near


@pytest.mark.parametrize("M,H,K", [(1, 64, 128), (256, 896, 5000), (100, 512, 3001), (300, 256, 1000),
                                   (7, 200, 129), (256, 96, 260)])
def test_pruned_head_parity(M, H, K):
    """The tcgen05 pruned LM head against the oracle's fp64 product: one and
    several N tiles (ragged last tile), one or two 128-row halves, a second
    group of hidden rows (M = 300), H not a multiple of the 64-column slab."""
    rng = np.random.default_rng(M * 7 + H + K)
    Vd, Vt = 2 * K + 17, K + 5
    hidden, weight, ids, d2t = _head_inputs(rng, M, H, K, Vd, Vt)
    T = 0.9
    stats = sd.new_stats()
    g = sd.tli_pruned_head(dev(hidden), dev(weight), dev(ids), dev(d2t), T, want_logits=True, stats=stats)
    torch.cuda.synchronize()
    o = oracle.pruned_head(np_logits(hidden), np_logits(weight), ids, d2t, T, want_logits=True)
    near = _head_compare(g, o, hidden, weight, np.arange(M), T)
    assert near <= max(1, M // 50)
    assert int(stats[sd.STATS["wait_timeout"]]) == 0


def test_pruned_head_full_size_sampled_rows():
    """The TLI workload's shapes: 256 draft rows, H = 896 (a 0.5B draft
    model's hidden size), K = 60000 intersection rows; the oracle recomputes
    sampled rows from both 128-row halves."""
    rng = np.random.default_rng(60000)
    M, H, K = 256, 896, 60000
    hidden, weight, ids, d2t = _head_inputs(rng, M, H, K, 151936, 128256)
    T = 1.0
    g = sd.tli_pruned_head(dev(hidden), dev(weight), dev(ids), dev(d2t), T, want_logits=True)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 127, 128, 200, 255])
    o = oracle.pruned_head(np_logits(hidden[rows]), np_logits(weight), ids, d2t, T, want_logits=True)
    assert _head_compare(g, o, hidden, weight, rows, T) <= 1


# ------------------------------------------------- target-side filtering

# top_k up to 512 takes the kernel's sorted-candidates path (unless ties
# overflow it), up to 4096 the radix top-k with sorted top-p, beyond that
# the radix top-k and top-p
FILTERS = [(1, 1.0), (5, 1.0), (0, 0.9), (20, 0.8), (0, 0.0), (3, 0.5), (0, 0.3), (600, 0.95), (5000, 0.9)]


@pytest.mark.parametrize("V,dtype", [(257, torch.float32), (4097, torch.bfloat16), (32000, torch.bfloat16),
                                     (1000, torch.float32)])
@pytest.mark.parametrize("top_k,top_p", FILTERS)
def test_filter_logits_kept_set(V, dtype, top_k, top_p):
    """The GPU filter keeps exactly the tokens the oracle's filter keeps
    (ties at the cut included: rows with long runs of equal logits), and
    leaves the kept logits untouched."""
    rng = np.random.default_rng(V + 31 * top_k + int(100 * top_p))
    R, T = 9, 0.8
    x = make_logits(rng, R, V, dtype, std=2.0)
    xf = x.float()
    xf[1, : V // 2] = xf[1].max()          # a long run tied at the top
    xf[2, 7:40] = xf[2, 7]                # ties inside the row
    xf[3, 100 % V] = float("nan")
    x = xf.to(dtype)
    g = sd.spec_filter_logits(dev(x.clone()), T, top_k, top_p)
    torch.cuda.synchronize()
    _, _, probs, _ = oracle.softmax_topk(np_logits(x), T, 1, want_probs=True)
    # the C ABI takes top_p in fp32: the oracle gets the same value (rows of
    # equal logits put the cut exactly at prefix / mass = top_p)
    kept = oracle.filter_probs(probs, top_k, float(np.float32(top_p))) > 0
    gk = torch.isfinite(g.float()).cpu().numpy() & ~np.isnan(g.float().cpu().numpy())
    np.testing.assert_array_equal(gk, kept)
    same = g.cpu()[torch.from_numpy(kept)]
    assert torch.equal(same, x[torch.from_numpy(kept)])


@pytest.mark.parametrize("top_k,top_p", [(3, 1.0), (0, 0.8), (8, 0.6)])
@pytest.mark.parametrize("chain", [False, True])
def test_filtered_verify_parity(top_k, top_p, chain):
    """Filtered logits through the stochastic verify (tree walk, or the chain
    launch) against the oracle's verify with the same top-k / top-p."""
    rng = np.random.default_rng(7 + top_k + int(10 * top_p) + (100 if chain else 0))
    B, V, T = 64, 2053, 0.9
    if chain:
        N = 5
        nt, ns = chain_meta(B, N)
        parent = np.array([-1] + list(range(N - 1)))
    else:
        N = 7  # root -> 1, 2; 1 -> 3, 4; 2 -> 5, 6
        nt = np.tile(np.array([1, 3, 5, -1, -1, -1, -1], np.int32), (B, 1))
        ns = np.tile(np.array([-1, 2, -1, 4, -1, 6, -1], np.int32), (B, 1))
        parent = np.array([-1, 0, 0, 1, 1, 2, 2])
    target = rng.normal(0, 2.0, (B, N, V)).astype(np.float32)
    q = _softmax64(target + rng.normal(0, 0.5, (B, N, V)).astype(np.float32), T).astype(np.float32)
    dt = np.zeros((B, N), np.int32)
    for b in range(B):
        for n in range(1, N):
            w = q[b, parent[n]].astype(np.float64)
            dt[b, n] = rng.choice(V, p=w / w.sum())
    coins = rng.random((B, N)).astype(np.float32)
    uf = rng.random(B).astype(np.float32)
    tf = sd.spec_filter_logits(dev(target), T, top_k, top_p)
    g = sd.spec_verify_sample(tf, T, dev(q), dev(dt), dev(nt), dev(ns), dev(coins), dev(uf), chain=chain)
    o = oracle.verify_sample(target, T, q, dt, nt, ns, coins, uf, top_k=top_k, top_p=float(np.float32(top_p)))
    torch.cuda.synchronize()
    exact = sum(verify_compare(g, o, b, b, "sample") for b in range(B))
    assert exact >= B - 1


@pytest.mark.parametrize("top_k,top_p", [(2, 1.0), (0, 0.7), (3, 0.8)])
def test_filtered_verify_law_monte_carlo_gpu(top_k, top_p):
    """With target-side filtering on the GPU (filter, then verify), the
    committed law of speculative rounds with i.i.d. drafts (tree of width 2,
    depth 2) is the law of sampling the filtered target alone."""
    from fractions import Fraction
    from oracle import exact
    from test_oracle_pins import chi2_pvalue, law_vector, markov_models, spec_rounds_with
    V, width, depth, M = 4, 2, 2, 2
    models, logP, Q = markov_models(V, seed=40 + top_k)
    tp = Fraction(top_p).limit_denominator(1000)
    P = [exact.filter_probs(models.p((v,)), top_k, tp) for v in range(V)]
    filtered = exact.ToyModels(V, lambda c: P[c[-1]], models.q)
    probs = law_vector(exact.target_law(filtered, (0,), M), V, M)

    def verify(target, qq, tok, nt, ns, coins, uf):
        t = sd.spec_filter_logits(dev(np.ascontiguousarray(target, np.float32)), 1.0, top_k, top_p)
        g = sd.spec_verify_sample(t, 1.0, dev(np.ascontiguousarray(qq, np.float32)), dev(tok), dev(nt), dev(ns),
                                  dev(coins), dev(uf))
        torch.cuda.synchronize()
        return {k: v.cpu().numpy() for k, v in g.items()}

    seqs = spec_rounds_with(verify, logP, Q, 0, M, width, depth, 100000, seed=5 + top_k)
    counts = np.bincount(np.ravel_multi_index(seqs.T, (V,) * M), minlength=V ** M)
    assert chi2_pvalue(counts, probs) > 1e-4
