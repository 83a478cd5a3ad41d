"""Pins for the CPU oracle: worked examples printed on the pages, closed forms,
exact rational laws, invariants and brute-force checks.  No GPU."""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import exact


def bf16_bits(x):
    import torch
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------ softmax / top-k

def test_bf16_decoding_and_specials():
    row = np.array([[0x3F80, 0x4000, 0xFF80, 0x7FC0]], np.uint16)  # 1.0, 2.0, -inf, NaN
    p, idx, probs, flag = oracle.softmax_topk(row, 1.0, 2, want_probs=True)
    assert list(idx[0]) == [1, 0]
    e = math.exp(-1.0)
    np.testing.assert_allclose(probs[0], [e / (1 + e), 1 / (1 + e), 0.0, 0.0], rtol=0, atol=1e-15)
    assert flag[0] == 0


def test_softmax_closed_forms():
    ln3 = math.log(3.0)
    _, _, pr, _ = oracle.softmax_topk(np.array([[0.0, ln3]], np.float32), 1.0, 1, want_probs=True)
    np.testing.assert_allclose(pr[0], [0.25, 0.75], atol=1e-7)
    _, _, pr, _ = oracle.softmax_topk(np.array([[0.0, 2 * ln3]], np.float32), 2.0, 1, want_probs=True)
    np.testing.assert_allclose(pr[0], [0.25, 0.75], atol=1e-7)
    _, _, pr, _ = oracle.softmax_topk(np.full((1, 37), 1.5, np.float32), 0.7, 1, want_probs=True)
    np.testing.assert_allclose(pr[0], np.full(37, 1 / 37), atol=1e-15)
    rng = np.random.default_rng(1)
    x = rng.normal(0, 3, (5, 301)).astype(np.float32)
    tp, ti, pr, _ = oracle.softmax_topk(x, 0.7, 4, want_probs=True)
    np.testing.assert_allclose(pr.sum(1), 1.0, atol=1e-12)
    # ratio of two probabilities is exp(difference / T)
    np.testing.assert_allclose(pr[:, 3] / pr[:, 7], np.exp((x[:, 3].astype(np.float64) - x[:, 7]) / 0.7), rtol=1e-12)
    np.testing.assert_allclose(tp, np.take_along_axis(pr, ti.astype(np.int64), 1), rtol=0, atol=0)
    np.testing.assert_array_equal(ti[:, 0], np.argmax(x, 1))


def test_topk_ties_go_to_lowest_index():
    x = np.array([[5, 7, 7, 1, 7]], np.float32)
    _, idx, _, _ = oracle.softmax_topk(x, 1.0, 3)
    assert list(idx[0]) == [1, 2, 4]
    _, idx, _, _ = oracle.softmax_topk(x, 1.0, 5)
    assert list(idx[0]) == [1, 2, 4, 0, 3]


def test_nonfinite_row_is_flagged():
    x = np.full((2, 6), -np.inf, np.float32)
    x[1, 2] = np.inf
    p, idx, pr, flag = oracle.softmax_topk(x, 1.0, 2, want_probs=True)
    assert list(flag) == [1, 1]
    assert np.all(pr == 0) and np.all(p == 0)
    assert list(idx[0]) == [0, 1] and idx[1, 0] == 2


def test_inverse_cdf_sampling():
    probs = np.array([[0.25, 0.5, 0.25]] * 6, np.float32)
    u = np.array([0.3, 0.25, 0.0, 0.75, 0.9999, 0.7499], np.float32)
    tok, prob, margin, fb = oracle.sample(u, probs=probs)
    assert list(tok) == [1, 1, 0, 2, 2, 1]
    assert not fb.any()
    assert abs(margin[0] - 0.05) < 1e-7
    np.testing.assert_allclose(prob, [0.5, 0.5, 0.25, 0.25, 0.25, 0.5])
    # a zero-mass entry is never drawn, even at u = 0
    tok, _, _, _ = oracle.sample(np.array([0.0], np.float32), probs=np.array([[0.0, 1.0]], np.float32))
    assert tok[0] == 1
    # logits path: softmax(l/T) then the same rule
    l = np.log(np.array([[1.0, 2.0, 1.0]], np.float32)) * 2.0
    tok, prob, _, _ = oracle.sample(np.array([0.3], np.float32), logits=l.astype(np.float32), T=2.0)
    assert tok[0] == 1 and abs(prob[0] - 0.5) < 1e-7


# --------------------------------------------------------------- draft tree

def _run_tree(topk_per_step, k, S, N, seq_len=100, root=7):
    pool = oracle.Pool(1, k, S)
    for s, (tp, ti) in enumerate(topk_per_step):
        oracle.tree_expand(pool, s, np.array(tp, np.float32), np.array(ti, np.int32))
    return pool, oracle.build_tree(pool, N, np.array([root]), np.array([seq_len]))


def test_tree_hand_example():
    # k=2, 2 steps.  Step 0 root row: p=[0.6,0.3] tokens [10,20].
    # Step 1 rows (frontier slot 0 = pool 1, slot 1 = pool 2).
    steps = [([0.6, 0.3], [10, 20]),
             ([[0.5, 0.4], [0.9, 0.05]], [[11, 12], [21, 22]])]
    pool, t = _run_tree(steps, 2, 2, 5)
    # pool ids 3..6 = (slot 0: 11, 12), (slot 1: 21, 22); scores are fp32 products
    f32 = np.float32
    assert pool.score[0, 3] == f32(0.6) * f32(0.5) == f32(0.3)
    assert list(pool.parent[0, :7]) == [-1, 0, 0, 1, 1, 2, 2]
    # pool 2 (0.3) and pool 3 (0.6*0.5 == 0.3 in fp32) tie: lower pool id first;
    # then pool 5 (0.27) makes the 4th non-root node.
    assert list(t["draft_token"][0]) == [7, 10, 20, 11, 21]
    assert list(t["parent"][0]) == [-1, 0, 0, 1, 2]
    assert list(t["positions"][0]) == [100, 101, 101, 102, 102]
    assert list(t["retrieve_next_token"][0]) == [1, 3, 4, -1, -1]
    assert list(t["retrieve_next_sibling"][0]) == [-1, 2, -1, -1, -1]
    assert list(t["retrieve_index"][0]) == [0, 1, 2, 3, 4]
    # draft-row table rows: root = 0; frontier of step 0 expanded at step 1 -> rows B + slot
    assert list(t["q_row"][0]) == [0, 1, 2, -1, -1]
    m = t["tree_mask"][0]
    assert m.tolist() == [[1, 0, 0, 0, 0], [1, 1, 0, 0, 0], [1, 0, 1, 0, 0], [1, 1, 0, 1, 0], [1, 0, 1, 0, 1]]
    # N=4: the tie decides -> pool 3 is out, pool 2 in
    _, t4 = _run_tree(steps, 2, 2, 4)
    assert list(t4["draft_token"][0]) == [7, 10, 20, 11]


def test_tree_scores_use_a_plain_softmax():
    """[SGLang] Multi-Layer EAGLE, section 3: the draft loop scores the tree
    with the top-k of a plain softmax (no temperature); the temperature of
    zero-to-sglang ch.10 5.1 belongs to the stored q.  Hand-worked case (k=2,
    2 steps, N=3) where the two temperatures grow different trees.

    Root row logits [0, -0.5]; the row of the root's best child a: [0, -0.2].
      T=1:   p(a) = 1/(1+e^-0.5) = 0.6224593, p(b) = 0.3775407,
             p(a0 | a) = 1/(1+e^-0.2) = 0.5498340,
             score(a0) = 0.3422493 < score(b)  ->  nodes {a, b}.
      T=0.7: p(a) = 1/(1+e^(-0.5/0.7)) = 0.6713475, p(b) = 0.3286525,
             p(a0 | a) = 1/(1+e^(-0.2/0.7)) = 0.5709466,
             score(a0) = 0.3833035 > score(b)  ->  nodes {a, a0}."""
    root = np.array([[0.0, -0.5]], np.float32)
    step1 = np.array([[0.0, -0.2], [0.0, -0.2]], np.float32)  # frontier slots a, b
    expect = {1.0: ([0.6224593, 0.3775407], [0.5498340, 0.4501660], [7, 0, 1], [-1, 0, 0]),
              0.7: ([0.6713475, 0.3286525], [0.5709466, 0.4290534], [7, 0, 0], [-1, 0, 1])}
    for score_T, (p0, p1, tokens, parents) in expect.items():
        # q's temperature (T) is held at 0.7: only score_T moves the tree
        tp0, ti0, q0, _ = oracle.softmax_topk(root, 0.7, 2, want_probs=True, score_T=score_T)
        tp1, ti1, _, _ = oracle.softmax_topk(step1, 0.7, 2, score_T=score_T)
        np.testing.assert_allclose(tp0[0], p0, atol=1e-7)
        np.testing.assert_allclose(tp1[0], p1, atol=1e-7)
        np.testing.assert_allclose(q0[0], [0.6713475, 0.3286525], atol=1e-7)  # q at T=0.7 either way
        _, t = _run_tree([(tp0[0], ti0[0]), (tp1, ti1)], 2, 2, 3)
        assert list(t["draft_token"][0]) == tokens, score_T
        assert list(t["parent"][0]) == parents, score_T
    from oracle.pipeline import SCORE_T
    assert SCORE_T == 1.0


def _random_topk(rng, rows, k):
    p = np.sort(rng.uniform(0.01, 1.0, (rows, k)).astype(np.float32), axis=1)[:, ::-1]
    p = np.ascontiguousarray(p / np.float32(k))
    idx = np.stack([rng.choice(1000, k, replace=False) for _ in range(rows)]).astype(np.int32)
    return p, idx


def test_tree_invariants_and_brute_force_selection():
    rng = np.random.default_rng(7)
    B, k, S, N = 6, 3, 4, 12
    pool = oracle.Pool(B, k, S)
    for s in range(S):
        p, idx = _random_topk(rng, B * (1 if s == 0 else k), k)
        oracle.tree_expand(pool, s, p, idx)
    seq = rng.integers(16, 2048, B).astype(np.int32)
    t = oracle.build_tree(pool, N, np.arange(B, dtype=np.int32), seq)
    for b in range(B):
        # brute force: the N-1 best candidates by (score desc, pool id asc), ids sorted
        cand = sorted(range(1, pool.P), key=lambda i: (-float(pool.score[b, i]), i))[: N - 1]
        pids = [0] + sorted(cand)
        assert [int(pool.token[b, i]) if i else b for i in pids] == list(t["draft_token"][b])
        par = t["parent"][b]
        depth = [0] * N
        for n in range(1, N):
            assert 0 <= par[n] < n  # parents precede children (ancestor-closed)
            assert pids.index(int(pool.parent[b, pids[n]])) == par[n]
            depth[n] = depth[par[n]] + 1
        assert list(t["positions"][b]) == [int(seq[b]) + d for d in depth]
        for n in range(N):
            anc = set()
            a = n
            while a >= 0:
                anc.add(a)
                a = par[a] if a else -1
            assert [int(x) for x in t["tree_mask"][b, n]] == [1 if m in anc else 0 for m in range(N)]
            kids = [c for c in range(N) if c > 0 and par[c] == n]
            assert t["retrieve_next_token"][b, n] == (kids[0] if kids else -1)
            # walking next_token / next_sibling lists exactly the children in order
            walk, c = [], t["retrieve_next_token"][b, n]
            while c >= 0:
                walk.append(int(c))
                c = t["retrieve_next_sibling"][b, c]
            assert walk == kids
            assert t["retrieve_index"][b, n] == b * N + n


def test_topk_one_gives_chain():
    rng = np.random.default_rng(3)
    B, S = 4, 6
    pool = oracle.Pool(B, 1, S)
    for s in range(S):
        p, idx = _random_topk(rng, B, 1)
        oracle.tree_expand(pool, s, p, idx)
    t = oracle.build_tree(pool, S + 1, np.zeros(B, np.int32), np.zeros(B, np.int32))
    for b in range(B):
        assert list(t["parent"][b]) == [-1] + list(range(S))
        assert list(t["q_row"][b]) == [b] + [B + s * B + b for s in range(S - 1)] + [-1]


def test_draft_exercise_counts(golden):
    g = golden("draft_exercise.json")
    k, S = g["topk"], g["num_steps"]
    rng = np.random.default_rng(11)
    pool = oracle.Pool(1, k, S)
    frontier_ids = set()
    for s in range(S):
        p, idx = _random_topk(rng, 1 if s == 0 else k, k)
        oracle.tree_expand(pool, s, p, idx)
        frontier_ids.update(int(i) for i in pool.frontier_id[0])
    assert S == g["draft_forwards"]
    assert len(frontier_ids) == g["per_step_topk_candidates"]
    assert len(frontier_ids) + 1 == g["tree_tokens_with_root"]
    # a tree of exactly those candidates is ancestor-closed and builds
    t = oracle.build_tree(pool, g["tree_tokens_with_root"], np.array([0]), np.array([0]))
    assert (t["parent"][0, 1:] >= 0).all()


# ------------------------------------------------------------------ greedy

def chain_meta(N):
    nt = np.array([n + 1 if n + 1 < N else -1 for n in range(N)], np.int32)
    return nt, np.full(N, -1, np.int32)


def rows_with_choices(choices, V, rng=None):
    rng = rng or np.random.default_rng(0)
    x = rng.normal(0, 1, (len(choices), V)).astype(np.float32)
    for r, c in enumerate(choices):
        if c is None:
            c = V - 1
        x[r, c] = x[r].max() + 5.0
    return x


def test_greedy_worked_rejection(golden):
    g = golden("greedy_worked_rejection.json")
    N = len(g["proposals"]) + 1
    nt, ns = chain_meta(N)
    tgt = rows_with_choices(g["target_choice_per_row"], 8)[None]
    draft = np.array([[99] + g["proposals"]], np.int32)
    o = oracle.verify_greedy(tgt, draft, nt[None], ns[None])
    c = o["committed"][0, : o["num_committed"][0]]
    assert list(c) == g["committed"]
    assert o["accept_length"][0] == g["accept_length"]
    assert list(o["accept_path"][0, :2]) == [0, 1]
    assert list(o["walk_info"][0]) == [1, 1, 1]  # final node 1, one rejected child, correction


def test_row_alignment(golden):
    g = golden("row_alignment.json")
    L, k = g["prefix_len"], g["draft_len"]
    V = 16
    proposals = [3, 9, 4]
    bonus = 11
    # full-prefix target output over tokens + proposals: L + k rows
    choices = [0] * (L + k)
    for i, r in enumerate(g["verify_rows"]):
        choices[r] = proposals[i]
    choices[g["bonus_row"]] = bonus
    full = rows_with_choices(choices, V)
    nt, ns = chain_meta(k + 1)
    draft = np.array([[1] + proposals], np.int32)
    o = oracle.verify_greedy(full[L - 1:][None], draft, nt[None], ns[None])
    assert list(o["committed"][0]) == proposals + [bonus]
    assert o["accept_length"][0] == k and o["walk_info"][0, 2] == 2  # bonus
    # node row n is full-prefix row L-1+n; shifting the rows by one breaks it
    o2 = oracle.verify_greedy(full[L - 2: L + k - 1][None], draft, nt[None], ns[None])
    assert list(o2["committed"][0, : o2["num_committed"][0]]) != proposals + [bonus]


def test_eos_and_budget(golden):
    g = golden("eos_and_budget.json")
    eos = g["eos_id"]
    for case in g["cases"]:
        N = len(case["proposals"]) + 1
        nt, ns = chain_meta(N)
        tgt = rows_with_choices(case["target_choice_per_row"], 12)[None]
        draft = np.array([[1] + case["proposals"]], np.int32)
        o = oracle.verify_greedy(tgt, draft, nt[None], ns[None], budget=np.array([case["remaining"]]), eos=eos)
        got = list(o["committed"][0, : o["num_committed"][0]])
        assert got == case["committed"], case["name"]
        ends = (len(got) > 0 and got[-1] == eos) or len(got) == case["remaining"]
        assert ends == case["ends_request"], case["name"]
        assert o["next_root"][0] == (got[-1] if got else -1)


class ToyLM:
    """Context-dependent fp32 logits: a table indexed by the last two tokens,
    plus a draft model = target + noise."""

    def __init__(self, V, seed, noise):
        rng = np.random.default_rng(seed)
        self.V = V
        self.tab = rng.normal(0, 2, (V * V, V)).astype(np.float32)
        self.dtab = (self.tab + rng.normal(0, noise, self.tab.shape)).astype(np.float32)

    def target(self, ctx):
        return self.tab[ctx[-2] * self.V + ctx[-1]]

    def draft(self, ctx):
        return self.dtab[ctx[-2] * self.V + ctx[-1]]


def greedy_spec_decode_oracle(lm, ctx, M, k, S, N):
    """Greedy speculative decoding through the oracle's draft (softmax/top-k,
    tree expansion, tree build) and verify steps, round by round."""
    out = list(ctx)
    while len(out) - len(ctx) < M:
        pool = oracle.Pool(1, k, S)
        pool_ctx = {0: tuple(out)}
        rows = [lm.draft(pool_ctx[0])]
        for s in range(S):
            tp, ti, _, _ = oracle.softmax_topk(np.stack(rows), 1.0, k)
            oracle.tree_expand(pool, s, tp, ti)
            # contexts of this step's new candidates
            lo = 1 if s == 0 else 1 + k + (s - 1) * k * k
            hi = 1 + k if s == 0 else lo + k * k
            for pid in range(lo, hi):
                pool_ctx[pid] = pool_ctx[int(pool.parent[0, pid])] + (int(pool.token[0, pid]),)
            rows = [lm.draft(pool_ctx[int(f)]) for f in pool.frontier_id[0]]
        t = oracle.build_tree(pool, N, np.array([out[-1]]), np.array([len(out) - 1]))
        # node contexts: follow parents through draft tokens
        nctx = [tuple(out)]
        for n in range(1, N):
            nctx.append(nctx[t["parent"][0, n]] + (int(t["draft_token"][0, n]),))
        tgt = np.stack([lm.target(c) for c in nctx])[None]
        o = oracle.verify_greedy(tgt, t["draft_token"], t["retrieve_next_token"], t["retrieve_next_sibling"])
        out += list(o["committed"][0, : o["num_committed"][0]])
    return out[len(ctx): len(ctx) + M]


def argmax_decode(lm, ctx, M):
    out = list(ctx)
    for _ in range(M):
        out.append(int(np.argmax(lm.target(tuple(out)))))
    return out[len(ctx):]


@pytest.mark.parametrize("k,S,N", [(1, 4, 5), (3, 3, 8), (2, 4, 9)])
def test_greedy_spec_decoding_equals_target_argmax(k, S, N):
    lm = ToyLM(24, seed=5 + k, noise=0.8)
    ctx = (3, 17)
    assert greedy_spec_decode_oracle(lm, ctx, 60, k, S, N) == argmax_decode(lm, ctx, 60)


# -------------------------------------------------------------- stochastic

def test_worked_example_exact(golden):
    g = golden("stochastic_worked_example.json")
    p = tuple(Fraction(x) for x in g["p"])
    q = tuple(Fraction(x) for x in g["q"])
    assert [min(Fraction(1), p[y] / q[y]) for y in range(2)] == [Fraction(x) for x in g["accept_prob"]]
    assert exact.one_draft_law(p, q) == tuple(Fraction(x) for x in g["law"])
    assert exact.one_draft_law(p, q, on_reject="p") == tuple(Fraction(x) for x in g["law_if_resampled_from_p"])


def test_acceptance_and_rejection_masses_sum_to_one():
    rng = np.random.default_rng(2)
    for _ in range(20):
        V = int(rng.integers(2, 9))
        p = exact.normalise([Fraction(int(x)) for x in rng.integers(0, 7, V) + (np.arange(V) == 0)])
        q = exact.normalise([Fraction(int(x)) for x in rng.integers(1, 7, V)])
        acc, rej = exact.acceptance_masses(p, q)
        assert acc + rej == 1
        law = exact.one_draft_law(p, q)
        assert law == p


def worked_example_oracle(trials, seed):
    rng = np.random.default_rng(seed)
    tgt = np.log(np.array([0.4, 0.6], np.float32)).astype(np.float32)
    q = np.array([0.8, 0.2], np.float32)
    B, N, V = trials, 2, 2
    target = np.broadcast_to(tgt, (B, N, V)).copy()
    qq = np.broadcast_to(q, (B, N, V)).copy()
    y = (rng.random(B) >= 0.8).astype(np.int32)  # y ~ q
    draft = np.stack([np.zeros(B, np.int32), y], 1)
    nt = np.tile(np.array([1, -1], np.int32), (B, 1))
    ns = np.full((B, 2), -1, np.int32)
    coins = rng.random((B, N)).astype(np.float32)
    uf = rng.random(B).astype(np.float32)
    return oracle.verify_sample(target, 1.0, qq, draft, nt, ns, coins, uf)


def test_worked_example_monte_carlo_oracle(golden):
    g = golden("stochastic_worked_example.json")
    n = g["monte_carlo"]["trials"]
    o = worked_example_oracle(n, seed=2024)
    first = o["committed"][:, 0]
    f0 = float(np.mean(first == 0))
    sigma = math.sqrt(0.4 * 0.6 / n)
    assert abs(f0 - 0.4) < g["monte_carlo"]["sigma_bound"] * sigma
    # the test has the power to see the wrong rule (0.56)
    assert abs(0.56 - 0.4) > 100 * sigma


def markov_models(V, seed):
    rng = np.random.default_rng(seed)
    Pw = rng.integers(0, 6, (V, V)) + np.eye(V, dtype=int)  # some zeros in p
    Qw = rng.integers(1, 6, (V, V))
    P = [exact.normalise([Fraction(int(w)) for w in row]) for row in Pw]
    Q = [exact.normalise([Fraction(int(w)) for w in row]) for row in Qw]
    models = exact.ToyModels(V, lambda c: P[c[-1]], lambda c: Q[c[-1]])
    Pf = np.array([[float(x) for x in r] for r in P])
    Qf = np.array([[float(x) for x in r] for r in Q], np.float32)
    with np.errstate(divide="ignore"):
        logP = np.log(Pf).astype(np.float32)
    return models, logP, Qf


@pytest.mark.parametrize("width,depth,M", [(1, 2, 3), (1, 3, 2), (2, 2, 2), (3, 1, 2)])
def test_losslessness_exact(width, depth, M):
    models, _, _ = markov_models(3, seed=10 + width * 7 + depth)
    assert exact.spec_law(models, (0,), M, width, depth) == exact.target_law(models, (0,), M)


def tree_shape(width, depth):
    """Node order: BFS levels, children of a node consecutive (draw order)."""
    parent = [-1]
    level = [0]
    for _ in range(depth):
        nxt = []
        for p in level:
            for _ in range(width):
                parent.append(p)
                nxt.append(len(parent) - 1)
        level = nxt
    N = len(parent)
    nt = [-1] * N
    ns = [-1] * N
    for c in range(1, N):
        if nt[parent[c]] < 0:
            nt[parent[c]] = c
        for d in range(c + 1, N):
            if parent[d] == parent[c]:
                ns[c] = d
                break
    return np.array(parent), np.array(nt, np.int32), np.array(ns, np.int32)


def spec_rounds_with(verify, logP, Q, start, M, width, depth, trials, seed, draws="iid"):
    """Markov toy models: every trial runs rounds of (drafts from q, verify)
    until M tokens are committed; returns the first M tokens.  draws: "iid"
    or "without" (siblings drawn one after another without replacement)."""
    rng = np.random.default_rng(seed)
    V = logP.shape[0]
    parent, nt, ns = tree_shape(width, depth)
    N = len(parent)
    out = np.full((trials, M), -1, np.int64)
    have = np.zeros(trials, np.int64)
    last = np.full(trials, start, np.int64)
    while True:
        act = np.nonzero(have < M)[0]
        if act.size == 0:
            return out
        B = act.size
        tok = np.zeros((B, N), np.int64)
        tok[:, 0] = last[act]
        cdf = np.cumsum(Q.astype(np.float64), 1)
        for n in range(1, N):
            u = rng.random(B)
            if draws == "iid":
                tok[:, n] = np.minimum((u[:, None] >= cdf[tok[:, parent[n]]]).sum(1), V - 1)
            else:
                w = Q[tok[:, parent[n]]].astype(np.float64)
                for m_ in range(1, n):
                    if parent[m_] == parent[n]:
                        w[np.arange(B), tok[:, m_]] = 0.0
                c = np.cumsum(w / w.sum(1, keepdims=True), 1)
                tok[:, n] = np.minimum((u[:, None] >= c).sum(1), V - 1)
        target = logP[tok]
        qq = Q[tok]
        o = verify(target, qq, tok.astype(np.int32), np.tile(nt, (B, 1)), np.tile(ns, (B, 1)),
                   rng.random((B, N)).astype(np.float32), rng.random(B).astype(np.float32))
        nc = o["num_committed"]
        for j in range(N):
            sel = (j < nc) & (have[act] < M)
            rows = act[sel]
            out[rows, have[rows]] = o["committed"][sel, j]
            have[rows] += 1
        last[act] = o["committed"][np.arange(B), nc - 1]


def chi2_pvalue(counts, probs):
    from scipy.stats import chi2
    n = counts.sum()
    keep = probs > 0
    assert counts[~keep].sum() == 0
    e = n * probs[keep]
    stat = float(((counts[keep] - e) ** 2 / e).sum())
    return chi2.sf(stat, keep.sum() - 1)


def law_vector(law, V, M):
    v = np.zeros(V ** M)
    for seq, pr in law.items():
        v[np.ravel_multi_index(seq, (V,) * M)] = float(pr)
    return v


@pytest.mark.parametrize("V,width,depth,M", [(3, 2, 2, 2), (3, 3, 1, 2), (3, 2, 1, 3), (4, 3, 2, 2), (4, 2, 2, 2)])
def test_losslessness_exact_without_replacement(V, width, depth, M):
    """Children drawn without replacement, each rejection followed by
    q_cur <- q_cur without the rejected token, renormalised: the committed
    law is exactly the target's.  Keeping q fixed for such draws is not
    (the test can tell the two updates apart)."""
    models, _, _ = markov_models(V, seed=10 + width * 7 + depth)
    target = exact.target_law(models, (0,), M)
    assert exact.spec_law(models, (0,), M, width, depth, "without", "renormalise") == target
    if width < V:
        assert exact.spec_law(models, (0,), M, width, depth, "without", "fixed") != target


def test_filter_probs_hand_examples():
    """Target-side filtering, worked by hand on p = [0.1, 0.2, 0.5, 0.2]:
    order 2, 1, 3, 0 (the tie 0.2 / 0.2 goes to the lower index).  top-k 3:
    {2, 1, 3}, mass 0.9 -> [0, 2/9, 5/9, 2/9].  Then top-p 0.6 on that:
    prefixes 0, 5/9 < 0.6 keep 2 and 1, 7/9 drops 3 -> [0, 2/7, 5/7, 0].  top-p
    0.5 alone: the first token carries 0.5, so only it stays -> [0, 0, 1, 0]."""
    p = np.array([0.1, 0.2, 0.5, 0.2])
    np.testing.assert_allclose(oracle.filter_probs(p, 3), [0, 2 / 9, 5 / 9, 2 / 9], atol=1e-15)
    np.testing.assert_allclose(oracle.filter_probs(p, 3, 0.6), [0, 2 / 7, 5 / 7, 0], atol=1e-15)
    np.testing.assert_allclose(oracle.filter_probs(p, 0, 0.5), [0, 0, 1, 0], atol=1e-15)
    np.testing.assert_array_equal(oracle.filter_probs(p, 0, 1.0), p)
    np.testing.assert_array_equal(oracle.filter_probs(p, 4, 1.0), p)
    np.testing.assert_allclose(oracle.filter_probs(p, 1, 1.0), [0, 0, 1, 0], atol=1e-15)
    np.testing.assert_array_equal(oracle.filter_probs(np.zeros(4), 2, 0.5), np.zeros(4))
    zero = (Fraction(0),) * 4  # the exact-arithmetic statement leaves a massless row as it is too
    assert exact.filter_probs(zero, 2, Fraction(1, 2)) == zero


@pytest.mark.parametrize("seed", range(5))
def test_filter_probs_properties(seed):
    """Kept tokens precede dropped ones in (p desc, index asc); top-k keeps at
    most k; top-p keeps the shortest prefix whose mass reaches top_p of the
    top-k mass; the result sums to 1 and equals the exact-arithmetic rule."""
    rng = np.random.default_rng(seed)
    V = 50
    w = rng.integers(0, 20, V)
    w[rng.integers(0, V, 5)] = 7  # ties
    p = w / w.sum()
    for k, tp in ((0, 0.8), (10, 1.0), (10, 0.5), (3, 0.99), (0, 0.3)):
        f = oracle.filter_probs(p, k, tp)
        order = sorted(range(V), key=lambda v: (-p[v], v))
        kept = [v for v in order if f[v] > 0]
        assert kept == order[:len(kept)] or all(p[v] == 0 for v in order[len(kept):])
        if k:
            assert len(kept) <= k
        assert abs(f.sum() - 1.0) < 1e-12
        top = order[:k] if k else order
        mk = p[top].sum()
        if tp < 1.0:
            mass = p[kept].sum() / mk
            assert mass >= tp - 1e-12 or len(kept) == len([v for v in top if p[v] > 0])
            assert (p[kept].sum() - p[kept[-1]]) / mk < tp
        want = exact.filter_probs(tuple(Fraction(int(x), int(w.sum())) for x in w), k,
                                  Fraction(tp).limit_denominator(1000))
        np.testing.assert_allclose(f, [float(x) for x in want], atol=1e-12)


@pytest.mark.parametrize("top_k,top_p", [(2, 1.0), (0, 0.7), (3, 0.8)])
def test_filtered_verify_law_monte_carlo_oracle(top_k, top_p):
    """With target-side filtering, the committed law of speculative rounds
    (i.i.d. drafts from q, a tree of width 2 and depth 2) is the law of
    sampling the filtered target alone."""
    V, width, depth, M = 4, 2, 2, 2
    models, logP, Q = markov_models(V, seed=40 + top_k)
    tp = Fraction(top_p).limit_denominator(1000)
    P = [exact.filter_probs(models.p((v,)), top_k, tp) for v in range(V)]
    filtered = exact.ToyModels(V, lambda c: P[c[-1]], models.q)
    probs = law_vector(exact.target_law(filtered, (0,), M), V, M)

    def verify(target, qq, tok, nt, ns, coins, uf):
        return oracle.verify_sample(np.ascontiguousarray(target), 1.0, qq, tok, nt, ns, coins, uf, top_k=top_k,
                                    top_p=top_p)

    seqs = spec_rounds_with(verify, logP, Q, 0, M, width, depth, 100000, seed=5 + top_k)
    counts = np.bincount(np.ravel_multi_index(seqs.T, (V,) * M), minlength=V ** M)
    assert chi2_pvalue(counts, probs) > 1e-4


@pytest.mark.parametrize("seed", range(6))
def test_residual_closed_form(seed):
    """The kernel's form of the fixed-q sibling update, in exact arithmetic,
    against the definition (p_cur <- (p_cur - q)+ normalised after each
    rejection): with A_0 = 0, W_0 = 1, A_{j+1} = A_j + W_j and W_{j+1} =
    sum max(0, p - A_{j+1} q), p_cur after j rejections is
    max(0, p - A_j q) / W_j."""
    rng = np.random.default_rng(100 + seed)
    V = 9
    p = exact.normalise([Fraction(int(x)) for x in rng.integers(0, 9, V) + (np.arange(V) == 0)])
    q = exact.normalise([Fraction(int(x)) for x in rng.integers(1, 9, V)])
    pc, A, W = p, Fraction(0), Fraction(1)
    for _ in range(6):
        if sum(max(Fraction(0), a - b) for a, b in zip(pc, q)) == 0:
            break
        pc = exact.positive_residual(pc, q)
        A = A + W
        w = [max(Fraction(0), a - A * b) for a, b in zip(p, q)]
        W = sum(w)
        assert tuple(x / W for x in w) == pc


@pytest.mark.parametrize("seed", range(6))
def test_without_replacement_closed_form(seed):
    """The kernel's form of the without-replacement update, in exact
    arithmetic, against the definition: for rejections of distinct tokens
    y_0, y_1, ... the definition replaces p_cur by (p_cur - q_cur)+
    normalised, then removes y_j from q_cur and renormalises.  The closed
    form keeps A (A_0 = 0), the mass W (W_0 = 1), S = 1 - q(rejected), and
    for a rejected token its weight at rejection: after rejecting y_j,
    A <- A + W / S, the weights are max(0, p - A q) off the rejected set and
    the frozen ones on it, W is their sum.  Both must give the same p_cur and
    the same acceptance ratio p_cur[y] / q_cur[y] at every step."""
    rng = np.random.default_rng(seed)
    V = 7
    p = exact.normalise([Fraction(int(x)) for x in rng.integers(0, 9, V) + (np.arange(V) == 0)])
    q = exact.normalise([Fraction(int(x)) for x in rng.integers(1, 9, V)])
    order = [int(v) for v in rng.permutation(V)[:5]]
    pc, qc = p, q
    A, W, S, frozen = Fraction(0), Fraction(1), Fraction(1), {}
    for y in order:
        # acceptance ratio of y before its rejection, both ways
        r_closed = frozen[y] if y in frozen else max(Fraction(0), p[y] - A * q[y])
        p_closed = r_closed / W
        q_closed = Fraction(0) if y in frozen else q[y] / S
        assert p_closed == pc[y] and q_closed == qc[y]
        # reject y
        if sum(max(Fraction(0), a - b) for a, b in zip(pc, qc)) == 0:
            break
        pc = exact.positive_residual(pc, qc)
        qc = exact.without(qc, y)
        A = A + W / S
        frozen[y] = max(Fraction(0), p[y] - A * q[y])
        S = S - q[y]
        w = [frozen[v] if v in frozen else max(Fraction(0), p[v] - A * q[v]) for v in range(V)]
        W = sum(w)
        assert tuple(x / W for x in w) == pc
        if S == 0:
            break


def test_without_replacement_hand_example():
    """Two sibling leaves y0 = 1, y1 = 2 under a root with p = [0.3, 0.3, 0.4],
    q = [0.1, 0.6, 0.3], coins 0.7 and 0.6.  y0: ratio 0.3 / 0.6 = 0.5 <= 0.7,
    rejected; p_cur = (p - q)+ normalised = [2/3, 0, 1/3].  y1 with q fixed:
    ratio (1/3) / 0.3 = 1.11 > 0.6, accepted (then the bonus of leaf 2).
    Without replacement q_cur = [0.1, 0, 0.3] / 0.4 = [0.25, 0, 0.75]: ratio
    (1/3) / 0.75 = 0.44 <= 0.6, rejected; p_cur = (p_cur - q_cur)+ = [5/12, 0,
    0] normalised = [1, 0, 0], so the correction is token 0."""
    p = np.array([0.3, 0.3, 0.4])
    q = np.zeros((1, 3, 3), np.float32)
    q[0, 0] = [0.1, 0.6, 0.3]
    target = np.zeros((1, 3, 3), np.float32)
    target[0, 0] = np.log(p)
    target[0, 1:] = 0.0  # leaves: uniform bonus rows
    draft = np.array([[0, 1, 2]], np.int32)
    nt = np.array([[1, -1, -1]], np.int32)
    ns = np.array([[-1, 2, -1]], np.int32)
    coins = np.array([[0.0, 0.7, 0.6]], np.float32)
    uf = np.array([0.5], np.float32)
    with_r = oracle.verify_sample(target, 1.0, q, draft, nt, ns, coins, uf)
    wo_r = oracle.verify_sample(target, 1.0, q, draft, nt, ns, coins, uf, without_replacement=True)
    assert with_r["accept_length"][0] == 1 and with_r["committed"][0, 0] == 2
    assert with_r["num_committed"][0] == 2 and with_r["walk_info"][0, 2] == 2  # then the leaf's bonus
    assert wo_r["accept_length"][0] == 0 and wo_r["num_committed"][0] == 1 and wo_r["committed"][0, 0] == 0
    assert wo_r["walk_info"][0, 1] == 2  # both siblings rejected
    assert min(with_r["margin"][0], wo_r["margin"][0]) > 0.1


@pytest.mark.parametrize("width,depth,M", [(2, 2, 2), (3, 1, 2)])
def test_losslessness_monte_carlo_oracle_without_replacement(width, depth, M):
    """The C oracle's without-replacement update on children drawn without
    replacement reproduces the target's law of the first M tokens."""
    V = 3
    models, logP, Q = markov_models(V, seed=10 + width * 7 + depth)
    probs = law_vector(exact.target_law(models, (0,), M), V, M)

    def verify(target, qq, tok, nt, ns, coins, uf):
        return oracle.verify_sample(np.ascontiguousarray(target), 1.0, qq, tok, nt, ns, coins, uf,
                                    without_replacement=True)

    seqs = spec_rounds_with(verify, logP, Q, 0, M, width, depth, 100000, seed=77 + width, draws="without")
    counts = np.bincount(np.ravel_multi_index(seqs.T, (V,) * M), minlength=V ** M)
    assert chi2_pvalue(counts, probs) > 1e-4


@pytest.mark.parametrize("width,depth,M", [(1, 2, 3), (2, 2, 2), (3, 1, 2)])
def test_losslessness_monte_carlo_oracle(width, depth, M):
    V = 3
    models, logP, Q = markov_models(V, seed=10 + width * 7 + depth)
    probs = law_vector(exact.target_law(models, (0,), M), V, M)

    def verify(target, qq, tok, nt, ns, coins, uf):
        return oracle.verify_sample(np.ascontiguousarray(target), 1.0, qq, tok, nt, ns, coins, uf)

    seqs = spec_rounds_with(verify, logP, Q, 0, M, width, depth, 100000, seed=99 + width)
    counts = np.bincount(np.ravel_multi_index(seqs.T, (V,) * M), minlength=V ** M)
    assert chi2_pvalue(counts, probs) > 1e-4


def test_q_zero_reading():
    # child y with q[y] == 0: accepted iff p[y] > 0
    B, N, V = 2, 2, 3
    target = np.log(np.array([[[0.5, 0.5, 1e-30], [1, 1, 1]]] * B, np.float32))
    target[1, 0, 1] = -np.inf  # p[1] == 0 in request 1
    q = np.array([[[1.0, 0.0, 0.0], [1 / 3] * 3]] * B, np.float32)
    draft = np.array([[0, 1], [0, 1]], np.int32)
    nt = np.array([[1, -1]] * B, np.int32)
    ns = np.full((B, N), -1, np.int32)
    coins = np.full((B, N), 0.999, np.float32)
    o = oracle.verify_sample(target, 1.0, q, draft, nt, ns, coins, np.full(B, 0.5, np.float32))
    assert o["accept_length"][0] == 1 and o["committed"][0, 0] == 1
    assert o["accept_length"][1] == 0 and o["committed"][1, 0] != 1
    assert o["q_zero"] == 2


def test_residual_after_rejection_sums_to_law():
    # single draft, deterministic coin above the ratio -> rejection; the token
    # must then come from (p - q)+ normalised: here only token 1 has mass
    target = np.log(np.array([[[0.4, 0.6], [0.5, 0.5]]], np.float32))
    q = np.array([[[0.8, 0.2], [0.5, 0.5]]], np.float32)
    for u in (0.0, 0.3, 0.99):
        o = oracle.verify_sample(target, 1.0, q, np.array([[0, 0]], np.int32), np.array([[1, -1]], np.int32),
                                 np.array([[-1, -1]], np.int32), np.array([[0, 0.9]], np.float32),
                                 np.array([u], np.float32))
        assert o["accept_length"][0] == 0 and o["committed"][0, 0] == 1 and o["walk_info"][0, 2] == 1


# -------------------------------------------------------------- compaction

def test_compaction_page1_race_case():
    rt = np.zeros((1, 32), np.int32)
    rt[0, 10:14] = [100, 101, 102, 103]
    o = oracle.compact_slots(np.array([10]), np.array([[0, 2, 3, -1]]), np.array([2]), rt, 1)
    assert o["new_kv_len"][0] == 13
    assert list(rt[0, 10:13]) == [100, 102, 103]
    assert list(o["freed"]) == [101]
    assert o["num_moves"][0] == 0


def test_compaction_paged_race_case_moves_payload():
    ps, sl, N = 4, 6, 8
    rt = np.zeros((1, 32), np.int32)
    pages = [9, 3, 7, 5]  # logical page -> physical page
    for pos in range(16):
        rt[0, pos] = pages[pos // ps] * ps + pos % ps
    slots = 40
    kv = np.arange(slots * 8, dtype=np.int64).astype(np.uint8).reshape(slots, 8).copy()
    orig = kv.copy()
    path = np.array([[0, 2, 3, -1, -1, -1, -1, -1]], np.int32)
    o = oracle.compact_slots(np.array([sl]), path, np.array([2]), rt, ps, kv_pool=kv)
    assert o["new_kv_len"][0] == 9
    assert o["num_moves"][0] == 2
    assert list(o["move_src"][0, :2]) == [rt[0, 8], rt[0, 9]]
    assert list(o["move_dst"][0, :2]) == [rt[0, 7], rt[0, 8]]
    # logical position sl+i now holds node path[i]'s payload (race case: node 2
    # must be read before node 3 overwrites its slot)
    for i, n in enumerate([0, 2, 3]):
        assert (kv[rt[0, sl + i]] == orig[rt[0, sl + n]]).all()
    assert list(o["freed"]) == [pages[3]]  # page of positions 12..15; 8..11 keeps pos 8


@pytest.mark.parametrize("ps", [1, 4, 16])
def test_compaction_properties_random(ps):
    rng = np.random.default_rng(ps)
    B, N = 9, 13
    max_ctx = 208
    seq = rng.integers(0, 150, B).astype(np.int32)
    seq[0] = 0
    npages = max_ctx // ps * B
    perm = rng.permutation(npages)
    rt = np.zeros((B, max_ctx), np.int32)
    for b in range(B):
        for pos in range(max_ctx):
            rt[b, pos] = perm[b * (max_ctx // ps) + pos // ps] * ps + pos % ps
    # random accepted paths: strictly increasing node ids starting at 0
    acc = rng.integers(0, N, B).astype(np.int32)
    acc[1], acc[2] = 0, N - 1
    path = np.full((B, N), -1, np.int32)
    for b in range(B):
        path[b, : acc[b] + 1] = [0] + sorted(rng.choice(np.arange(1, N), acc[b], replace=False))
    path[2, :] = np.arange(N)  # full chain: no moves
    bps = 4
    kv = rng.integers(0, 256, (npages * ps, bps)).astype(np.uint8)
    orig_kv, orig_rt = kv.copy(), rt.copy()
    o = oracle.compact_slots(seq, path, acc, rt, ps, kv_pool=kv if ps > 1 else None)
    freed = list(o["freed"])
    for b in range(B):
        sl, a = int(seq[b]), int(acc[b])
        assert o["new_kv_len"][b] == sl + 1 + a
        for i in range(a + 1):
            src_slot = orig_rt[b, sl + path[b, i]]
            if ps == 1:
                assert rt[b, sl + i] == src_slot
            else:
                assert (kv[rt[b, sl + i]] == orig_kv[src_slot]).all()
    if ps == 1:
        kept = {int(orig_rt[b, seq[b] + path[b, i]]) for b in range(B) for i in range(acc[b] + 1)}
        tree = {int(orig_rt[b, seq[b] + n]) for b in range(B) for n in range(N)}
        assert set(freed) | kept == tree and not (set(freed) & kept) and len(freed) == len(set(freed))
    else:
        expect = []
        for b in range(B):
            sl, nk = int(seq[b]), int(seq[b]) + 1 + int(acc[b])
            for lp in range(-(-sl // ps), (sl + N - 1) // ps + 1):
                if lp * ps >= nk:
                    expect.append(int(orig_rt[b, lp * ps]) // ps)
        assert freed == expect
    assert o["num_moves"][2] == 0


# --------------------------------------------------------------------- TLI

def test_tli_hand_example():
    d2t = np.array([2, -1, 0, -1, 4, 1], np.int32)
    t2d = np.array([2, 5, 0, -1, 4], np.int32)
    x = np.array([[1, 9, 3, 8, 3, 0]], np.float32)
    o = oracle.tli_constrain_map(x, d2t, t2d, 1.0, want_q=True)
    Z = math.e ** 1 + 2 * math.e ** 3 + 1.0
    assert o["top1_draft"][0] == 2 and o["top1_target"][0] == 0
    assert abs(o["top1_p"][0] - math.e ** 3 / Z) < 1e-15
    np.testing.assert_allclose(o["q_target"][0], [math.e ** 3 / Z, 1 / Z, math.e / Z, 0.0, math.e ** 3 / Z],
                               atol=1e-15)
    # temperature 2 on the same row
    o = oracle.tli_constrain_map(x, d2t, t2d, 2.0)
    Z2 = math.e ** 0.5 + 2 * math.e ** 1.5 + 1.0
    assert abs(o["top1_p"][0] - math.e ** 1.5 / Z2) < 1e-15


def test_tli_random_maps_and_empty_intersection():
    rng = np.random.default_rng(4)
    Vd, Vt, K = 300, 200, 120
    dids = np.sort(rng.choice(Vd, K, replace=False))
    tids = rng.choice(Vt, K, replace=False)
    d2t = np.full(Vd, -1, np.int32)
    d2t[dids] = tids
    t2d = np.full(Vt, -1, np.int32)
    t2d[tids] = dids
    x = rng.normal(0, 3, (7, Vd)).astype(np.float32)
    x[3, dids] = -np.inf  # nothing finite in the intersection
    o = oracle.tli_constrain_map(x, d2t, t2d, 1.0, want_q=True)
    assert list(o["row_flag"]) == [0, 0, 0, 1, 0, 0, 0]
    assert o["top1_draft"][3] == -1 and o["top1_target"][3] == -1 and not o["q_target"][3].any()
    for r in (0, 1, 2, 4, 5, 6):
        d = o["top1_draft"][r]
        assert d2t[d] >= 0  # never leaves the intersection
        assert d == dids[np.argmax(x[r, dids])]
        assert o["top1_target"][r] == d2t[d]
        np.testing.assert_allclose(o["q_target"][r].sum(), 1.0, atol=1e-12)
        assert (o["q_target"][r][t2d < 0] == 0).all()
    # the two maps are inverse on the intersection; others fall back
    back = oracle.map_ids(oracle.map_ids(dids, d2t, -7), t2d, -7)
    assert (back == dids).all()
    miss = np.setdiff1d(np.arange(Vd), dids)[:5]
    assert (oracle.map_ids(miss, d2t, 42) == 42).all()
    assert (oracle.map_ids(np.array([-1, Vd, Vd + 5]), d2t, 42) == 42).all()


def test_tli_plan_against_sorted_intersection():
    """The plan's ranks are positions in the sorted intersection_draft_ids
    (searchsorted), its bitmap reproduces the mask id by id, K is the
    intersection size; partners outside the intersection or the vocabulary
    and the padding take their codes."""
    rng = np.random.default_rng(11)
    for Vd, Vt, K in ((300, 203, 120), (64, 6, 5), (1000, 999, 0), (77, 77, 77)):
        dids = np.sort(rng.choice(Vd, K, replace=False))
        tids = rng.choice(Vt, K, replace=False) if K <= Vt else None
        if tids is None:
            continue
        d2t = np.full(Vd, -1, np.int32)
        d2t[dids] = tids
        t2d = np.full(Vt, -1, np.int32)
        t2d[tids] = dids
        free = np.setdiff1d(np.arange(Vt), tids)
        outside = np.setdiff1d(np.arange(Vd), dids)
        planted = {}
        if len(free) >= 2 and len(outside) >= 1:
            t2d[free[0]] = outside[0]
            t2d[free[1]] = Vd + 4
            planted = {int(free[0]): -2 - int(outside[0]), int(free[1]): -1}
        o = oracle.tli_plan(d2t, t2d)
        assert int(o["K"][0]) == K
        words = len(o["bits"])
        assert words % 2 == 0 and words * 32 >= Vd > (words - 2) * 32
        for v in range(words * 32):
            bit = (int(o["bits"][v >> 5]) >> (v & 31)) & 1
            assert bit == (1 if v < Vd and d2t[v] >= 0 else 0)
        assert int(o["before"][0]) == 0
        for w in range(1, words):
            assert int(o["before"][w]) == int(o["before"][w - 1]) + bin(int(o["bits"][w - 1])).count("1")
        assert len(o["t2r"]) == (Vt + 3) // 4 * 4
        for t in range(len(o["t2r"])):
            if t >= Vt:
                expect = -1
            elif t in planted:
                expect = planted[t]
            elif t2d[t] < 0:
                expect = -1
            else:
                expect = int(np.searchsorted(dids, t2d[t]))
                assert dids[expect] == t2d[t]
            assert int(o["t2r"][t]) == expect


def test_tli_config_constraints(golden):
    g = golden("tli_constraints.json")
    for c in g["valid"]:
        assert oracle.tli_check_config(*c)
    for c in g["invalid"]:
        assert not oracle.tli_check_config(*c)


# ----------------------------------------------------- pruned draft LM head

def test_pruned_head_hand_example():
    """[TLI] Modifications (_try_prune_draft_lm_head): logits only for the
    intersection's weight rows.  Worked by hand: hidden [1, 0.5] against
    weight rows [1, 0], [0, 2], [1, 1] gives logits [1, 1, 1.5]; the top-1 is
    row 2 (draft id 9, target id 4) with p = 1 / (1 + 2 e^-0.5) = 0.4518628.
    hidden [2, 0] gives [2, 0, 2]: the tie goes to row 0 (the lower draft id)."""
    hidden = np.array([[1.0, 0.5], [2.0, 0.0]], np.float32)
    weight = np.array([[1.0, 0.0], [0.0, 2.0], [1.0, 1.0]], np.float32)
    ids = np.array([3, 7, 9], np.int32)
    d2t = np.full(12, -1, np.int32)
    d2t[[3, 7, 9]] = [11, 0, 4]
    o = oracle.pruned_head(hidden, weight, ids, d2t, 1.0, want_logits=True)
    np.testing.assert_array_equal(o["logits"], [[1.0, 1.0, 1.5], [2.0, 0.0, 2.0]])
    assert list(o["top1_rank"]) == [2, 0]
    assert list(o["top1_draft"]) == [9, 3] and list(o["top1_target"]) == [4, 11]
    assert abs(o["top1_p"][0] - 0.4518628) < 1e-7
    # row 2: p of each tied top = 1 / (2 + e^-2) = 1 / 2.1353353 = 0.4683105
    assert abs(o["top1_p"][1] - 0.4683105) < 1e-7
    assert list(o["row_flag"]) == [0, 0]


@pytest.mark.parametrize("seed", range(3))
def test_pruned_head_equals_constrain_on_the_full_row(seed):
    """With integer-valued inputs every product and sum is exact, so the
    pruned head must equal the TLI constraint applied to the full draft row
    (the K logits at their draft ids, -inf elsewhere) -- a transposed or
    misindexed weight operand, or a rank / id mix-up, fails here.  The logits
    also equal an fp64 matrix product computed independently."""
    rng = np.random.default_rng(seed)
    M, H, K, Vd, Vt = 7, 24, 50, 300, 80
    hidden = rng.integers(-3, 4, (M, H)).astype(np.float32)
    weight = rng.integers(-2, 3, (K, H)).astype(np.float32)
    ids = np.sort(rng.choice(Vd, K, replace=False)).astype(np.int32)
    d2t = np.full(Vd, -1, np.int32)
    d2t[ids] = rng.choice(Vt, K, replace=False)
    t2d = np.full(Vt, -1, np.int32)
    t2d[d2t[ids]] = ids
    T = 0.9
    o = oracle.pruned_head(bf16_bits(hidden), bf16_bits(weight), ids, d2t, T, want_logits=True)
    np.testing.assert_array_equal(o["logits"], hidden.astype(np.float64) @ weight.astype(np.float64).T)
    full = np.full((M, Vd), -np.inf, np.float32)
    full[:, ids] = o["logits"].astype(np.float32)
    c = oracle.tli_constrain_map(full, d2t, t2d, T)
    np.testing.assert_array_equal(o["top1_draft"], c["top1_draft"])
    np.testing.assert_array_equal(o["top1_target"], c["top1_target"])
    np.testing.assert_allclose(o["top1_p"], c["top1_p"], rtol=1e-12)
    np.testing.assert_array_equal(ids[o["top1_rank"]], o["top1_draft"])
    np.testing.assert_allclose(o["row_z"], np.exp((o["logits"] - o["row_max"][:, None]) / T).sum(1), rtol=1e-12)
