"""The oracle's side of one whole speculative step, request by request.

TEST INFRASTRUCTURE ONLY (parity tests and the bench's CPU-baseline leg).
``fetch_request`` copies one request's inputs (a ``workloads`` dict of
tensors) to numpy; ``run_request`` then runs, on the CPU only, the draft
steps (softmax/top-k, draft sampling or the TLI constraint), tree expansion
and build, the target rows in node order, verification and (optionally) KV
compaction, through the oracle.  Nothing here reads a GPU result.
"""
from __future__ import annotations

import numpy as np
import torch

from . import build_tree, compact_slots, sample, softmax_topk, tli_constrain_map, tree_expand
from . import verify_greedy, verify_sample, Pool


# "[SGLang] Multi-Layer EAGLE" section 3: the draft loop's scores are the
# top-k of a plain softmax of the draft logits (no temperature).  The
# temperature of zero-to-sglang ch.10 5.1 applies to the stored draft
# distribution q that acceptance reads.
SCORE_T = 1.0


def np_logits(t: torch.Tensor) -> np.ndarray:
    """float32 array, or uint16 array of bf16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy().astype(np.float32, copy=False)


def step_offsets(B, topk, steps):
    return [0] + [B + (s - 1) * B * topk for s in range(1, steps)]


def table_rows_of(cfg, b):
    """Step-major draft-table rows of request b, per step."""
    offs = step_offsets(cfg.B, cfg.topk, cfg.steps)
    return [[b] if s == 0 else [offs[s] + b * cfg.topk + j for j in range(cfg.topk)] for s in range(cfg.steps)]


def full_row(cfg, b, qrow_single):
    """Draft-table row of request b for a row number of a one-request pool."""
    if qrow_single < 0:
        return -1
    if qrow_single == 0:
        return b
    offs = step_offsets(cfg.B, cfg.topk, cfg.steps)
    s = 1 + (qrow_single - 1) // cfg.topk
    return offs[s] + b * cfg.topk + (qrow_single - 1) % cfg.topk


def fetch_request(cfg, work, b):
    """One request's inputs as numpy arrays."""
    rows = table_rows_of(cfg, b)
    flat = [r for rs in rows for r in rs]
    dt = work["draft_table"]
    d = {"b": b, "rows": rows,
         "draft": dict(zip(flat, np_logits(dt[torch.tensor(flat, device=dt.device)])))}
    if "target" in work:
        d["target"] = np_logits(work["target"][b])
    else:
        te = work["target_exp"]
        d["target_exp"] = dict(zip(flat, np_logits(te[torch.tensor(flat, device=te.device)])))
        d["target_leaf"] = np_logits(work["target_leaf"][b])
    for name in ("root_token", "seq_lens", "coins", "u_final", "budget"):
        if name in work:
            d[name] = work[name][b:b + 1].cpu().numpy()
    d["draft_u"] = work["draft_u"].cpu().numpy()[flat]
    d["draft_u"] = dict(zip(flat, d["draft_u"]))
    d["eos"] = int(work["eos_id"])
    if cfg.kind == "tli":
        d["d2t"] = np_logits(work["d2t"]).astype(np.int32)
        d["t2d"] = np_logits(work["t2d"]).astype(np.int32)
    if "req_to_token" in work:
        d["req_to_token"] = work["req_to_token"][b:b + 1].cpu().numpy().copy()
    return d


def run_request(cfg, d, mode, compact=False, kv_pool=None):
    """Oracle step for one fetched request: returns (tree, q rows keyed by
    draft-table row, target [N, V], verify outputs, compaction outputs).
    The verify outputs carry "draft_margin": the smallest distance of a
    sampled draft's uniform to a CDF boundary of its draw (inf for drafts
    taken by top-k), so that a draft sampled differently can be told apart
    from an error.
    kv_pool (uint8 [slots, bytes], host): the whole slot payload pool, whose
    moved slots the compaction copies in place."""
    b, T, N = d["b"], cfg.T, cfg.N
    want_q = mode == "sample"
    sampled = cfg.kind == "chain" and mode == "sample"
    pool = Pool(1, cfg.topk, cfg.steps)
    q = {}
    draft_margin = np.inf  # the draft draws' closest approach to a CDF boundary
    for s, rows in enumerate(d["rows"]):
        x = np.stack([d["draft"][r] for r in rows])
        if cfg.kind == "tli":
            o = tli_constrain_map(x, d["d2t"], d["t2d"], T, want_q=want_q)
            tree_expand(pool, s, o["top1_p"].astype(np.float32), o["top1_target"])
            probs = o["q_target"]
        elif sampled:
            _, _, probs, _ = softmax_topk(x, T, 1, want_probs=True)
            u = np.array([d["draft_u"][r] for r in rows], np.float32)
            tok, prob, margin, _ = sample(u, logits=x, T=T)
            draft_margin = min(draft_margin, float(margin.min()))
            tree_expand(pool, s, prob.astype(np.float32), tok)
        else:
            tp, ti, probs, _ = softmax_topk(x, T, cfg.topk, want_probs=want_q, score_T=SCORE_T)
            tree_expand(pool, s, tp.astype(np.float32), ti)
        if want_q:
            for i, r in enumerate(rows):
                q[r] = probs[i]
    tree = build_tree(pool, N, d["root_token"], d["seq_lens"])
    tree["q_row"] = np.array([[full_row(cfg, b, int(r)) for r in tree["q_row"][0]]], np.int32)
    if "target" in d:
        target = d["target"]
    else:
        target = d["target_leaf"].copy()
        for n, r in enumerate(tree["q_row"][0]):
            if r >= 0:
                target[n] = d["target_exp"][int(r)]
    budget = d.get("budget")
    if mode == "greedy":
        v = verify_greedy(target[None], tree["draft_token"], tree["retrieve_next_token"],
                          tree["retrieve_next_sibling"], budget=budget, eos=d["eos"])
    else:
        qn = np.zeros((1, N, target.shape[-1]), np.float32)
        for n, r in enumerate(tree["q_row"][0]):
            if r >= 0 and int(r) in q:
                qn[0, n] = q[int(r)].astype(np.float32)
        v = verify_sample(target[None], T, qn, tree["draft_token"], tree["retrieve_next_token"],
                          tree["retrieve_next_sibling"], d["coins"], d["u_final"], budget=budget, eos=d["eos"])
    v["draft_margin"] = draft_margin
    c = None
    if compact and "req_to_token" in d:
        c = compact_slots(d["seq_lens"], v["accept_path"], v["accept_length"], d["req_to_token"], cfg.page_size,
                          kv_pool=kv_pool)
    return tree, q, target, v, c
