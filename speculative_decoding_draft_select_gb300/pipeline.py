"""One speculative-decoding step over a batch, composed from the C ABI.

Draft side (one launch per draft step: the draft kernel also expands the
candidate pool for its step, the spec_tree_expand step fused), as in
"[SGLang] Multi-Layer EAGLE" sections 2-3 and "EAGLE speculative decoding
in four parts", "Drafting, verification and slots":
  - EAGLE tree:  spec_softmax_topk on the step's draft rows (writing the
                 draft distribution q into the step-major table when the
                 verify samples);
  - sampled chain: spec_softmax_sample (q or its row statistics, and the
                 draw with the step's uniforms, in one pass), k = 1;
  - TLI chain:   tli_plan_build once per vocabulary-map pair (the maps'
                 plan, rebuilt when the maps change), then per draft step
                 tli_constrain_map with it (q in
                 target order, the mapped top-1 expanded) (SGLang PR #22883);
                 with q_mode "logits", tli_constrain_map_qlogits (the
                 partners' logits in target order and each row's (max,
                 normaliser): half the bytes of fp32 q for bf16 logits).
then spec_build_tree.  Verify: spec_verify_greedy, or for sampling either
spec_verify_sample on the written q table (q_mode "probs") or
spec_verify_sample_qlogits on the draft logits plus the per-row (max,
normaliser) the draft kernel records (q_mode "logits": no q is written; the
q values are bit-identical).  Compaction: spec_compact_slots.

All buffers are allocated once in ``StepBuffers``; a step only enqueues
kernels on the current stream, so a whole step can be captured once in a
CUDA graph (``capture_step``) and replayed: the same kernels, without the
per-launch host cost and the gaps between launches.
"""
from __future__ import annotations

import torch

from . import (new_pool, new_stats, spec_build_tree, spec_compact_freed_capacity, spec_compact_slots,
               spec_softmax_sample, spec_softmax_topk, spec_verify_greedy, spec_verify_sample,
               spec_verify_sample_qlogits, spec_verify_ws_size, tli_constrain_map, tli_constrain_map_qlogits,
               tli_plan_build, tli_plan_bytes)


# The draft loop's tree scores are the top-k of a plain softmax ("[SGLang]
# Multi-Layer EAGLE", section 3); the temperature (zero-to-sglang ch.10 5.1)
# belongs to the stored q.
SCORE_T = 1.0


def step_offsets(B, topk, steps):
    offs = [0] + [B + (s - 1) * B * topk for s in range(1, steps)]
    return offs, B + (steps - 1) * B * topk


class StepBuffers:
    """Preallocated device buffers of one step.

    kind: "tree" (EAGLE top-k tree), "chain" (topk 1; drafts by argmax, or
    sampled when ``sampled``), "tli" (chain with the TLI constraint).
    """

    def __init__(self, kind, B, topk, steps, N, V, device, want_q, sampled=False, V_t=None, page_size=0,
                 max_ctx=0, q_mode="probs", q_logit_dtype=torch.bfloat16):
        if q_mode not in ("probs", "logits"):
            raise ValueError("q_mode must be 'probs' or 'logits'")
        self.kind, self.B, self.topk, self.steps, self.N, self.V = kind, B, topk, steps, N, V
        self.sampled, self.want_q, self.q_mode = sampled, want_q, q_mode
        self.Vq = V_t if kind == "tli" else V
        self.offs, self.rows = step_offsets(B, topk, steps)
        dev = torch.device(device)
        self.device = dev
        self.pool = new_pool(B, topk, steps, dev)
        kk = topk
        self.topk_p = [torch.empty((B * (1 if s == 0 else kk), kk), dtype=torch.float32, device=dev)
                       for s in range(steps)]
        self.topk_idx = [torch.empty((B * (1 if s == 0 else kk), kk), dtype=torch.int32, device=dev)
                         for s in range(steps)]
        # q for the verify: fp32 probabilities ("probs"); in logit form the
        # draft table itself, or for TLI the draft logits mapped into target
        # order (q_logit_dtype, the draft table's dtype)
        self.q = None
        if want_q and q_mode == "probs":
            self.q = torch.empty((self.rows, self.Vq), dtype=torch.float32, device=dev)
        elif want_q and kind == "tli":
            self.q = torch.empty((self.rows, self.Vq), dtype=q_logit_dtype, device=dev)
        self.q_stats = (torch.empty((self.rows, 2), dtype=torch.float32, device=dev)
                        if want_q and q_mode == "logits" else None)
        self.draft_table = None
        self.T_draft = None
        self.tok = torch.empty((self.rows,), dtype=torch.int32, device=dev)
        self.prob = torch.empty((self.rows,), dtype=torch.float32, device=dev)
        self.top1_draft = torch.empty((self.rows,), dtype=torch.int32, device=dev)
        self.tli_plan = (torch.empty(tli_plan_bytes(V, V_t), dtype=torch.uint8, device=dev)
                         if kind == "tli" else None)
        self.tli_plan_key = None  # the maps the plan was built from
        self.tree = None
        self.ws = torch.empty(max(spec_verify_ws_size(B, N), 256), dtype=torch.uint8, device=dev)
        self.verify_out = None
        self.stats = new_stats(dev)
        self.compact_out = None
        if page_size:
            cap = spec_compact_freed_capacity(B, N, page_size)
            self.compact_out = {
                "move_src": torch.empty((B, N), dtype=torch.int32, device=dev),
                "move_dst": torch.empty((B, N), dtype=torch.int32, device=dev),
                "num_moves": torch.empty((B,), dtype=torch.int32, device=dev),
                "freed": torch.empty((max(cap, 1),), dtype=torch.int32, device=dev),
                "num_freed": torch.empty((1,), dtype=torch.int32, device=dev),
                "new_kv_len": torch.empty((B,), dtype=torch.int32, device=dev),
            }
        self._alloc_tree()

    def _alloc_tree(self):
        B, N, dev = self.B, self.N, self.device
        self.tree = {name: torch.empty((B, N), dtype=torch.int32, device=dev)
                     for name in ("draft_token", "parent", "positions", "retrieve_index", "retrieve_next_token",
                                  "retrieve_next_sibling", "q_row")}
        self.tree["tree_mask"] = torch.empty((B, N, N), dtype=torch.uint8, device=dev)
        self.verify_out = {
            "committed": torch.empty((B, N), dtype=torch.int32, device=dev),
            "num_committed": torch.empty((B,), dtype=torch.int32, device=dev),
            "accept_length": torch.empty((B,), dtype=torch.int32, device=dev),
            "accept_path": torch.empty((B, N), dtype=torch.int32, device=dev),
            "next_root": torch.empty((B,), dtype=torch.int32, device=dev),
            "walk_info": torch.empty((B, 3), dtype=torch.int32, device=dev),
        }


def run_draft(buf: StepBuffers, draft_table, T, root_token, seq_lens, draft_u=None, d2t=None, t2d=None, timer=None):
    """Draft steps + tree build.  Returns buf.tree.  ``timer`` (optional) has
    begin(step) / end(step), called around each step's softmax/top-k or TLI
    launch."""
    B, k = buf.B, buf.topk
    buf.draft_table, buf.T_draft = draft_table, T
    if buf.kind == "tli":
        # the plan depends on the vocabulary maps alone (fixed for a model
        # pair): built on first use and again whenever the maps are other
        # tensors or were modified in place
        key = (d2t.data_ptr(), d2t._version, d2t.numel(), t2d.data_ptr(), t2d._version, t2d.numel())
        if buf.tli_plan_key != key:
            tli_plan_build(d2t, t2d, plan=buf.tli_plan)
            buf.tli_plan_key = key
    for s in range(buf.steps):
        r = B * (1 if s == 0 else k)
        a = buf.offs[s]
        rows = draft_table[a:a + r]
        qs = buf.q[a:a + r] if buf.q is not None else None
        st = buf.q_stats[a:a + r] if buf.q_stats is not None else None
        if timer is not None:
            timer.begin(s)
        # each draft launch also expands the candidate pool for its step
        if buf.kind == "tli" and st is not None:
            # q in logit form: the partners' logits in target order and (m, Z)
            tli_constrain_map_qlogits(rows, d2t, t2d, T, plan=buf.tli_plan, top1_draft=buf.top1_draft[a:a + r],
                                      top1_target=buf.tok[a:a + r], top1_p=buf.prob[a:a + r], q_logits=qs,
                                      q_stats=st, stats=buf.stats, expand=(buf.pool, s))
        elif buf.kind == "tli":
            tli_constrain_map(rows, d2t, T, t2d=t2d, top1_draft=buf.top1_draft[a:a + r],
                              top1_target=buf.tok[a:a + r], top1_p=buf.prob[a:a + r], q_target=qs,
                              stats=buf.stats, plan=buf.tli_plan, expand=(buf.pool, s))
        elif buf.kind == "chain" and buf.sampled:
            # softmax (q or its row statistics) and the draw in one pass
            spec_softmax_sample(rows, T, draft_u[a:a + r], out_token=buf.tok[a:a + r], out_prob=buf.prob[a:a + r],
                                row_stats=st, probs=qs, stats=buf.stats, expand=(buf.pool, s))
        else:
            spec_softmax_topk(rows, T, k, topk_p=buf.topk_p[s], topk_idx=buf.topk_idx[s], probs=qs, row_stats=st,
                              stats=buf.stats, expand=(buf.pool, s), score_T=SCORE_T)
        if timer is not None:
            timer.end(s)
    spec_build_tree(buf.pool, buf.N, root_token, seq_lens, out=buf.tree)
    return buf.tree


def run_verify(buf: StepBuffers, target, mode, T=1.0, coins=None, u_final=None, budget=None, eos_id=-1,
               without_replacement=False, chain=None):
    """Greedy or stochastic verify of buf.tree against target [B, N, V];
    without_replacement selects the stochastic sibling update for children
    drawn without replacement (q renormalised without each rejected child).
    chain selects the chain verify launch (SPEC_VERIFY_CHAIN) for the
    stochastic verify of chains; the default is the tree walk, which measured
    faster on chains too (B=256 x 5 nodes: 117 vs 128 us; B=1024 x 16: 725 vs
    798 us)."""
    t = buf.tree
    chain = False if chain is None else chain
    if mode == "greedy":
        return spec_verify_greedy(target, t["draft_token"], t["retrieve_next_token"], t["retrieve_next_sibling"],
                                  budget=budget, eos_id=eos_id, out=buf.verify_out, ws=buf.ws, stats=buf.stats)
    if buf.q_mode == "logits":
        q_logits = buf.q if buf.kind == "tli" else buf.draft_table
        return spec_verify_sample_qlogits(target, T, q_logits, buf.q_stats, buf.T_draft, t["draft_token"],
                                          t["retrieve_next_token"], t["retrieve_next_sibling"], coins, u_final,
                                          q_row=t["q_row"], budget=budget, eos_id=eos_id, out=buf.verify_out,
                                          ws=buf.ws, stats=buf.stats, without_replacement=without_replacement,
                                          chain=chain)
    return spec_verify_sample(target, T, buf.q, t["draft_token"], t["retrieve_next_token"],
                              t["retrieve_next_sibling"], coins, u_final, q_row=t["q_row"], budget=budget,
                              eos_id=eos_id, out=buf.verify_out, ws=buf.ws, stats=buf.stats,
                              without_replacement=without_replacement, chain=chain)


def run_compact(buf: StepBuffers, seq_lens, req_to_token, page_size, kv_pool=None):
    v = buf.verify_out
    return spec_compact_slots(seq_lens, v["accept_path"], v["accept_length"], req_to_token, page_size,
                              kv_pool=kv_pool, out=buf.compact_out, stats=buf.stats)


def capture_step(fn, warm=True):
    """Capture the launches ``fn()`` enqueues (one step on preallocated
    buffers) in a CUDA graph; ``graph.replay()`` re-runs them on the same
    buffers.  With ``warm``, ``fn`` first runs once eagerly on a side stream
    so that every kernel's attributes are set before the capture (a caller
    that has already run the step may skip it)."""
    if warm:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn()
        torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    return graph


def kernels_per_step(buf: StepBuffers, mode, compact: bool, kv_pool: bool) -> int:
    """Number of kernel launches one step enqueues."""
    per_step = 1  # softmax/top-k (or softmax and draw, or TLI constrain) with the pool expansion
    n = buf.steps * per_step + 1  # + build_tree
    # (TLI: the map plan's three launches run only when the maps change)
    n += 2 if mode == "greedy" else 1  # verify: row argmax + walk, or the one stochastic launch
    if compact:
        n += 1 + (1 if (kv_pool and buf.compact_out is not None) else 0)
    return n
