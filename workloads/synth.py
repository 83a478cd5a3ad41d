"""Workload shapes and seeded synthetic logits.

Five workloads (the shapes of the speculative-decoding benchmark set):

  c1  tiny chain:   B=4, 3 drafts (topk 1, N=4), V=32, fp32.  Target rows
                    N(0, 2^2) i.i.d.; draft = target + N(0, 1).  Drafts are
                    sampled from softmax(draft) with per-step uniforms; greedy
                    and stochastic verify at T=1.
  c2  EAGLE tree, greedy: B=64, topk 4, 5 steps, N=16, V=32000, bf16.
                    Target N(0, 3^2) plus +6 on one uniform random token per
                    row; draft = target + N(0, 1.5^2).
  c3  EAGLE tree, stochastic: B=128, topk 8, 6 steps, N=64, V=128256, bf16.
                    Target N(0, 3^2) - 1.1 ln(rank), the rank of each token
                    under a per-request random permutation of the vocabulary;
                    draft = target + N(0, 1).  T=0.7.  KV compaction with
                    page size 16 over a shuffled page pool, 4096-byte slots.
  c4  TLI chain:    B=256, topk 1, 4 steps (N=5), V_d=151936, V_t=128256,
                    bf16.  A random injective map of K=60000 ids (draft ids
                    drawn without replacement and sorted, paired with distinct
                    random target ids).  Draft N(0, 3^2); target t = draft of
                    its partner + N(0, 1) on the intersection, N(0, 3^2) +
                    N(0, 1) elsewhere.  T=1.
  c5  MTP chain:    B=1024, 15 drafts (N=16), V=129280, bf16.  Target
                    N(0, 3^2); draft = target + N(0, 0.8^2).  A stop id; each
                    (request, row) with probability 1/16 gets target[eos] =
                    row max + 4 (inherited by the draft through the noise).
                    Budget uniform in {1..20}.  Greedy and stochastic (T=0.8).

Layout.  Draft rows and the draft distributions computed from them live in a
step-major table: step 0 holds one row per request (the root), rows [0, B);
step s >= 1 holds topk rows per request, rows B + (s-1)*B*topk + b*topk +
slot.  For EAGLE trees every draft-table row also owns a target row (the
node the draft model expanded: its target row is the draft row's source);
nodes that are never expanded get fresh rows.  ``assemble_target`` lays the
target rows out in node order once a tree is known (node n uses its
draft-table row when it has one).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch


@dataclasses.dataclass
class Cfg:
    name: str
    kind: str  # "chain", "tree" or "tli"
    B: int
    topk: int
    steps: int
    N: int
    V: int
    dtype: torch.dtype
    T: float
    seed: int
    V_t: int = 0           # TLI target vocabulary
    K: int = 0             # TLI intersection size
    target_std: float = 3.0
    draft_noise: float = 1.0
    boost: float = 0.0     # c2: planted bonus on one token per target row
    zipf_s: float = 0.0    # c3: -s ln(rank) offsets
    eos_planted: bool = False
    budget_max: int = 0    # c5: budgets uniform in {1..budget_max}
    page_size: int = 0
    bytes_per_slot: int = 0
    modes: tuple = ("greedy",)

    @property
    def table_rows(self) -> int:
        return self.B + (self.steps - 1) * self.B * self.topk

    def scaled(self, **kw) -> "Cfg":
        return dataclasses.replace(self, **kw)


CONFIGS: Dict[str, Cfg] = {
    "c1": Cfg("c1", "chain", B=4, topk=1, steps=3, N=4, V=32, dtype=torch.float32, T=1.0, seed=1001,
              target_std=2.0, draft_noise=1.0, modes=("greedy", "sample")),
    "c2": Cfg("c2", "tree", B=64, topk=4, steps=5, N=16, V=32000, dtype=torch.bfloat16, T=1.0, seed=1002,
              target_std=3.0, draft_noise=1.5, boost=6.0, modes=("greedy",)),
    "c3": Cfg("c3", "tree", B=128, topk=8, steps=6, N=64, V=128256, dtype=torch.bfloat16, T=0.7, seed=1003,
              target_std=3.0, draft_noise=1.0, zipf_s=1.1, page_size=16, bytes_per_slot=4096,
              modes=("sample",)),
    "c4": Cfg("c4", "tli", B=256, topk=1, steps=4, N=5, V=151936, dtype=torch.bfloat16, T=1.0, seed=1004,
              V_t=128256, K=60000, target_std=3.0, draft_noise=1.0, modes=("sample",)),
    "c5": Cfg("c5", "chain", B=1024, topk=1, steps=15, N=16, V=129280, dtype=torch.bfloat16, T=0.8, seed=1005,
              target_std=3.0, draft_noise=0.8, eos_planted=True, budget_max=20, modes=("greedy", "sample")),
}


def step_offsets(cfg: Cfg):
    """First row of each draft step in the step-major table, plus the total."""
    offs = [0]
    for s in range(1, cfg.steps):
        offs.append(cfg.B + (s - 1) * cfg.B * cfg.topk)
    return offs, cfg.table_rows


def _gen(cfg: Cfg, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(cfg.seed * 1009 + stream)
    return g


# streams
_TARGET, _DRAFT_NOISE, _PERM, _COINS, _UFINAL, _DRAFT_U, _MISC, _MAP, _LEAF, _BOOST, _KV = range(11)


def _normal(shape, std, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std


def _chunks(n, size):
    for a in range(0, n, size):
        yield a, min(n, a + size)


def generate(cfg: Cfg, device="cpu", with_kv: bool = True) -> Dict[str, torch.Tensor]:
    """All inputs of one workload, on ``device``."""
    dev = torch.device(device)
    out: Dict[str, torch.Tensor] = {}
    B, V, N = cfg.B, cfg.V, cfg.N
    gm = _gen(cfg, _MISC, dev)
    out["root_token"] = torch.randint(0, V if cfg.kind != "tli" else cfg.V_t, (B,), generator=gm, device=dev,
                                      dtype=torch.int32)
    out["seq_lens"] = torch.randint(16, 2049, (B,), generator=gm, device=dev, dtype=torch.int32)
    out["coins"] = torch.rand((B, N), generator=_gen(cfg, _COINS, dev), device=dev, dtype=torch.float32)
    out["u_final"] = torch.rand((B,), generator=_gen(cfg, _UFINAL, dev), device=dev, dtype=torch.float32)
    out["draft_u"] = torch.rand((cfg.table_rows,), generator=_gen(cfg, _DRAFT_U, dev), device=dev,
                                dtype=torch.float32)
    if cfg.budget_max:
        out["budget"] = torch.randint(1, cfg.budget_max + 1, (B,), generator=gm, device=dev, dtype=torch.int32)
    out["eos_id"] = torch.tensor(-1, dtype=torch.int32)
    if cfg.kind == "tli":
        _gen_tli(cfg, dev, out)
    elif cfg.kind == "chain":
        _gen_chain(cfg, dev, out)
    else:
        _gen_tree(cfg, dev, out)
    if cfg.page_size and with_kv:
        _gen_kv(cfg, dev, out)
    return out


def _to(x, dtype):
    return x.to(dtype)


def _gen_chain(cfg: Cfg, dev, out):
    """Target rows per chain node [B, N, V]; draft rows for nodes 0..N-2 in
    the step-major table (row s*B + b is node s of request b)."""
    B, N, V = cfg.B, cfg.N, cfg.V
    gt, gd = _gen(cfg, _TARGET, dev), _gen(cfg, _DRAFT_NOISE, dev)
    target = torch.empty((B, N, V), dtype=cfg.dtype, device=dev)
    draft = torch.empty((cfg.table_rows, V), dtype=cfg.dtype, device=dev)
    eos = -1
    if cfg.eos_planted:
        eos = int(torch.randint(0, V, (1,), generator=_gen(cfg, _MISC + 100, dev), device=dev).item())
        plant = torch.rand((B, N), generator=_gen(cfg, _BOOST, dev), device=dev) < (1.0 / 16)
    for n in range(N):
        t = _normal((B, V), cfg.target_std, gt, dev)
        if cfg.eos_planted:
            rowmax = t.max(dim=1).values
            t[:, eos] = torch.where(plant[:, n], rowmax + 4.0, t[:, eos])
        target[:, n] = _to(t, cfg.dtype)
        d = t + _normal((B, V), cfg.draft_noise, gd, dev)
        if n < N - 1:
            draft[n * B:(n + 1) * B] = _to(d, cfg.dtype)
    out["target"] = target
    out["draft_table"] = draft
    out["eos_id"] = torch.tensor(eos, dtype=torch.int32)


def _gen_tree(cfg: Cfg, dev, out):
    """Draft-table rows (one per expanded node slot) with their own target
    rows, and fresh target rows for every (request, node) that is not
    expanded."""
    B, N, V = cfg.B, cfg.N, cfg.V
    rows = cfg.table_rows
    gt, gd, gl = _gen(cfg, _TARGET, dev), _gen(cfg, _DRAFT_NOISE, dev), _gen(cfg, _LEAF, dev)
    gb = _gen(cfg, _BOOST, dev)
    offset = None
    if cfg.zipf_s:
        gp = _gen(cfg, _PERM, dev)
        offset = torch.empty((B, V), dtype=torch.float32, device=dev)
        for b in range(B):
            rank = torch.randperm(V, generator=gp, device=dev).to(torch.float32) + 1.0
            offset[b] = -cfg.zipf_s * torch.log(rank)
    offs, _ = step_offsets(cfg)

    def request_of(r0, r1):
        # request index of step-major table rows [r0, r1)
        r = torch.arange(r0, r1, device=dev)
        req = torch.where(r < B, r, (r - B) % (B * cfg.topk) // cfg.topk)
        return req

    def shape_rows(t, req):
        if cfg.boost:
            j = torch.randint(0, V, (t.shape[0],), generator=gb, device=dev)
            t[torch.arange(t.shape[0], device=dev), j] += cfg.boost
        if offset is not None:
            t += offset[req]
        return t

    t_exp = torch.empty((rows, V), dtype=cfg.dtype, device=dev)
    draft = torch.empty((rows, V), dtype=cfg.dtype, device=dev)
    for a, b in _chunks(rows, 256):
        t = shape_rows(_normal((b - a, V), cfg.target_std, gt, dev), request_of(a, b))
        t_exp[a:b] = _to(t, cfg.dtype)
        draft[a:b] = _to(t + _normal((b - a, V), cfg.draft_noise, gd, dev), cfg.dtype)
    leaf = torch.empty((B, N, V), dtype=cfg.dtype, device=dev)
    for b in range(B):
        t = shape_rows(_normal((N, V), cfg.target_std, gl, dev), torch.full((N,), b, device=dev))
        leaf[b] = _to(t, cfg.dtype)
    out["target_exp"] = t_exp
    out["target_leaf"] = leaf
    out["draft_table"] = draft


def assemble_target(work: Dict[str, torch.Tensor], q_row: torch.Tensor) -> torch.Tensor:
    """Target logits [B, N, V] in node order: node n takes the target row of
    its draft-table row when it has one (q_row >= 0), else its fresh row."""
    if "target" in work:
        return work["target"]
    leaf = work["target_leaf"]
    t_exp = work["target_exp"]
    q_row = q_row.to(leaf.device).long()
    out = leaf.clone()
    has = q_row >= 0
    out[has] = t_exp[q_row[has]]
    return out


def _gen_tli(cfg: Cfg, dev, out):
    B, N, Vd, Vt, K = cfg.B, cfg.N, cfg.V, cfg.V_t, cfg.K
    gmap = _gen(cfg, _MAP, dev)
    draft_ids = torch.sort(torch.randperm(Vd, generator=gmap, device=dev)[:K]).values
    target_ids = torch.randperm(Vt, generator=gmap, device=dev)[:K]
    d2t = torch.full((Vd,), -1, dtype=torch.int32, device=dev)
    d2t[draft_ids] = target_ids.to(torch.int32)
    t2d = torch.full((Vt,), -1, dtype=torch.int32, device=dev)
    t2d[target_ids] = draft_ids.to(torch.int32)
    out["d2t"], out["t2d"] = d2t, t2d
    out["intersection_draft_ids"] = draft_ids.to(torch.int32)
    gt, gd, gl = _gen(cfg, _TARGET, dev), _gen(cfg, _DRAFT_NOISE, dev), _gen(cfg, _LEAF, dev)
    target = torch.empty((B, N, Vt), dtype=cfg.dtype, device=dev)
    draft = torch.empty((cfg.table_rows, Vd), dtype=cfg.dtype, device=dev)
    in_t = t2d >= 0
    src = t2d.clamp(min=0).long()
    for n in range(N):
        d = _normal((B, Vd), cfg.target_std, gd, dev).to(cfg.dtype).float()
        if n < N - 1:
            draft[n * B:(n + 1) * B] = d.to(cfg.dtype)
        t = torch.where(in_t[None, :], d[:, src], _normal((B, Vt), cfg.target_std, gl, dev))
        t = t + _normal((B, Vt), cfg.draft_noise, gt, dev)
        target[:, n] = t.to(cfg.dtype)
    out["target"] = target
    out["draft_table"] = draft
    # fallback id for unmapped accepted ids (a chosen eos of the draft vocab)
    out["fallback_id"] = torch.tensor(int(draft_ids[0].item()), dtype=torch.int32)


def _gen_kv(cfg: Cfg, dev, out):
    """Paged slot mapping: each request's logical pages come from a shuffled
    pool; slot = page * page_size + position % page_size."""
    B, ps = cfg.B, cfg.page_size
    max_ctx = ((2048 + cfg.N + ps) + ps - 1) // ps * ps
    pages_per_req = max_ctx // ps
    g = _gen(cfg, _KV, dev)
    perm = torch.randperm(B * pages_per_req, generator=g, device=dev).to(torch.int32)
    pos = torch.arange(max_ctx, device=dev, dtype=torch.int32)
    page = perm.view(B, pages_per_req)[:, (pos // ps).long()]
    out["req_to_token"] = (page * ps + pos % ps).contiguous()
    out["num_slots"] = torch.tensor(B * pages_per_req * ps)
    if cfg.bytes_per_slot:
        out["kv_pool"] = torch.randint(0, 256, (B * pages_per_req * ps, cfg.bytes_per_slot), generator=g,
                                       device=dev, dtype=torch.uint8)
