"""Exact (rational-arithmetic) laws of speculative sampling on tiny vocabularies.

TEST INFRASTRUCTURE ONLY (same rule as the rest of ``oracle/``).

This module states the stochastic acceptance rule of zero-to-sglang ch.10
"Speculative decoding (code walk-through)", section 5.1 -- a draft y drawn
from q is accepted with probability min(1, p[y]/q[y]); on rejection the token
is drawn from the normalised positive residual (p - q)+; after full acceptance
the bonus is drawn from p -- with ``fractions.Fraction`` so that laws come out
exactly.  It is used to pin the C oracle: the pages' worked example (p = [0.4,
0.6], q = [0.8, 0.2] gives exactly 0.4 / 0.6, and resampling from p instead
gives 0.56 / 0.44), and the losslessness claim of the same section (the law of
the committed tokens equals the target's own autoregressive law) for chains
and for trees whose children are i.i.d. draws from q, tried sibling by sibling
against the updated residual -- and, for children drawn without replacement,
with q renormalised after each rejected sibling (the "without replacement"
variant of the sibling update).
"""
from __future__ import annotations

from fractions import Fraction
from typing import Callable, Dict, Sequence, Tuple

Dist = Tuple[Fraction, ...]
Law = Dict[Tuple[int, ...], Fraction]


def normalise(w: Sequence[Fraction]) -> Dist:
    s = sum(w)
    return tuple(x / s for x in w)


def positive_residual(p: Dist, q: Dist) -> Dist:
    """(p - q)+ normalised (section 5.1).  Only called after a rejection,
    where the residual has positive mass."""
    r = [max(Fraction(0), a - b) for a, b in zip(p, q)]
    return normalise(r)


def one_draft_law(p: Dist, q: Dist, on_reject: str = "residual") -> Dist:
    """Law of the token output by one draft y ~ q verified against p.
    on_reject='residual' is the rule of section 5.1; 'p' resamples from p,
    the mistake the same section warns about."""
    out = [Fraction(0)] * len(p)
    reject_mass = Fraction(0)
    for y, qy in enumerate(q):
        if qy == 0:
            continue
        a = min(Fraction(1), p[y] / qy)
        out[y] += qy * a
        reject_mass += qy * (1 - a)
    if reject_mass > 0:
        r = positive_residual(p, q) if on_reject == "residual" else p
        for v in range(len(p)):
            out[v] += reject_mass * r[v]
    return tuple(out)


def acceptance_masses(p: Dist, q: Dist) -> Tuple[Fraction, Fraction]:
    """(sum_v min(p, q), sum_v (p - q)+): the mass the acceptance branch
    contributes and the mass the rejection branch must supply."""
    acc = sum(min(a, b) for a, b in zip(p, q))
    rej = sum(max(Fraction(0), a - b) for a, b in zip(p, q))
    return acc, rej


def filter_probs(p: Dist, top_k: int = 0, top_p: Fraction = Fraction(1)) -> Dist:
    """Target-side top-k / top-p filtering in exact arithmetic (the rule of
    the C oracle's oracle_filter_probs): order by (p desc, index asc), keep
    the first top_k (0: all), then every kept token whose exclusive prefix of
    the renormalised top-k mass is below top_p (the first always), and
    renormalise.  A row with no mass is returned unchanged, as the C oracle
    leaves it."""
    if sum(p) == 0:
        return tuple(p)
    order = sorted(range(len(p)), key=lambda v: (-p[v], v))
    keep = order[:top_k] if 0 < top_k < len(p) else order
    mk = sum(p[v] for v in keep)
    if top_p < 1 and mk > 0:
        kept, prefix = [], Fraction(0)
        for i, v in enumerate(keep):
            if i > 0 and not prefix / mk < top_p:
                break
            kept.append(v)
            prefix += p[v]
        keep = kept
    m = sum(p[v] for v in keep)
    return tuple((p[v] / m if v in keep else Fraction(0)) for v in range(len(p)))


class ToyModels:
    """A target p(.|context) and a draft q(.|context) over a tiny vocabulary,
    given as exact distributions by two callables on token tuples."""

    def __init__(self, V: int, target: Callable[[Tuple[int, ...]], Dist],
                 draft: Callable[[Tuple[int, ...]], Dist]):
        self.V, self.p, self.q = V, target, draft


def _add(law: Law, seq: Tuple[int, ...], pr: Fraction) -> None:
    if pr:
        law[seq] = law.get(seq, Fraction(0)) + pr


def without(q: Dist, y: int) -> Dist:
    """q with token y removed and the rest renormalised (all zero when
    nothing is left)."""
    w = [Fraction(0) if v == y else x for v, x in enumerate(q)]
    return normalise(w) if sum(w) > 0 else tuple(Fraction(0) for _ in w)


def round_law(m: ToyModels, ctx: Tuple[int, ...], width: int, depth: int, draws: str = "iid",
              q_update: str = "fixed") -> Law:
    """Law of the tokens committed in one verification round when every tree
    node has ``width`` children drawn from q(.|node context) down to
    ``depth`` levels (width 1 = a chain of ``depth`` drafts).  Children are
    tried in sibling order against p_cur, which each rejection replaces with
    the positive residual (p_cur - q_cur)+; with no child accepted the token
    is drawn from p_cur; at a leaf the bonus is drawn from p.

    draws: "iid" -- the children are i.i.d. draws from q; "without" -- drawn
    one after another without replacement (each from q with the earlier
    siblings' tokens removed and renormalised).  q_update: "fixed" -- q_cur
    stays q for every sibling; "renormalise" -- after a rejection of y,
    q_cur loses y and is renormalised (the without-replacement update)."""

    def node(c: Tuple[int, ...], d: int) -> Law:
        q = m.q(c)
        return siblings(c, m.p(c), q, q, width if d > 0 else 0, d)

    def siblings(c: Tuple[int, ...], pc: Dist, qc: Dist, qdraw: Dist, left: int, d: int) -> Law:
        law: Law = {}
        if left == 0 or sum(qdraw) == 0:
            for t, pt in enumerate(pc):
                _add(law, (t,), pt)
            return law
        for y, qy in enumerate(qdraw):
            if qy == 0:
                continue
            a = min(Fraction(1), pc[y] / qc[y]) if qc[y] > 0 else Fraction(1 if pc[y] > 0 else 0)
            if a > 0:
                for seq, pr in node(c + (y,), d - 1).items():
                    _add(law, (y,) + seq, qy * a * pr)
            if a < 1:
                # a residual without mass (possible only when the draws and
                # the q update do not match) leaves p_cur as it is
                massless = sum(max(Fraction(0), a_ - b_) for a_, b_ in zip(pc, qc)) == 0
                r = pc if massless else positive_residual(pc, qc)
                qn = without(qc, y) if q_update == "renormalise" else qc
                dn = without(qdraw, y) if draws == "without" else qdraw
                for seq, pr in siblings(c, r, qn, dn, left - 1, d).items():
                    _add(law, seq, qy * (1 - a) * pr)
        return law

    return node(ctx, depth)


def spec_law(m: ToyModels, ctx: Tuple[int, ...], M: int, width: int, depth: int, draws: str = "iid",
             q_update: str = "fixed") -> Law:
    """Law of the first M committed tokens over as many rounds as needed."""
    if M <= 0:
        return {(): Fraction(1)}
    law: Law = {}
    for seq, pr in round_law(m, ctx, width, depth, draws, q_update).items():
        if len(seq) >= M:
            _add(law, seq[:M], pr)
        else:
            for rest, pr2 in spec_law(m, ctx + seq, M - len(seq), width, depth, draws, q_update).items():
                _add(law, seq + rest, pr * pr2)
    return law


def target_law(m: ToyModels, ctx: Tuple[int, ...], M: int) -> Law:
    """Autoregressive law of M tokens sampled from the target alone."""
    law: Law = {(): Fraction(1)}
    for _ in range(M):
        nxt: Law = {}
        for seq, pr in law.items():
            for t, pt in enumerate(m.p(ctx + seq)):
                _add(nxt, seq + (t,), pr * pt)
        law = nxt
    return law
