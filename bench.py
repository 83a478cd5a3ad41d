"""Benchmark: one whole speculative step (draft steps, tree build, batched
verify, KV compaction) over a batch of synthetic logits, on GB300.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config c3] [--mode sample]
                  [--impl ours|reference]

Prints one JSON line (rank 0).  The default workload is the EAGLE tree with
stochastic verification: B=128 requests, topk 8, 6 draft steps, 64 tree
nodes, vocabulary 128256, bf16 logits, temperature 0.7, KV compaction over a
page-16 slot pool with 4096-byte slots.  Inputs (draft logits 1.35 GB,
target logits 2.1 GB) are larger than L2, so no flush is needed between
steps.  ``--impl reference`` times the CPU oracle on a bounded sample of the
same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import CONFIGS, assemble_target, generate  # noqa: E402

METRIC = "verified tokens/s (whole draft + tree + verify + compaction step)"
FALLBACK_HBM_GBS = 6800.0
DOMINANT = "softmax_topk_kernel"


def describe(cfg, mode):
    w = (f"{cfg.name}: {cfg.kind} B={cfg.B} topk={cfg.topk} steps={cfg.steps} N={cfg.N} V={cfg.V}"
         + (f" V_t={cfg.V_t} K={cfg.K}" if cfg.kind == "tli" else "")
         + f" {str(cfg.dtype).replace('torch.', '')} logits, {mode} verify T={cfg.T}"
         + (f", KV compaction page {cfg.page_size} x {cfg.bytes_per_slot} B slots" if cfg.page_size else ""))
    return w


def default_mode(cfg):
    return cfg.modes[-1]


def config_dict(cfg, mode, q_mode, world):
    """The workload's description; the same dict for both arms."""
    return {"workload": describe(cfg, mode), "B": cfg.B, "topk": cfg.topk, "num_steps": cfg.steps,
            "N": cfg.N, "V": cfg.V, "mode": mode, "T": cfg.T, "q": q_mode if mode == "sample" else None,
            "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (draft + target logits), no flush" if input_bytes(cfg) > L2_BYTES
            else "inputs fit in L2: warm (resident) figures; cold figures with a 512 MB scrub under 'cold'"}


L2_BYTES = 129 * 2 ** 20
SCRUB_BYTES = 512 * 2 ** 20


def input_bytes(cfg):
    esz = 2 if cfg.dtype == torch.bfloat16 else 4
    return (cfg.table_rows * cfg.V + cfg.B * cfg.N * (cfg.V_t or cfg.V)) * esz


def host_info():
    """Host cores and CPU model (lscpu, else /proc/cpuinfo)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if model is None:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith(("model name", "cpu part", "hardware")):
                    model = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    import platform
    return {"nproc": os.cpu_count(), "cpu_model": model, "machine": platform.machine()}


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# The sources each profiled kernel is built from (its file and the headers
# it includes); a committed ncu summary counts only while their hash matches.
KERNEL_SOURCES = {
    "softmax_topk_kernel": ["draft.cu", "common.cuh", "cdf.cuh", "expand.cuh"],
    "softmax_sample_kernel": ["draft.cu", "common.cuh", "cdf.cuh", "expand.cuh"],
    "sample_verify_kernel": ["verify.cu", "walk.cuh", "cdf.cuh", "common.cuh", "chain.h"],
    "row_argmax_kernel": ["verify.cu", "walk.cuh", "cdf.cuh", "common.cuh", "chain.h"],
    "tli_planned_kernel": ["tli.cu", "common.cuh", "expand.cuh"],
    "pruned_head_kernel": ["head.cu", "common.cuh"],
    "filter_kernel": ["filter.cu", "common.cuh"],
}


def kernel_source_hash(kernel=None):
    """Hash of the sources of `kernel` (every source without one)."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "speculative_decoding_draft_select_gb300", "csrc")
    files = KERNEL_SOURCES.get(kernel) or sorted(os.listdir(d))
    for f in sorted(files):
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(p):
        return None
    vals = {}
    for line in open(p):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("source_sha256") != kernel_source_hash(kernel):
        return None
    try:
        return float(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out = ""

    def summary(self):
        if self.proc is None:
            return None
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sms.append(float(f[1]))
                maxes.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(sms)}


# ---------------------------------------------------------------------------


def rank_config(cfg, rank, world):
    """Weak scaling: with several ranks every rank verifies its own batch of
    the same shape (its own seed)."""
    return cfg.scaled(seed=cfg.seed + 7919 * rank) if world > 1 else cfg


def reduce_over_ranks(total_ms, tokens, world, device):
    """(the longest rank's timed span, the verified tokens of all ranks)."""
    if world == 1:
        return float(total_ms), float(tokens)
    span = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
    tok = torch.tensor([float(tokens)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(span, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.all_reduce(tok, op=torch.distributed.ReduceOp.SUM)
    return float(span.item()), float(tok.item())


def run_ours(args, cfg, mode, rank, world, steps=None, warmup=None, flush=False, do_e2e=True):
    """Time ``steps`` whole steps of one workload (after ``warmup``).  flush:
    write a 512 MB scrub buffer before every timed step (outside the step's
    events), so that inputs that fit in L2 are read cold."""
    import speculative_decoding_draft_select_gb300 as sd
    from speculative_decoding_draft_select_gb300 import pipeline as pl
    from speculative_decoding_draft_select_gb300.build import build

    build()
    sd.lib()
    steps = args.steps if steps is None else steps
    warmup = args.warmup if warmup is None else warmup
    dev = torch.device("cuda", torch.cuda.current_device())
    cfg = rank_config(cfg, rank, world)
    work = generate(cfg, dev)
    compact = bool(cfg.page_size)
    sampled = cfg.kind == "chain" and mode == "sample"
    q_mode = args.q or "logits"
    buf = pl.StepBuffers(cfg.kind, cfg.B, cfg.topk, cfg.steps, cfg.N, cfg.V, dev, want_q=(mode == "sample"),
                         sampled=sampled, V_t=cfg.V_t or None, page_size=cfg.page_size, q_mode=q_mode,
                         q_logit_dtype=cfg.dtype)
    eos = int(work["eos_id"])
    kv = work.get("kv_pool")
    # the target model's output for this tree (deterministic draft -> same tree every step)
    pl.run_draft(buf, work["draft_table"], cfg.T, work["root_token"], work["seq_lens"], draft_u=work["draft_u"],
                 d2t=work.get("d2t"), t2d=work.get("t2d"))
    target = assemble_target(work, buf.tree["q_row"]).contiguous()
    row_bytes = cfg.V * (2 if cfg.dtype == torch.bfloat16 else 4)

    stream = torch.cuda.current_stream()
    dom_events = []
    # timing events inside a captured graph must be event-record nodes
    # ("external" events); without that, steps run eagerly
    use_graph = not args.no_graph
    if use_graph:
        try:
            torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            use_graph = False

    def timing_event():
        if use_graph:
            return torch.cuda.Event(enable_timing=True, external=True)
        return torch.cuda.Event(enable_timing=True)

    class Timer:
        """CUDA events around the draft steps' softmax/top-k (softmax/draw, TLI) launches
        with R = B*topk rows (steps >= 1), on the launching stream."""
        record = False

        def begin(self, s):
            self.ev = None
            if self.record and s >= 1:
                self.ev = (timing_event(), timing_event())
                self.ev[0].record(torch.cuda.current_stream())

        def end(self, s):
            if self.ev is not None:
                self.ev[1].record(torch.cuda.current_stream())
                dom_events.append((self.ev, cfg.B * cfg.topk))

    timer = Timer()
    verify_events = []

    def step(record, inp=None):
        """One step; ``inp`` (e2e) replaces the per-step inputs."""
        w = dict(work, target=target) if inp is None else dict(work, **inp)
        timer.record = record
        pl.run_draft(buf, w["draft_table"], cfg.T, w["root_token"], w["seq_lens"], draft_u=w["draft_u"],
                     d2t=w.get("d2t"), t2d=w.get("t2d"), timer=timer)
        if record:
            ev = (timing_event(), timing_event())
            ev[0].record(torch.cuda.current_stream())
        pl.run_verify(buf, w["target"], mode, cfg.T, w["coins"], w["u_final"], w.get("budget"), eos)
        if record:
            ev[1].record(torch.cuda.current_stream())
            verify_events.append(ev)
        if compact:
            pl.run_compact(buf, w["seq_lens"], w["req_to_token"], cfg.page_size, kv_pool=kv)

    for _ in range(warmup):
        step(False)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # one CUDA graph per timed step (each holds its own timing events, so
    # every step's launch times can be read after the loop); each is
    # replayed once untimed first
    graphs = None
    if use_graph:
        graphs = [pl.capture_step(lambda: step(True), warm=False) for _ in range(steps)]
        for g in graphs:
            g.replay()
        torch.cuda.synchronize()
    scrub = torch.empty(SCRUB_BYTES, dtype=torch.uint8, device=dev) if flush else None
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    committed = 0
    with ClockSampler(torch.cuda.current_device()) as clk:
        t0 = time.perf_counter()
        for i in range(steps):
            if scrub is not None:
                scrub.fill_(i & 0xFF)  # evicts the step's inputs from L2
            starts[i].record(stream)
            if graphs is not None:
                graphs[i].replay()
            else:
                step(True)
            ends[i].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    # steps back to back: first start to last end; with a flush between
    # steps, the sum of the steps' own intervals (the scrubs left out)
    total_ms = sum(step_ms) if flush else starts[0].elapsed_time(ends[-1])
    committed = int(buf.verify_out["num_committed"].sum().item())
    accept = float(buf.verify_out["accept_length"].float().mean().item())
    dom_ms = [ev[0].elapsed_time(ev[1]) for ev, _ in dom_events]
    dom_rows = [r for _, r in dom_events]

    total_ms_max, tokens_all = reduce_over_ranks(total_ms, committed * steps, world, dev)
    value = tokens_all / (total_ms_max / 1e3)

    peak, peak_kind = hbm_peak()
    # the draft kernel: the draft-step softmax/top-k (or softmax+draw, or TLI
    # constrain) launches of steps >= 1, each timed on its own
    if cfg.kind == "tli":
        # the draft row read, and q written in target order: fp32
        # probabilities, or the partners' logits and the row's (m, Z)
        q_row = 0
        if mode == "sample":
            q_row = cfg.V_t * 4 if q_mode == "probs" else cfg.V_t * (row_bytes // cfg.V) + 8
        per_row = row_bytes + q_row
        kname = "tli_planned_kernel"
    else:
        per_row = row_bytes + (cfg.V * 4 if buf.q is not None else 0)  # read + written q
        kname = "softmax_sample_kernel" if (cfg.kind == "chain" and mode == "sample") else DOMINANT
    dom_avg_ms = statistics.mean(dom_ms) if dom_ms else None
    dom_bytes = per_row * statistics.mean(dom_rows) if dom_rows else None
    draft_roof = None
    if dom_ms:
        achieved = dom_bytes / (dom_avg_ms * 1e-3) / 1e9
        draft_roof = {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1), "peak": peak,
                      "peak_source": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                      "bytes_per_launch": int(dom_bytes), "avg_launch_us": round(dom_avg_ms * 1e3, 2),
                      "launches_per_step": len(dom_ms) // max(steps, 1),
                      "traffic": ncu_traffic(kname, cfg.name)}

    # the batched verify (row statistics of every target row + tree walk):
    # target-logit bytes read / its time.  Stochastic: one launch
    # (sample_verify_kernel; its flag reset is a 4-byte-per-row memset in the
    # same timed interval); greedy: the argmax pass and the walk.
    verify = None
    verify_roof = None
    if verify_events:
        v_ms = statistics.mean(a.elapsed_time(b) for a, b in verify_events)
        v_bytes = cfg.B * cfg.N * (cfg.V_t or cfg.V) * (2 if cfg.dtype == torch.bfloat16 else 4)  # target rows
        v_gbs = v_bytes / (v_ms * 1e-3) / 1e9
        verify = {"us_per_step": round(v_ms * 1e3, 2), "logit_bytes": int(v_bytes), "achieved": round(v_gbs, 1),
                  "peak": peak, "unit": "GB/s", "frac": round(v_gbs / peak, 4)}
        if mode == "sample":
            # the walks' own bytes, from the walk records of the last step (every
            # step walks the same trees): one residual pass over a target row and
            # a q row per rejected child, one pass over the target row per bonus
            # draw at a leaf (a correction reuses its last pass)
            wi = buf.verify_out["walk_info"].cpu().numpy()
            s_t = 2 if cfg.dtype == torch.bfloat16 else 4
            s_q = 4 if q_mode == "probs" else s_t
            Vt = cfg.V_t or cfg.V
            rej = int(wi[:, 1].astype(np.int64).sum())
            bonus = int((wi[:, 2] == 2).sum())
            walk_bytes = rej * Vt * (s_t + s_q) + bonus * Vt * s_t
            w_gbs = (v_bytes + walk_bytes) / (v_ms * 1e-3) / 1e9
            verify.update({"residual_passes": rej, "bonus_draws": bonus, "walk_bytes": int(walk_bytes),
                           "achieved_with_walks": round(w_gbs, 1), "frac_with_walks": round(w_gbs / peak, 4)})
        vname = "sample_verify_kernel" if mode == "sample" else "row_argmax_kernel"
        verify_roof = {"bound": "hbm", "kernel": vname if mode == "sample" else vname + " (+ greedy_walk_kernel)",
                       "achieved": round(v_gbs, 1), "peak": peak, "peak_source": peak_kind, "unit": "GB/s",
                       "frac": round(v_gbs / peak, 4), "bytes_per_launch": int(v_bytes),
                       "avg_launch_us": round(v_ms * 1e3, 2), "launches_per_step": 1,
                       "traffic": ncu_traffic(vname, cfg.name)}
    # the dominant kernel is the one with the larger time per step
    roofline = draft_roof
    if verify_roof and (draft_roof is None or verify_roof["avg_launch_us"] >
                        draft_roof["avg_launch_us"] * draft_roof["launches_per_step"]):
        roofline = verify_roof

    # e2e: host buffers through the same API, copies inside the timed region
    e2e = run_e2e(args, cfg, mode, work, buf, target, step, compact) if (do_e2e and not args.no_e2e) else None

    launches = pl.kernels_per_step(buf, mode, compact, kv is not None) * steps
    clocks = clk.summary()
    ms_per_step = total_ms_max / steps
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "input_dtype": str(cfg.dtype).replace("torch.", ""),
        "data": "synthetic (seeded; shapes and value distributions of the workload, no model weights)",
        "config": config_dict(cfg, mode, q_mode, world), "cuda_graph": graphs is not None,
        "l2_flush": flush,
        "us_per_step_median": round(statistics.median(step_ms) * 1e3, 2),
        "verified_tokens_per_step": committed, "mean_accept_length": round(accept, 3),
        "roofline": roofline, "rooflines": {"draft": draft_roof, "verify": verify_roof}, "verify": verify,
        "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
        "stats": buf.stats.cpu().tolist(),
    }
    return line, work, buf


def run_e2e(args, cfg, mode, work, buf, target, step_fn, compact):
    """Per step: pinned-host -> device copies of the step's inputs, the step,
    device -> host copy of its results.  The copies of step i+1 run on a
    copy stream while step i computes (two device input sets); each step
    waits for its own inputs, and its results are read back before the
    step's end is timed."""
    inputs = {"draft_table": work["draft_table"], "target": target, "coins": work["coins"],
              "u_final": work["u_final"], "root_token": work["root_token"], "seq_lens": work["seq_lens"]}
    host = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in inputs.items()}
    for k, v in inputs.items():
        host[k].copy_(v)
    dev_sets = [inputs, {k: torch.empty_like(v) for k, v in inputs.items()}]
    outs = {"committed": buf.verify_out["committed"], "num_committed": buf.verify_out["num_committed"],
            "accept_length": buf.verify_out["accept_length"], "next_root": buf.verify_out["next_root"]}
    if compact:
        outs.update({"new_kv_len": buf.compact_out["new_kv_len"], "num_freed": buf.compact_out["num_freed"],
                     "freed": buf.compact_out["freed"]})
    host_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in outs.items()}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    n = max(1, min(args.steps, 10))
    compute = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    copied = [torch.cuda.Event() for _ in range(2)]   # inputs of set j landed
    consumed = [torch.cuda.Event() for _ in range(2)]  # set j's step done with its inputs

    def upload(i):
        j = i % 2
        with torch.cuda.stream(copy):
            if i >= 2:
                copy.wait_event(consumed[j])
            for k, v in dev_sets[j].items():
                v.copy_(host[k], non_blocking=True)
            copied[j].record(copy)

    torch.cuda.synchronize()
    t0 = time.perf_counter()
    tokens = 0
    upload(0)
    for i in range(n):
        j = i % 2
        if i + 1 < n:
            upload(i + 1)
        compute.wait_event(copied[j])
        step_fn(False, inp=dev_sets[j])
        consumed[j].record(compute)
        for k, v in outs.items():
            host_out[k].copy_(v, non_blocking=True)
        compute.synchronize()
        tokens += int(host_out["num_committed"].sum())
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    return {"value": round(tokens / dt, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": n, "ms_per_step": round(dt / n * 1e3, 3),
            "h2d_gbs": round(h2d / (dt / n) / 1e9, 1),
            "copy_overlap": "inputs of step i+1 copied while step i computes"}


# ---------------------------------------------------------------- reference


def oracle_sample(cfg, mode, work, budget_s, start=0, kv_host=None, keep=None):
    """The CPU oracle, single-threaded, on requests start, start+1, ... (mod
    B) until ``budget_s`` seconds of oracle time are spent (at least one).
    kv_host: the slot payload pool as a host array, moved in place by the
    oracle's compaction.  keep: a list that receives (b, oracle outputs)."""
    from oracle.pipeline import fetch_request, run_request

    tokens, secs, reqs = 0, 0.0, 0
    for i in range(cfg.B):
        b = (start + i) % cfg.B
        d = fetch_request(cfg, work, b)
        t0 = time.perf_counter()
        tree, _, _, v, _ = run_request(cfg, d, mode, compact=bool(cfg.page_size), kv_pool=kv_host)
        secs += time.perf_counter() - t0
        tokens += int(v["num_committed"][0])
        reqs += 1
        if keep is not None:
            keep.append((b, tree, v))
        if secs >= budget_s:
            break
    return tokens, secs, reqs


VERIFY_FIELDS = ("committed", "num_committed", "accept_length", "accept_path", "next_root", "walk_info")


def compare_with_oracle(cfg, mode, buf, kept, boundary=1e-5):
    """The GPU step's tree and verify outputs against the oracle's, request
    by request: exact, differing only within ``boundary`` of a stochastic
    decision boundary (the oracle's margin), or a mismatch."""
    import numpy as np
    tree = {k: v.cpu().numpy() for k, v in buf.tree.items()}
    out = {k: v.cpu().numpy() for k, v in buf.verify_out.items()}
    exact = near = bad = 0
    for b, ot, o in kept:
        same_tree = all(np.array_equal(tree[k][b], ot[k][0] + (b * cfg.N if k == "retrieve_index" else 0))
                        for k in ("draft_token", "parent", "positions", "retrieve_index", "retrieve_next_token",
                                  "retrieve_next_sibling"))
        same = same_tree and all(np.array_equal(out[k][b], o[k][0]) for k in VERIFY_FIELDS)
        if same:
            exact += 1
        elif (same_tree and mode == "sample" and o["margin"][0] < boundary) or o["draft_margin"] < boundary:
            near += 1
        else:
            bad += 1
    return {"compared": len(kept), "exact": exact, "boundary": near, "mismatch": bad,
            "rule": "a request may differ only where the oracle's uniform lies within 1e-5 of a decision boundary"}


def cpu_baseline(cfg, mode, work, buf=None, budget_s=15.0):
    keep = [] if buf is not None else None
    tokens, secs, reqs = oracle_sample(cfg, mode, work, budget_s, keep=keep)
    line = {"value": round(tokens / secs, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{reqs} of {cfg.B} requests of {cfg.name}, one at a time (full draft, tree, verify"
                      f"{', compaction index work' if cfg.page_size else ''}); {tokens} tokens in {secs:.2f} s",
            "host": host_info()}
    parity = compare_with_oracle(cfg, mode, buf, keep) if buf is not None else None
    return line, parity


def run_reference(args, cfg, mode, rank, world):
    """The oracle as the reference arm: each timed step is a bounded sample
    of the workload's requests (consecutive steps take consecutive
    requests), timed on one host core, including the compaction's payload
    moves on a host copy of the slot pool."""
    if rank != 0:
        return None
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    work = generate(cfg, dev)
    kv_host = work["kv_pool"].cpu().numpy() if "kv_pool" in work else None
    per_step_budget = max(1.0, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
    nxt = 0
    for _ in range(args.warmup):
        _, _, r = oracle_sample(cfg, mode, work, per_step_budget / 4, start=nxt, kv_host=kv_host)
        nxt += r
    tok, sec = 0, 0.0
    reqs = 0
    for _ in range(args.steps):
        t, s, r = oracle_sample(cfg, mode, work, per_step_budget, start=nxt, kv_host=kv_host)
        tok, sec, reqs, nxt = tok + t, sec + s, reqs + r, nxt + r
    value = tok / sec
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec / args.steps * 1e3, 3),
        "ms_per_step_kind": (f"oracle time of one bounded sample per step ({reqs / args.steps:.1f} of "
                             f"{cfg.B} requests on average), not of the whole batch"),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; same generator as the GPU arm)",
        "config": config_dict(cfg, mode, args.q or "logits", world),
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"{reqs} requests over {args.steps} steps, one at a time, fp64 C oracle",
                         "host": host_info()},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="c3", choices=sorted(CONFIGS))
    ap.add_argument("--mode", default=None, choices=[None, "greedy", "sample"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--filter-only", action="store_true", help="time target-side filtering alone")
    ap.add_argument("--q", default=None, choices=[None, "logits", "probs"],
                    help="draft distribution for stochastic verify: logit rows + row stats, or written fp32 rows")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=None, help="override B (profiling a smaller case)")
    ap.add_argument("--no-graph", action="store_true", help="launch every kernel eagerly (no CUDA graph)")
    ap.add_argument("--head-only", action="store_true",
                    help="time only the pruned draft LM head (the TLI workload's tensor-core GEMM) and print it")
    ap.add_argument("--no-configs", action="store_true",
                    help="measure only the chosen workload (by default the c3 line also carries c1, c2, c4, c5)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    cfg = CONFIGS[args.config]
    if args.batch:
        cfg = cfg.scaled(B=args.batch)
    mode = args.mode or default_mode(cfg)

    if args.impl == "reference":
        line = run_reference(args, cfg, mode, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    torch.cuda.set_device(local)
    if args.filter_only:
        from speculative_decoding_draft_select_gb300.build import build
        build()
        print(json.dumps(filter_leg(B=args.batch or 128)), flush=True)
        return
    if args.head_only:
        from speculative_decoding_draft_select_gb300.build import build
        build()
        print(json.dumps(pruned_head_leg()), flush=True)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    line, work, buf = run_ours(args, cfg, mode, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"], line["boundary_cases"] = cpu_baseline(cfg, mode, work, buf)
        del work, buf
        torch.cuda.empty_cache()
        if not args.no_configs and world == 1 and args.config == "c3" and not args.batch:
            line["configs"] = other_configs(args)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# the other workloads, each measured after the headline one (same process,
# one at a time); those whose inputs fit in L2 also cold
OTHER_CONFIGS = [("c1", "greedy"), ("c1", "sample"), ("c2", "greedy"), ("c4", "sample"), ("c5", "greedy"),
                 ("c5", "sample")]


def summarize(line):
    v, d = line["verify"], line["rooflines"]["draft"]
    out = {"workload": line["config"]["workload"], "tokens_per_s": line["value"], "ms_per_step": line["ms_per_step"],
           "steps": line["steps"], "mean_accept_length": line["mean_accept_length"],
           "verify": None if v is None else dict({"us": v["us_per_step"], "gbs": v["achieved"], "frac": v["frac"],
                                                   "logit_bytes": v["logit_bytes"]},
                                                  **{k: v[k] for k in ("walk_bytes", "frac_with_walks") if k in v}),
           "draft": None if d is None else {"kernel": d["kernel"], "avg_launch_us": d["avg_launch_us"],
                                             "launches_per_step": d["launches_per_step"], "gbs": d["achieved"],
                                             "frac": d["frac"]},
           "clocks": line["clocks"], "stats": line["stats"]}
    return out


def tensor_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (burst)"
    except Exception:
        return 1900.0, "fallback"


def pruned_head_leg(M=256, H=896, K=60000, Vd=151936, Vt=128256, launches=20):
    """The TLI draft step with the pruned LM head (tli_pruned_head): the
    hidden states [M, H] of one draft step times the K intersection rows of a
    synthetic bf16 LM head [K, H] (H = 896, a 0.5B draft model's width), top-1
    and softmax statistics fused.  Timed per launch with CUDA events, cold
    (a 512 MB scrub before each launch: the 107.5 MB of weights would
    otherwise stay in L2) and warm."""
    import speculative_decoding_draft_select_gb300 as sd
    dev = torch.device("cuda", torch.cuda.current_device())
    g = torch.Generator(device=dev)
    g.manual_seed(1004 * 1009 + 77)
    hidden = torch.randn((M, H), generator=g, device=dev).to(torch.bfloat16)
    weight = (torch.randn((K, H), generator=g, device=dev) * (3.0 / H ** 0.5)).to(torch.bfloat16)
    ids = torch.sort(torch.randperm(Vd, generator=g, device=dev)[:K]).values.to(torch.int32)
    d2t = torch.full((Vd,), -1, dtype=torch.int32, device=dev)
    d2t[ids.long()] = torch.randperm(Vt, generator=g, device=dev)[:K].to(torch.int32)
    out = sd.tli_pruned_head(hidden, weight, ids, d2t, 1.0)
    ws = torch.empty(max(int(sd.lib().tli_pruned_head_ws_size(M, K)), 256), dtype=torch.uint8, device=dev)
    scrub = torch.empty(SCRUB_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    res = {}
    for mode in ("cold", "warm"):
        for _ in range(3):
            sd.tli_pruned_head(hidden, weight, ids, d2t, 1.0, out=out, ws=ws)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(launches)]
        for a, b in ev:
            if mode == "cold":
                scrub.fill_(1)
            a.record(stream)
            sd.tli_pruned_head(hidden, weight, ids, d2t, 1.0, out=out, ws=ws)
            b.record(stream)
        torch.cuda.synchronize()
        us = statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3
        flops = 2.0 * M * K * H
        byts = (K * H + M * H) * 2
        tpk, tsrc = tensor_peak()
        hpk, _ = hbm_peak()
        res[mode] = {"us": round(us, 2), "tflops": round(flops / (us * 1e-6) / 1e12, 1),
                     "tensor_frac": round(flops / (us * 1e-6) / 1e12 / tpk, 4),
                     "gbs": round(byts / (us * 1e-6) / 1e9, 1), "hbm_frac": round(byts / (us * 1e-6) / 1e9 / hpk, 4)}
    res.update({"workload": f"pruned draft LM head M={M} H={H} K={K} bf16, tcgen05 GEMM + fused top-1 and softmax "
                            f"statistics (2 launches: GEMM with epilogue, partial merge)",
                "flops_per_launch": 2 * M * K * H, "bytes_per_launch": (K * H + M * H) * 2,
                "tensor_peak_tflops": tensor_peak()[0], "tensor_peak_source": tensor_peak()[1],
                "traffic": ncu_traffic("pruned_head_kernel", "c4")})
    return res


def filter_leg(B=128, N=64, V=128256, T=0.7, top_k=50, top_p=0.9, launches=10):
    """Target-side top-k / top-p filtering (spec_filter_logits) of the c3
    target logits [B*N, V] bf16 in place, timed per launch with CUDA events.
    Each launch gets a fresh copy of the unfiltered logits first (untimed;
    2.1 GB, so L2 holds none of it).  Algorithmic bytes: every row read once
    and every dropped element written once."""
    import speculative_decoding_draft_select_gb300 as sd
    dev = torch.device("cuda", torch.cuda.current_device())
    g = torch.Generator(device=dev)
    g.manual_seed(1003 * 1009 + 55)
    src = (torch.randn((B * N, V), generator=g, device=dev) * 3.0).to(torch.bfloat16)
    x = torch.empty_like(src)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        x.copy_(src)
        sd.spec_filter_logits(x, T, top_k, top_p)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(launches)]
    for a, b in ev:
        x.copy_(src)
        a.record(stream)
        sd.spec_filter_logits(x, T, top_k, top_p)
        b.record(stream)
    torch.cuda.synchronize()
    us = statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3
    dropped = int(torch.isinf(x).sum()) - int(torch.isinf(src).sum())
    byts = B * N * V * 2 + dropped * 2
    hpk, hsrc = hbm_peak()
    gbs = byts / (us * 1e-6) / 1e9
    del src, x
    torch.cuda.empty_cache()
    return {"workload": f"target-side filtering of the c3 target logits: {B * N} rows x V={V} bf16 in place, "
                        f"T={T}, top_k={top_k}, top_p={top_p}",
            "us": round(us, 2), "bytes_per_launch": byts, "dropped_per_row": round(dropped / (B * N), 1),
            "gbs": round(gbs, 1), "hbm_frac": round(gbs / hpk, 4), "peak_source": hsrc,
            "traffic": ncu_traffic("filter_kernel", "c3") if B * N == 8192 else None}


def other_configs(args):
    res = {}
    try:
        res["c4_pruned_head"] = pruned_head_leg()
    except Exception as e:  # reported, not hidden
        res["c4_pruned_head"] = {"error": f"{type(e).__name__}: {e}"}
    torch.cuda.empty_cache()
    try:
        res["c3_filter"] = filter_leg()
    except Exception as e:  # reported, not hidden
        res["c3_filter"] = {"error": f"{type(e).__name__}: {e}"}
    for name, mode in OTHER_CONFIGS:
        cfg = CONFIGS[name]
        steps = max(3, min(args.steps, 10))
        warm, w, b = run_ours(args, cfg, mode, 0, 1, steps=steps, warmup=3, do_e2e=False)
        del w, b
        entry = summarize(warm)
        if input_bytes(cfg) <= L2_BYTES:
            cold, w, b = run_ours(args, cfg, mode, 0, 1, steps=steps, warmup=3, flush=True, do_e2e=False)
            del w, b
            entry["cold"] = {k: summarize(cold)[k] for k in ("tokens_per_s", "ms_per_step", "verify", "draft",
                                                             "clocks")}
        torch.cuda.empty_cache()
        res[f"{name}_{mode}"] = entry
    return res


if __name__ == "__main__":
    main()
