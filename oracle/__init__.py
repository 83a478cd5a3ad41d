"""CPU oracle for the speculative-decoding draft/verify path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  It is a plain,
single-threaded fp64 statement of the method (``specdec_oracle.c``) plus a
ctypes wrapper over numpy arrays; it shares no code with the CUDA library.

Every function here forwards to the C routine of the same name without extra
arithmetic; see the comments in ``specdec_oracle.c`` for the passage each one
follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "specdec_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_liboracle.so")
_lib = None

F32 = 0
BF16 = 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
             "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _lib.oracle_pool_size.restype = ctypes.c_int64
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"{name}: invalid arguments (rc={rc})")


def logits_buffer(x):
    """(contiguous array, dtype code) for a float32 array or a uint16 array
    holding bf16 bit patterns."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.uint16:
        return x, BF16
    raise TypeError("logits must be float32 or uint16 (bf16 bits)")


def pool_size(k: int, num_steps: int) -> int:
    return int(lib().oracle_pool_size(ctypes.c_int(k), ctypes.c_int(num_steps)))


def softmax_topk(logits, T: float, k: int, want_probs: bool = False, score_T=None):
    """Top-k of each row with their probabilities at ``score_T`` (None: at
    T), and optionally the full distribution at T (oracle_softmax_topk)."""
    score_T = T if score_T is None else score_T
    x, dt = logits_buffer(logits)
    V = x.shape[-1]
    R = x.size // V
    topk_p = np.zeros((R, k), np.float64)
    topk_idx = np.zeros((R, k), np.int32)
    probs = np.zeros((R, V), np.float64) if want_probs else None
    flag = np.zeros(R, np.int32)
    rc = lib().oracle_softmax_topk(_p(x), ctypes.c_int(dt), ctypes.c_int64(R), ctypes.c_int64(V),
                                   ctypes.c_double(T), ctypes.c_double(score_T), ctypes.c_int(k),
                                   _p(topk_p), _p(topk_idx),
                                   _p(probs), _p(flag))
    _check(rc, "softmax_topk")
    return topk_p, topk_idx, probs, flag


def sample(u, logits=None, probs=None, T: float = 1.0):
    u = _c(u, np.float32)
    R = u.size
    if probs is not None:
        pr = _c(probs, np.float32)
        V = pr.shape[-1]
        x, dt = None, F32
    else:
        x, dt = logits_buffer(logits)
        V = x.shape[-1]
        pr = None
    tok = np.zeros(R, np.int32)
    prob = np.zeros(R, np.float64)
    margin = np.zeros(R, np.float64)
    fb = np.zeros(R, np.int32)
    rc = lib().oracle_sample(_p(x), ctypes.c_int(dt), _p(pr), ctypes.c_int64(R), ctypes.c_int64(V),
                             ctypes.c_double(T), _p(u), _p(tok), _p(prob), _p(margin), _p(fb))
    _check(rc, "sample")
    return tok, prob, margin, fb


class Pool:
    """Candidate pool [B, P] plus the frontier [B, k] of the draft tree."""

    def __init__(self, B: int, k: int, num_steps: int):
        self.B, self.k, self.num_steps = B, k, num_steps
        self.P = pool_size(k, num_steps)
        self.score = np.zeros((B, self.P), np.float32)
        self.token = np.full((B, self.P), -1, np.int32)
        self.parent = np.full((B, self.P), -1, np.int32)
        self.qrow = np.full((B, self.P), -1, np.int32)
        self.frontier_score = np.zeros((B, k), np.float32)
        self.frontier_id = np.zeros((B, k), np.int32)


def tree_expand(pool: Pool, step: int, topk_p, topk_idx):
    tp = _c(topk_p, np.float32)
    ti = _c(topk_idx, np.int32)
    rc = lib().oracle_tree_expand(ctypes.c_int(step), ctypes.c_int(pool.num_steps), ctypes.c_int(pool.B),
                                  ctypes.c_int(pool.k), _p(tp), _p(ti), _p(pool.score), _p(pool.token),
                                  _p(pool.parent), _p(pool.qrow), _p(pool.frontier_score),
                                  _p(pool.frontier_id))
    _check(rc, "tree_expand")
    return pool


def build_tree(pool: Pool, N: int, root_token, seq_lens):
    B = pool.B
    root = _c(root_token, np.int32)
    sl = _c(seq_lens, np.int32)
    out = {
        "draft_token": np.zeros((B, N), np.int32),
        "parent": np.zeros((B, N), np.int32),
        "positions": np.zeros((B, N), np.int32),
        "tree_mask": np.zeros((B, N, N), np.uint8),
        "retrieve_index": np.zeros((B, N), np.int32),
        "retrieve_next_token": np.zeros((B, N), np.int32),
        "retrieve_next_sibling": np.zeros((B, N), np.int32),
        "q_row": np.zeros((B, N), np.int32),
    }
    rc = lib().oracle_build_tree(
        ctypes.c_int(B), ctypes.c_int(pool.k), ctypes.c_int(pool.num_steps), ctypes.c_int(N),
        _p(pool.score), _p(pool.token), _p(pool.parent), _p(pool.qrow), _p(root), _p(sl),
        _p(out["draft_token"]), _p(out["parent"]), _p(out["positions"]), _p(out["tree_mask"]),
        _p(out["retrieve_index"]), _p(out["retrieve_next_token"]), _p(out["retrieve_next_sibling"]),
        _p(out["q_row"]))
    _check(rc, "build_tree")
    return out


def _verify_outputs(B, N):
    return {
        "committed": np.zeros((B, N), np.int32),
        "num_committed": np.zeros(B, np.int32),
        "accept_length": np.zeros(B, np.int32),
        "accept_path": np.zeros((B, N), np.int32),
        "next_root": np.zeros(B, np.int32),
        "walk_info": np.zeros((B, 3), np.int32),
    }


def verify_greedy(target, draft_token, next_token, next_sibling, budget=None, eos: int = -1):
    x, dt = logits_buffer(target)
    B, N, V = x.shape
    dtok = _c(draft_token, np.int32)
    nt = _c(next_token, np.int32)
    ns = _c(next_sibling, np.int32)
    bud = None if budget is None else _c(budget, np.int32)
    o = _verify_outputs(B, N)
    rc = lib().oracle_verify_greedy(
        ctypes.c_int(B), ctypes.c_int(N), ctypes.c_int64(V), ctypes.c_int(dt), _p(x), _p(dtok), _p(nt),
        _p(ns), _p(bud), ctypes.c_int32(eos), _p(o["committed"]), _p(o["num_committed"]),
        _p(o["accept_length"]), _p(o["accept_path"]), _p(o["next_root"]), _p(o["walk_info"]))
    _check(rc, "verify_greedy")
    return o


def verify_sample(target, T: float, q, draft_token, next_token, next_sibling, coins, u_final,
                  q_row=None, budget=None, eos: int = -1, without_replacement: bool = False,
                  top_k: int = 0, top_p: float = 1.0):
    x, dt = logits_buffer(target)
    B, N, V = x.shape
    qq = _c(q, np.float32)
    qr = None if q_row is None else _c(q_row, np.int32)
    dtok = _c(draft_token, np.int32)
    nt = _c(next_token, np.int32)
    ns = _c(next_sibling, np.int32)
    co = _c(coins, np.float32)
    uf = _c(u_final, np.float32)
    bud = None if budget is None else _c(budget, np.int32)
    o = _verify_outputs(B, N)
    o["margin"] = np.zeros(B, np.float64)
    counters = np.zeros(4, np.int64)
    rc = lib().oracle_verify_sample(
        ctypes.c_int(B), ctypes.c_int(N), ctypes.c_int64(V), ctypes.c_int(dt), _p(x), ctypes.c_double(T),
        _p(qq), _p(qr), _p(dtok), _p(nt), _p(ns), _p(co), _p(uf), _p(bud), ctypes.c_int32(eos),
        _p(o["committed"]), _p(o["num_committed"]), _p(o["accept_length"]), _p(o["accept_path"]),
        _p(o["next_root"]), _p(o["walk_info"]), _p(o["margin"]), _p(counters),
        ctypes.c_int(1 if without_replacement else 0), ctypes.c_int64(int(top_k)), ctypes.c_double(float(top_p)))
    _check(rc, "verify_sample")
    o["q_zero"], o["residual_fallback"], o["cdf_fallback"], o["nonfinite_rows"] = (int(c) for c in counters)
    return o


def filter_probs(p, top_k: int = 0, top_p: float = 1.0):
    """Target-side top-k / top-p filtering of probability rows [..., V]
    (oracle_filter_probs), returned as a new fp64 array."""
    x = np.array(p, dtype=np.float64, copy=True)
    V = x.shape[-1]
    rows = x.reshape(-1, V)
    for r in range(rows.shape[0]):
        row = np.ascontiguousarray(rows[r])
        rc = lib().oracle_filter_probs(ctypes.c_int64(V), _p(row), ctypes.c_int64(int(top_k)),
                                       ctypes.c_double(float(top_p)))
        _check(rc, "filter_probs")
        rows[r] = row
    return rows.reshape(x.shape)


def compact_slots(seq_lens, accept_path, accept_length, req_to_token, page_size: int,
                  kv_pool=None, bytes_per_slot: int = 0):
    """Returns outputs; req_to_token and kv_pool (uint8 [slots, bytes]) are
    updated in place like the device call."""
    sl = _c(seq_lens, np.int32)
    ap = _c(accept_path, np.int32)
    al = _c(accept_length, np.int32)
    assert req_to_token.dtype == np.int32 and req_to_token.flags.c_contiguous
    B, N = ap.shape
    max_ctx = req_to_token.shape[1]
    cap = B * (N - 1) if page_size == 1 else B * (-(-N // page_size) + 1)
    o = {
        "move_src": np.zeros((B, N), np.int32),
        "move_dst": np.zeros((B, N), np.int32),
        "num_moves": np.zeros(B, np.int32),
        "freed": np.full(max(cap, 1), -1, np.int32),
        "num_freed": np.zeros(1, np.int32),
        "new_kv_len": np.zeros(B, np.int32),
        "bad": np.zeros(1, np.int32),
    }
    num_slots = 0
    if kv_pool is not None:
        assert kv_pool.dtype == np.uint8 and kv_pool.flags.c_contiguous
        num_slots = kv_pool.shape[0]
        bytes_per_slot = kv_pool.shape[1]
    rc = lib().oracle_compact_slots(
        ctypes.c_int(B), ctypes.c_int(N), ctypes.c_int(page_size), _p(sl), _p(ap), _p(al),
        _p(req_to_token), ctypes.c_int64(max_ctx), _p(o["move_src"]), _p(o["move_dst"]),
        _p(o["num_moves"]), _p(o["freed"]), _p(o["num_freed"]), _p(o["new_kv_len"]),
        _p(kv_pool), ctypes.c_int64(num_slots), ctypes.c_int64(bytes_per_slot), _p(o["bad"]))
    _check(rc, "compact_slots")
    o["freed"] = o["freed"][: int(o["num_freed"][0])]
    return o


def tli_constrain_map(draft_logits, d2t, t2d, T: float, want_q: bool = False):
    x, dt = logits_buffer(draft_logits)
    Vd = x.shape[-1]
    R = x.size // Vd
    d2 = _c(d2t, np.int32)
    t2 = _c(t2d, np.int32)
    Vt = t2.size
    o = {
        "top1_draft": np.zeros(R, np.int32),
        "top1_target": np.zeros(R, np.int32),
        "top1_p": np.zeros(R, np.float64),
        "q_target": np.zeros((R, Vt), np.float64) if want_q else None,
        "row_flag": np.zeros(R, np.int32),
    }
    rc = lib().oracle_tli_constrain_map(
        ctypes.c_int64(R), ctypes.c_int64(Vd), ctypes.c_int64(Vt), _p(x), ctypes.c_int(dt), _p(d2), _p(t2),
        ctypes.c_double(T), _p(o["top1_draft"]), _p(o["top1_target"]), _p(o["top1_p"]),
        _p(o["q_target"]), _p(o["row_flag"]))
    _check(rc, "tli_constrain_map")
    return o


def pruned_head(hidden, weight, ids, d2t, T: float, want_logits: bool = False):
    """The pruned draft LM head (oracle_pruned_head): hidden [M, H] and
    weight [K, H] (float32, or uint16 bf16 bits), ids [K], d2t [V_d]."""
    h, hdt = logits_buffer(hidden)
    w, wdt = logits_buffer(weight)
    M, H = h.shape
    K = w.shape[0]
    assert w.shape[1] == H
    idv = _c(ids, np.int32)
    d2 = _c(d2t, np.int32)
    o = {"logits": np.zeros((M, K), np.float64) if want_logits else None,
         "top1_rank": np.zeros(M, np.int32), "top1_draft": np.zeros(M, np.int32),
         "top1_target": np.zeros(M, np.int32), "top1_p": np.zeros(M, np.float64),
         "row_max": np.zeros(M, np.float64), "row_z": np.zeros(M, np.float64), "row_flag": np.zeros(M, np.int32)}
    rc = lib().oracle_pruned_head(
        ctypes.c_int64(M), ctypes.c_int64(H), ctypes.c_int64(K), _p(h), ctypes.c_int(hdt), _p(w), ctypes.c_int(wdt),
        _p(idv), _p(d2), ctypes.c_double(T), _p(o["logits"]), _p(o["top1_rank"]), _p(o["top1_draft"]),
        _p(o["top1_target"]), _p(o["top1_p"]), _p(o["row_max"]), _p(o["row_z"]), _p(o["row_flag"]))
    _check(rc, "pruned_head")
    return o


def tli_plan(d2t, t2d):
    """The TLI map plan of (d2t, t2d): K, bitmap words, intersection ids
    before each word, each target's partner rank (layout of tli_plan_build;
    words = ceil(V_d / 32) rounded up to even, t2r padded to a multiple of 4)."""
    d2 = _c(d2t, np.int32)
    t2 = _c(t2d, np.int32)
    Vd, Vt = d2.size, t2.size
    words = (Vd + 31) // 32
    words += words & 1
    Vt4 = (Vt + 3) // 4 * 4
    o = {"K": np.zeros(1, np.int32), "bits": np.zeros(words, np.uint32), "before": np.zeros(words, np.uint32),
         "t2r": np.zeros(Vt4, np.int32)}
    rc = lib().oracle_tli_plan(ctypes.c_int64(Vd), ctypes.c_int64(Vt), _p(d2), _p(t2), _p(o["K"]), _p(o["bits"]),
                               _p(o["before"]), ctypes.c_int64(words), _p(o["t2r"]), ctypes.c_int64(Vt4))
    _check(rc, "tli_plan")
    return o


def map_ids(ids, table, fallback: int):
    a = _c(ids, np.int32)
    t = _c(table, np.int32)
    out = np.zeros_like(a)
    lib().oracle_map_ids(_p(a), _p(out), ctypes.c_int64(a.size), _p(t), ctypes.c_int64(t.size),
                         ctypes.c_int32(fallback))
    return out


def tli_check_config(topk: int, num_steps: int, num_draft_tokens: int) -> bool:
    return lib().oracle_tli_check_config(ctypes.c_int(topk), ctypes.c_int(num_steps),
                                         ctypes.c_int(num_draft_tokens)) == 0
