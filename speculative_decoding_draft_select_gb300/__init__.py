"""Python binding of libspecdec.so (include/specdec.h).

Argument marshalling only: every function checks that its tensors live on
the GPU, are contiguous and have the expected dtype, allocates outputs the
caller did not pass (torch.empty on the same device), and calls the C entry
point of the same name on torch's current CUDA stream.  All computation runs
in the library's CUDA kernels; there is no CPU path.  If the library is not
built, the first call raises.  With SPECDEC_DEBUG=1 in the environment the
bounds-checking build, libspecdec_debug.so, is loaded instead (build it with
build(debug=True)); spec_debug_bounds reads its count.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "SpecError", "F32", "BF16", "STATS", "lib", "library_path",
    "spec_softmax_topk", "spec_softmax_sample", "spec_sample", "spec_tree_pool_size", "spec_tree_expand", "spec_build_tree",
    "spec_verify_ws_size", "spec_verify_greedy", "spec_verify_greedy_noalloc", "spec_verify_sample",
    "spec_verify_sample_qlogits", "WITHOUT_REPLACEMENT", "CHAIN", "spec_compact_freed_capacity",
    "spec_compact_slots", "tli_constrain_map", "tli_constrain_map_qlogits", "tli_plan_bytes", "tli_plan_build",
    "tli_map_ids",
    "tli_check_config", "tli_pruned_head", "spec_filter_logits", "spec_wait_probe", "spec_debug_bounds",
    "new_stats", "new_pool",
]

F32 = 0
BF16 = 1
STATS = {"nonfinite_row": 0, "q_zero": 1, "residual_fallback": 2, "cdf_fallback": 3,
         "empty_intersection": 4, "bad_request": 5, "wait_timeout": 6, "bounds": 7}
NUM_STATS = 8
_ERRORS = {-1: "invalid argument", -2: "unsupported", -3: "CUDA launch failed", -4: "workspace too small"}

library_path = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                            "libspecdec_debug.so" if os.environ.get("SPECDEC_DEBUG") == "1" else "libspecdec.so")
_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_F = ctypes.c_float
_SZ = ctypes.c_size_t

_SIGS = {
    "spec_softmax_topk": (_I, [_P, _I, _I64, _I64, _F, _F, _I, _P, _P, _P, _P, _P, _P]),
    "spec_sample": (_I, [_P, _I, _P, _I64, _I64, _F, _P, _P, _P, _P, _P, _P]),
    "spec_softmax_sample": (_I, [_P, _I, _I64, _I64, _F, _P, _P, _P, _P, _P, _P, _P]),
    "spec_tree_pool_size": (_I64, [_I, _I]),
    "spec_tree_expand": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "spec_build_tree": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "spec_verify_ws_size": (_SZ, [_I, _I]),
    "spec_verify_greedy": (_I, [_I, _I, _I64, _I, _P, _P, _P, _P, _P, _I32, _P, _P, _P, _P, _P, _P, _P, _P,
                                _SZ, _P]),
    "spec_verify_sample": (_I, [_I, _I, _I64, _I, _P, _F, _P, _P, _P, _P, _P, _P, _P, _P, _I32, _P, _P, _P,
                                _P, _P, _P, _P, _P, _SZ, _P]),
    "spec_verify_sample_qlogits": (_I, [_I, _I, _I64, _I, _P, _F, _P, _I, _P, _F, _P, _P, _P, _P, _P, _P, _P,
                                        _I32, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "spec_verify_sample_flags": (_I, [_I, _I, _I64, _I, _P, _F, _P, _P, _P, _P, _P, _P, _P, _P, _I32, _P, _P, _P,
                                      _P, _P, _P, _P, _P, _SZ, _I, _P]),
    "spec_verify_sample_qlogits_flags": (_I, [_I, _I, _I64, _I, _P, _F, _P, _I, _P, _F, _P, _P, _P, _P, _P, _P,
                                              _P, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I, _P]),
    "spec_compact_freed_capacity": (_I64, [_I, _I, _I]),
    "spec_compact_slots": (_I, [_I, _I, _I, _P, _P, _P, _P, _I64, _P, _P, _P, _P, _I64, _P, _P, _P, _I64,
                                _I64, _P, _P]),
    "tli_constrain_map": (_I, [_I64, _I64, _I64, _P, _I, _P, _P, _F, _P, _P, _P, _P, _P, _P]),
    "tli_plan_bytes": (_I64, [_I64, _I64]),
    "tli_plan_build": (_I, [_I64, _I64, _P, _P, _P, _P]),
    "tli_constrain_map_planned": (_I, [_I64, _I64, _I64, _P, _I, _P, _P, _P, _F, _P, _P, _P, _P, _P, _P]),
    "tli_constrain_map_planned_expand": (_I, [_I64, _I64, _I64, _P, _I, _P, _P, _P, _F, _P, _P, _P, _P, _P, _P,
                                              _P]),
    "tli_constrain_map_qlogits": (_I, [_I64, _I64, _I64, _P, _I, _P, _P, _P, _F, _P, _P, _P, _P, _P, _P, _P, _P]),
    "spec_softmax_topk_expand": (_I, [_P, _I, _I64, _I64, _F, _F, _I, _P, _P, _P, _P, _P, _P, _P]),
    "spec_softmax_sample_expand": (_I, [_P, _I, _I64, _I64, _F, _P, _P, _P, _P, _P, _P, _P, _P]),
    "spec_verify_sample_qlogits_mapped": (_I, [_I, _I, _I64, _I, _P, _F, _P, _I, _P, _F, _P, _P, _P, _P, _P, _P,
                                               _P, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I, _P, _P]),
    "spec_verify_greedy_noalloc": (_I, [_I, _I, _I64, _I, _P, _P, _P, _P, _P, _I32, _P, _P, _P, _P, _P, _P, _P,
                                        _P]),
    "tli_map_ids": (_I, [_P, _P, _I64, _P, _I64, _I32, _P]),
    "spec_wait_probe": (_I, [_P, _I64, _P, _P, _P]),
    "spec_debug_bounds": (_I, [_P, _I]),
    "tli_check_config": (_I, [_I, _I, _I]),
    "spec_filter_logits": (_I, [_P, _I, _I64, _I64, _F, _I64, _F, _P, _P]),
    "tli_pruned_head_ws_size": (_SZ, [_I64, _I64]),
    "tli_pruned_head": (_I, [_I64, _I64, _I64, _P, _P, _P, _P, _I64, _F, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
}


class _Expand(ctypes.Structure):
    """spec_expand_t of include/specdec.h."""
    _fields_ = [("step", ctypes.c_int), ("num_steps", ctypes.c_int), ("B", ctypes.c_int), ("k", ctypes.c_int),
                ("pool_score", _P), ("pool_token", _P), ("pool_parent", _P), ("pool_qrow", _P),
                ("frontier_score", _P), ("frontier_id", _P), ("counters", _P)]


def _expand(expand):
    """(pool, step) -> a ctypes pointer to its spec_expand_t (None -> None)."""
    if expand is None:
        return None
    pool, step = expand
    x = _Expand(int(step), pool["num_steps"], pool["B"], pool["k"], *(pool[n].data_ptr() for n in (
        "score", "token", "parent", "qrow", "frontier_score", "frontier_id", "counters")))
    return ctypes.pointer(x)


class SpecError(RuntimeError):
    def __init__(self, name: str, rc: int):
        super().__init__(f"{name}: {_ERRORS.get(rc, 'error')} (rc={rc})")
        self.rc = rc


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise RuntimeError(f"{library_path} is missing: build it with "
                               "speculative_decoding_draft_select_gb300.build.build()")
        l = ctypes.CDLL(library_path)
        for name, (res, args) in _SIGS.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def _call(name, *args):
    rc = getattr(lib(), name)(*args)
    if rc != 0:
        raise SpecError(name, rc)


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _logit_code(t):
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise ValueError("logits must be float32 or bfloat16")


def _out(t, shape, dtype, like, name):
    if t is None:
        return torch.empty(shape, dtype=dtype, device=like.device)
    return _dev(t, dtype, name)


def new_stats(device="cuda"):
    """A zeroed int32[8] stats array."""
    return torch.zeros(NUM_STATS, dtype=torch.int32, device=device)


# ------------------------------------------------------------------- draft

def spec_softmax_topk(logits, T, k, topk_p=None, topk_idx=None, probs=None, want_probs=False, row_stats=None,
                      stats=None, expand=None, score_T=None):
    """logits [R, V] -> (topk_p [R, k] f32, topk_idx [R, k] i32, probs [R, V] f32 or None).
    probs and row_stats [R, 2] f32 (optional: each row's (max, normaliser))
    are at temperature T; topk_p at score_T (None: T).
    expand = (pool, step): the step's pool expansion in the same launch."""
    score_T = T if score_T is None else score_T
    _dev(logits, name="logits")
    V = logits.shape[-1]
    R = logits.numel() // V
    topk_p = _out(topk_p, (R, k), torch.float32, logits, "topk_p")
    topk_idx = _out(topk_idx, (R, k), torch.int32, logits, "topk_idx")
    if want_probs and probs is None:
        probs = torch.empty((R, V), dtype=torch.float32, device=logits.device)
    _dev(probs, torch.float32, "probs")
    _dev(row_stats, torch.float32, "row_stats")
    _dev(stats, torch.int32, "stats")
    if expand is not None:
        _call("spec_softmax_topk_expand", _ptr(logits), _logit_code(logits), R, V, float(T), float(score_T), int(k),
              _ptr(topk_p),
              _ptr(topk_idx), _ptr(probs), _ptr(row_stats), _ptr(stats), _expand(expand), _stream())
    else:
        _call("spec_softmax_topk", _ptr(logits), _logit_code(logits), R, V, float(T), float(score_T), int(k),
              _ptr(topk_p),
              _ptr(topk_idx), _ptr(probs), _ptr(row_stats), _ptr(stats), _stream())
    return topk_p, topk_idx, probs


def spec_softmax_sample(logits, T, u, out_token=None, out_prob=None, row_stats=None, probs=None, want_probs=False,
                        stats=None, expand=None):
    """Draft softmax and one inverse-CDF token per row in one pass:
    logits [R, V], u [R] -> (out_token [R] i32, out_prob [R] f32, probs or
    None); row_stats [R, 2] (optional) receives (max, normaliser)."""
    _dev(logits, name="logits")
    _dev(u, torch.float32, "u")
    V = logits.shape[-1]
    R = logits.numel() // V
    out_token = _out(out_token, (R,), torch.int32, logits, "out_token")
    out_prob = _out(out_prob, (R,), torch.float32, logits, "out_prob")
    if want_probs and probs is None:
        probs = torch.empty((R, V), dtype=torch.float32, device=logits.device)
    _dev(probs, torch.float32, "probs")
    _dev(row_stats, torch.float32, "row_stats")
    _dev(stats, torch.int32, "stats")
    if expand is not None:
        _call("spec_softmax_sample_expand", _ptr(logits), _logit_code(logits), R, V, float(T), _ptr(u),
              _ptr(out_token), _ptr(out_prob), _ptr(row_stats), _ptr(probs), _ptr(stats), _expand(expand), _stream())
    else:
        _call("spec_softmax_sample", _ptr(logits), _logit_code(logits), R, V, float(T), _ptr(u), _ptr(out_token),
              _ptr(out_prob), _ptr(row_stats), _ptr(probs), _ptr(stats), _stream())
    return out_token, out_prob, probs


def spec_sample(u, logits=None, probs=None, T=1.0, out_token=None, out_prob=None, stats=None, row_stats=None):
    """One token per row by inverse CDF with uniforms u [R].  row_stats
    [R, 2] (logits only, optional): the rows' (max, normaliser) from
    spec_softmax_topk, so that each row is read once."""
    src = probs if probs is not None else logits
    _dev(src, name="probs/logits")
    _dev(u, torch.float32, "u")
    V = src.shape[-1]
    R = src.numel() // V
    out_token = _out(out_token, (R,), torch.int32, src, "out_token")
    out_prob = _out(out_prob, (R,), torch.float32, src, "out_prob")
    _dev(stats, torch.int32, "stats")
    _dev(row_stats, torch.float32, "row_stats")
    if probs is not None:
        _dev(probs, torch.float32, "probs")
        code = F32
    else:
        code = _logit_code(logits)
    _call("spec_sample", _ptr(logits if probs is None else None), code, _ptr(probs), R, V, float(T), _ptr(u),
          _ptr(out_token), _ptr(out_prob), _ptr(row_stats if probs is None else None), _ptr(stats), _stream())
    return out_token, out_prob


def spec_tree_pool_size(k, num_steps):
    return int(lib().spec_tree_pool_size(int(k), int(num_steps)))


def new_pool(B, k, num_steps, device="cuda"):
    """Pool [B, P] (score, token, parent, qrow) and frontier [B, k] tensors."""
    P = spec_tree_pool_size(k, num_steps)
    return {
        "score": torch.empty((B, P), dtype=torch.float32, device=device),
        "token": torch.empty((B, P), dtype=torch.int32, device=device),
        "parent": torch.empty((B, P), dtype=torch.int32, device=device),
        "qrow": torch.empty((B, P), dtype=torch.int32, device=device),
        "frontier_score": torch.empty((B, k), dtype=torch.float32, device=device),
        "frontier_id": torch.empty((B, k), dtype=torch.int32, device=device),
        "counters": torch.zeros((B,), dtype=torch.int32, device=device),  # fused expansions: zero between steps
        "B": B, "k": k, "num_steps": num_steps, "P": P,
    }


def spec_tree_expand(pool, step, topk_p, topk_idx):
    _dev(topk_p, torch.float32, "topk_p")
    _dev(topk_idx, torch.int32, "topk_idx")
    _call("spec_tree_expand", int(step), pool["num_steps"], pool["B"], pool["k"], _ptr(topk_p), _ptr(topk_idx),
          _ptr(pool["score"]), _ptr(pool["token"]), _ptr(pool["parent"]), _ptr(pool["qrow"]),
          _ptr(pool["frontier_score"]), _ptr(pool["frontier_id"]), _stream())
    return pool


def spec_build_tree(pool, N, root_token, seq_lens, out=None):
    """Returns a dict of [B, N] tensors (tree_mask [B, N, N] uint8)."""
    B = pool["B"]
    dev = pool["score"].device
    _dev(root_token, torch.int32, "root_token")
    _dev(seq_lens, torch.int32, "seq_lens")
    if out is None:
        out = {name: torch.empty((B, N), dtype=torch.int32, device=dev)
               for name in ("draft_token", "parent", "positions", "retrieve_index", "retrieve_next_token",
                            "retrieve_next_sibling", "q_row")}
        out["tree_mask"] = torch.empty((B, N, N), dtype=torch.uint8, device=dev)
    _call("spec_build_tree", B, pool["k"], pool["num_steps"], int(N), _ptr(pool["score"]), _ptr(pool["token"]),
          _ptr(pool["parent"]), _ptr(pool["qrow"]), _ptr(root_token), _ptr(seq_lens), _ptr(out["draft_token"]),
          _ptr(out["parent"]), _ptr(out["positions"]), _ptr(out["tree_mask"]), _ptr(out["retrieve_index"]),
          _ptr(out["retrieve_next_token"]), _ptr(out["retrieve_next_sibling"]), _ptr(out["q_row"]), _stream())
    return out


# ------------------------------------------------------------------ verify

def spec_verify_ws_size(B, N):
    return int(lib().spec_verify_ws_size(int(B), int(N)))


def _verify_outputs(B, N, dev, out):
    if out is not None:
        return out
    return {
        "committed": torch.empty((B, N), dtype=torch.int32, device=dev),
        "num_committed": torch.empty((B,), dtype=torch.int32, device=dev),
        "accept_length": torch.empty((B,), dtype=torch.int32, device=dev),
        "accept_path": torch.empty((B, N), dtype=torch.int32, device=dev),
        "next_root": torch.empty((B,), dtype=torch.int32, device=dev),
        "walk_info": torch.empty((B, 3), dtype=torch.int32, device=dev),
    }


def _workspace(B, N, dev, ws):
    need = spec_verify_ws_size(B, N)
    if ws is None:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _dev(ws, torch.uint8, "ws")
    return ws


def spec_verify_greedy(target, draft_token, next_token, next_sibling, budget=None, eos_id=-1, out=None, ws=None,
                       stats=None):
    """target [B, N, V] (f32 or bf16)."""
    _dev(target, name="target")
    B, N, V = target.shape
    for name, t in (("draft_token", draft_token), ("next_token", next_token), ("next_sibling", next_sibling)):
        _dev(t, torch.int32, name)
    _dev(budget, torch.int32, "budget")
    _dev(stats, torch.int32, "stats")
    out = _verify_outputs(B, N, target.device, out)
    ws = _workspace(B, N, target.device, ws)
    _call("spec_verify_greedy", B, N, V, _logit_code(target), _ptr(target), _ptr(draft_token), _ptr(next_token),
          _ptr(next_sibling), _ptr(budget), int(eos_id), _ptr(out["committed"]), _ptr(out["num_committed"]),
          _ptr(out["accept_length"]), _ptr(out["accept_path"]), _ptr(out["next_root"]), _ptr(out.get("walk_info")),
          _ptr(stats), _ptr(ws), ws.numel(), _stream())
    return out


def spec_verify_greedy_noalloc(target, draft_token, next_token, next_sibling, budget=None, eos_id=-1, out=None,
                               stats=None):
    """Greedy verify for callers that cannot allocate device scratch: the
    library keeps the per-row argmax in its own fixed 1 MiB device array
    (B*N <= 262144 rows).  Outputs are still the caller's tensors (allocated
    here only when not passed).  Calls that overlap on the GPU race on the
    shared array."""
    _dev(target, name="target")
    B, N, V = target.shape
    for name, t in (("draft_token", draft_token), ("next_token", next_token), ("next_sibling", next_sibling)):
        _dev(t, torch.int32, name)
    _dev(budget, torch.int32, "budget")
    _dev(stats, torch.int32, "stats")
    out = _verify_outputs(B, N, target.device, out)
    _call("spec_verify_greedy_noalloc", B, N, V, _logit_code(target), _ptr(target), _ptr(draft_token),
          _ptr(next_token), _ptr(next_sibling), _ptr(budget), int(eos_id), _ptr(out["committed"]),
          _ptr(out["num_committed"]), _ptr(out["accept_length"]), _ptr(out["accept_path"]), _ptr(out["next_root"]),
          _ptr(out.get("walk_info")), _ptr(stats), _stream())
    return out


WITHOUT_REPLACEMENT = 1  # SPEC_VERIFY_WITHOUT_REPLACEMENT
CHAIN = 2  # SPEC_VERIFY_CHAIN


def spec_verify_sample(target, T, q, draft_token, next_token, next_sibling, coins, u_final, q_row=None,
                       budget=None, eos_id=-1, out=None, ws=None, stats=None, without_replacement=False,
                       chain=False):
    """target [B, N, V]; q fp32 rows of length V (a [rows, V] table with q_row [B, N], or [B, N, V]).
    without_replacement: the sibling update for children drawn without
    replacement (spec_verify_sample_flags with SPEC_VERIFY_WITHOUT_REPLACEMENT);
    chain: the trees are chains (SPEC_VERIFY_CHAIN: the chain verify launch)."""
    _dev(target, name="target")
    B, N, V = target.shape
    _dev(q, torch.float32, "q")
    if q.shape[-1] != V:
        raise ValueError("q rows must have length V")
    for name, t in (("draft_token", draft_token), ("next_token", next_token), ("next_sibling", next_sibling)):
        _dev(t, torch.int32, name)
    _dev(q_row, torch.int32, "q_row")
    _dev(coins, torch.float32, "coins")
    _dev(u_final, torch.float32, "u_final")
    _dev(budget, torch.int32, "budget")
    _dev(stats, torch.int32, "stats")
    out = _verify_outputs(B, N, target.device, out)
    ws = _workspace(B, N, target.device, ws)
    args = (B, N, V, _logit_code(target), _ptr(target), float(T), _ptr(q), _ptr(q_row), _ptr(draft_token),
            _ptr(next_token), _ptr(next_sibling), _ptr(coins), _ptr(u_final), _ptr(budget), int(eos_id),
            _ptr(out["committed"]), _ptr(out["num_committed"]), _ptr(out["accept_length"]), _ptr(out["accept_path"]),
            _ptr(out["next_root"]), _ptr(out.get("walk_info")), _ptr(stats), _ptr(ws), ws.numel())
    flags = (WITHOUT_REPLACEMENT if without_replacement else 0) | (CHAIN if chain else 0)
    if flags:
        _call("spec_verify_sample_flags", *args, flags, _stream())
    else:
        _call("spec_verify_sample", *args, _stream())
    return out


def spec_verify_sample_qlogits(target, T, q_logits, q_stats, T_q, draft_token, next_token, next_sibling, coins,
                               u_final, q_row=None, budget=None, eos_id=-1, out=None, ws=None, stats=None,
                               without_replacement=False, chain=False, id_map=None):
    """Stochastic verify with q given as draft-logit rows [rows, V] plus their
    (max, normaliser) [rows, 2] from spec_softmax_topk(row_stats=...).
    id_map = (table, fallback_id) (chains only): the committed ids are also
    mapped through table into out["committed_mapped"] in the same launch
    (spec_verify_sample_qlogits_mapped; TLI's target-to-draft map)."""
    _dev(target, name="target")
    B, N, V = target.shape
    _dev(q_logits, name="q_logits")
    if q_logits.shape[-1] != V:
        raise ValueError("q_logits rows must have length V")
    _dev(q_stats, torch.float32, "q_stats")
    for name, t in (("draft_token", draft_token), ("next_token", next_token), ("next_sibling", next_sibling)):
        _dev(t, torch.int32, name)
    _dev(q_row, torch.int32, "q_row")
    _dev(coins, torch.float32, "coins")
    _dev(u_final, torch.float32, "u_final")
    _dev(budget, torch.int32, "budget")
    _dev(stats, torch.int32, "stats")
    out = _verify_outputs(B, N, target.device, out)
    ws = _workspace(B, N, target.device, ws)
    args = (B, N, V, _logit_code(target), _ptr(target), float(T), _ptr(q_logits), _logit_code(q_logits),
            _ptr(q_stats), float(T_q), _ptr(q_row), _ptr(draft_token), _ptr(next_token), _ptr(next_sibling),
            _ptr(coins), _ptr(u_final), _ptr(budget), int(eos_id), _ptr(out["committed"]),
            _ptr(out["num_committed"]), _ptr(out["accept_length"]), _ptr(out["accept_path"]), _ptr(out["next_root"]),
            _ptr(out.get("walk_info")), _ptr(stats), _ptr(ws), ws.numel())
    flags = (WITHOUT_REPLACEMENT if without_replacement else 0) | (CHAIN if chain else 0)
    if id_map is not None:
        table, fallback = id_map
        _dev(table, torch.int32, "id_map table")
        if "committed_mapped" not in out:
            out["committed_mapped"] = torch.empty((B, N), dtype=torch.int32, device=target.device)
        m = SpecIdMap(ctypes.c_void_p(table.data_ptr()), table.numel(), int(fallback),
                      ctypes.c_void_p(out["committed_mapped"].data_ptr()))
        _call("spec_verify_sample_qlogits_mapped", *args, flags, ctypes.byref(m), _stream())
    elif flags:
        _call("spec_verify_sample_qlogits_flags", *args, flags, _stream())
    else:
        _call("spec_verify_sample_qlogits", *args, _stream())
    return out


class SpecIdMap(ctypes.Structure):
    """spec_id_map_t"""
    _fields_ = [("table", ctypes.c_void_p), ("table_len", ctypes.c_int64), ("fallback_id", ctypes.c_int32),
                ("out", ctypes.c_void_p)]


def spec_filter_logits(logits, T, top_k=0, top_p=1.0, stats=None):
    """Target-side top-k / top-p filtering of logit rows [..., V], in place:
    logits outside the kept set become -inf (spec_filter_logits).  Returns
    the same tensor."""
    _dev(logits, name="logits")
    _dev(stats, torch.int32, "stats")
    V = logits.shape[-1]
    R = logits.numel() // V
    _call("spec_filter_logits", _ptr(logits), _logit_code(logits), R, V, float(T), int(top_k), float(top_p),
          _ptr(stats), _stream())
    return logits


# -------------------------------------------------------------- compaction

def spec_compact_freed_capacity(B, N, page_size):
    return int(lib().spec_compact_freed_capacity(int(B), int(N), int(page_size)))


def spec_compact_slots(seq_lens, accept_path, accept_length, req_to_token, page_size, kv_pool=None, out=None,
                       stats=None):
    """req_to_token [B, max_ctx] int32 and kv_pool [slots, bytes] uint8 are updated in place."""
    _dev(seq_lens, torch.int32, "seq_lens")
    _dev(accept_path, torch.int32, "accept_path")
    _dev(accept_length, torch.int32, "accept_length")
    _dev(req_to_token, torch.int32, "req_to_token")
    _dev(kv_pool, torch.uint8, "kv_pool")
    _dev(stats, torch.int32, "stats")
    B, N = accept_path.shape
    max_ctx = req_to_token.shape[1]
    cap = spec_compact_freed_capacity(B, N, page_size)
    dev = accept_path.device
    if out is None:
        out = {
            "move_src": torch.empty((B, N), dtype=torch.int32, device=dev),
            "move_dst": torch.empty((B, N), dtype=torch.int32, device=dev),
            "num_moves": torch.empty((B,), dtype=torch.int32, device=dev),
            "freed": torch.empty((max(cap, 1),), dtype=torch.int32, device=dev),
            "num_freed": torch.empty((1,), dtype=torch.int32, device=dev),
            "new_kv_len": torch.empty((B,), dtype=torch.int32, device=dev),
        }
    slots = kv_pool.shape[0] if kv_pool is not None else 0
    bps = kv_pool.shape[1] if kv_pool is not None else 0
    _call("spec_compact_slots", B, N, int(page_size), _ptr(seq_lens), _ptr(accept_path), _ptr(accept_length),
          _ptr(req_to_token), max_ctx, _ptr(out["move_src"]), _ptr(out["move_dst"]), _ptr(out["num_moves"]),
          _ptr(out["freed"]), out["freed"].numel(), _ptr(out["num_freed"]), _ptr(out["new_kv_len"]), _ptr(kv_pool),
          slots, bps, _ptr(stats), _stream())
    return out


# --------------------------------------------------------------------- TLI

def spec_wait_probe(flag, limit_cycles, stats=None, seen=None):
    """Runs the verify's bounded flag wait once (see include/specdec.h);
    returns the int32 device tensor `seen` (1: the flag was set)."""
    _dev(flag, torch.int32, "flag")
    _dev(stats, torch.int32, "stats")
    seen = _out(seen, (1,), torch.int32, flag, "seen")
    _call("spec_wait_probe", _ptr(flag), int(limit_cycles), _ptr(stats), _ptr(seen), _stream())
    return seen


def spec_debug_bounds(reset=False) -> int:
    """Out-of-range indices the debug build's kernels have met since the
    last reset (synchronises the device); SpecError (unsupported) from the
    release library."""
    n = ctypes.c_int64(0)
    _call("spec_debug_bounds", ctypes.byref(n), 1 if reset else 0)
    return int(n.value)


def tli_plan_bytes(Vd, Vt) -> int:
    n = lib().tli_plan_bytes(int(Vd), int(Vt))
    if n < 0:
        raise SpecError("tli_plan_bytes", -2)
    return n


def tli_plan_build(d2t, t2d, plan=None):
    """The map plan of (d2t, t2d) as a uint8 device tensor (see
    tli_plan_build in include/specdec.h)."""
    _dev(d2t, torch.int32, "d2t")
    _dev(t2d, torch.int32, "t2d")
    n = tli_plan_bytes(d2t.numel(), t2d.numel())
    if plan is None:
        plan = torch.empty(n, dtype=torch.uint8, device=d2t.device)
    elif plan.numel() < n or plan.dtype != torch.uint8 or not plan.is_cuda or plan.data_ptr() % 16:
        raise ValueError(f"plan must be a 16-byte aligned uint8 device tensor of >= {n} bytes")
    _call("tli_plan_build", d2t.numel(), t2d.numel(), _ptr(d2t), _ptr(t2d), _ptr(plan), _stream())
    return plan


def tli_constrain_map(draft_logits, d2t, T, t2d=None, want_q=False, top1_draft=None, top1_target=None,
                      top1_p=None, q_target=None, stats=None, plan=None, expand=None):
    _dev(draft_logits, name="draft_logits")
    _dev(d2t, torch.int32, "d2t")
    _dev(t2d, torch.int32, "t2d")
    Vd = draft_logits.shape[-1]
    R = draft_logits.numel() // Vd
    if d2t.numel() != Vd:
        raise ValueError("d2t must have V_d entries")
    Vt = t2d.numel() if t2d is not None else 1
    top1_draft = _out(top1_draft, (R,), torch.int32, draft_logits, "top1_draft")
    top1_target = _out(top1_target, (R,), torch.int32, draft_logits, "top1_target")
    top1_p = _out(top1_p, (R,), torch.float32, draft_logits, "top1_p")
    if want_q and q_target is None:
        q_target = torch.empty((R, Vt), dtype=torch.float32, device=draft_logits.device)
    _dev(q_target, torch.float32, "q_target")
    _dev(stats, torch.int32, "stats")
    if plan is not None:
        if plan.dtype != torch.uint8 or not plan.is_cuda or plan.numel() < tli_plan_bytes(Vd, Vt):
            raise ValueError("plan must come from tli_plan_build for these vocabulary sizes")
        if expand is not None:
            _call("tli_constrain_map_planned_expand", R, Vd, Vt, _ptr(draft_logits), _logit_code(draft_logits),
                  _ptr(d2t), _ptr(t2d), _ptr(plan), float(T), _ptr(top1_draft), _ptr(top1_target), _ptr(top1_p),
                  _ptr(q_target), _ptr(stats), _expand(expand), _stream())
        else:
            _call("tli_constrain_map_planned", R, Vd, Vt, _ptr(draft_logits), _logit_code(draft_logits),
                  _ptr(d2t), _ptr(t2d), _ptr(plan), float(T), _ptr(top1_draft), _ptr(top1_target), _ptr(top1_p),
                  _ptr(q_target), _ptr(stats), _stream())
    else:
        if expand is not None:
            raise ValueError("a fused expansion needs the map plan")
        _call("tli_constrain_map", R, Vd, Vt, _ptr(draft_logits), _logit_code(draft_logits), _ptr(d2t),
              _ptr(t2d), float(T), _ptr(top1_draft), _ptr(top1_target), _ptr(top1_p), _ptr(q_target),
              _ptr(stats), _stream())
    return top1_draft, top1_target, top1_p, q_target


def tli_constrain_map_qlogits(draft_logits, d2t, t2d, T, plan=None, top1_draft=None, top1_target=None,
                              top1_p=None, q_logits=None, q_stats=None, stats=None, expand=None):
    """tli_constrain_map with q in logit form: q_logits [R, V_t] (the draft
    dtype, each target id's partner logit, -inf without one) and q_stats
    [R, 2] (max, normaliser) for spec_verify_sample_qlogits with T_q = T."""
    _dev(draft_logits, name="draft_logits")
    _dev(d2t, torch.int32, "d2t")
    _dev(t2d, torch.int32, "t2d")
    if t2d is None:
        raise ValueError("t2d is required")
    Vd = draft_logits.shape[-1]
    R = draft_logits.numel() // Vd
    if d2t.numel() != Vd:
        raise ValueError("d2t must have V_d entries")
    Vt = t2d.numel()
    top1_draft = _out(top1_draft, (R,), torch.int32, draft_logits, "top1_draft")
    top1_target = _out(top1_target, (R,), torch.int32, draft_logits, "top1_target")
    top1_p = _out(top1_p, (R,), torch.float32, draft_logits, "top1_p")
    q_logits = _out(q_logits, (R, Vt), draft_logits.dtype, draft_logits, "q_logits")
    q_stats = _out(q_stats, (R, 2), torch.float32, draft_logits, "q_stats")
    _dev(stats, torch.int32, "stats")
    if plan is not None and (plan.dtype != torch.uint8 or not plan.is_cuda or plan.numel() < tli_plan_bytes(Vd, Vt)):
        raise ValueError("plan must come from tli_plan_build for these vocabulary sizes")
    _call("tli_constrain_map_qlogits", R, Vd, Vt, _ptr(draft_logits), _logit_code(draft_logits), _ptr(d2t), _ptr(t2d),
          _ptr(plan), float(T), _ptr(top1_draft), _ptr(top1_target), _ptr(top1_p), _ptr(q_logits), _ptr(q_stats),
          _ptr(stats), _expand(expand) if expand is not None else None, _stream())
    return top1_draft, top1_target, top1_p, q_logits, q_stats


def tli_map_ids(ids, table, fallback_id, out=None):
    _dev(ids, torch.int32, "ids")
    _dev(table, torch.int32, "table")
    out = _out(out, ids.shape, torch.int32, ids, "out")
    _call("tli_map_ids", _ptr(ids), _ptr(out), ids.numel(), _ptr(table), table.numel(), int(fallback_id), _stream())
    return out


def tli_pruned_head(hidden, weight, ids, d2t, T, want_logits=False, out=None, ws=None, stats=None):
    """Pruned draft LM head on the tensor cores: hidden [M, H] and weight
    [K, H] bf16 (row k belongs to draft id ids[k]), d2t [V_d].  Returns a
    dict with top1_draft, top1_target, top1_rank [M] int32, top1_p [M],
    row_stats [M, 2] and, with want_logits, logits [M, K] fp32."""
    _dev(hidden, torch.bfloat16, "hidden")
    _dev(weight, torch.bfloat16, "weight")
    _dev(ids, torch.int32, "ids")
    _dev(d2t, torch.int32, "d2t")
    _dev(stats, torch.int32, "stats")
    M, H = hidden.shape
    K = weight.shape[0]
    if weight.shape[1] != H or ids.numel() != K:
        raise ValueError("weight must be [K, H] and ids [K]")
    dev = hidden.device
    if out is None:
        out = {"top1_draft": torch.empty(M, dtype=torch.int32, device=dev),
               "top1_target": torch.empty(M, dtype=torch.int32, device=dev),
               "top1_rank": torch.empty(M, dtype=torch.int32, device=dev),
               "top1_p": torch.empty(M, dtype=torch.float32, device=dev),
               "row_stats": torch.empty((M, 2), dtype=torch.float32, device=dev)}
        if want_logits:
            out["logits"] = torch.empty((M, K), dtype=torch.float32, device=dev)
    need = int(lib().tli_pruned_head_ws_size(M, K))
    if ws is None:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _call("tli_pruned_head", M, H, K, _ptr(hidden), _ptr(weight), _ptr(ids), _ptr(d2t), d2t.numel(), float(T),
          _ptr(out["top1_draft"]), _ptr(out["top1_target"]), _ptr(out["top1_p"]), _ptr(out.get("top1_rank")),
          _ptr(out.get("row_stats")), _ptr(out.get("logits")), _ptr(stats), _ptr(ws), ws.numel(), _stream())
    return out


def tli_check_config(topk, num_steps, num_draft_tokens) -> bool:
    return lib().tli_check_config(int(topk), int(num_steps), int(num_draft_tokens)) == 0
