"""fp64 CPU oracle for the speculative-decoding verify step.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check of
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this
package.  The product library never calls it and shares no source with it.

The arithmetic lives in ``sd_oracle.c`` (plain C, double precision, written
step by step from the pages; see the header of that file for the passages
each function follows).  This module only compiles it with gcc and marshals
numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sd_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1
ST_BAD_TOKEN, ST_NONFINITE, ST_BAD_PARENT, ST_ZERO_MASS = 1, 2, 4, 8


def build(force: bool = False) -> str:
    """Compile sd_oracle.c into liboracle.so (gcc, -O2, no -march flags)."""
    stale = (not os.path.exists(_LIB)) or (
        os.path.getmtime(_LIB) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB + ".%d.tmp" % os.getpid()
        subprocess.check_call(
            ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-Wall",
             "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _bind(path):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    D = ctypes.c_double
    lib.orc_verify_linear.argtypes = [P, P, I, P, P, I, I, I, D,
                                      P, P, P, P, P, P, P, P, P, P, P, P]
    lib.orc_verify_kcand.argtypes = [P, P, I, P, P, I, I, I, I, D,
                                     P, P, P, P, P, P, P, P, P, P, P, P]
    lib.orc_verify_tree.argtypes = [P, P, I, P, P, P, I, I, I, D,
                                    P, P, P, P, P, P, P, P, P, P, P]
    lib.orc_verify_tree_det.argtypes = [P, I, P, P, P, I, I, I, D,
                                        P, P, P, P, P, P, P, P, P, P, P]
    lib.orc_kcand_trie.argtypes = [P, P, I, I, I, P, P, P, P, P, P, P]
    lib.orc_presto_expand.argtypes = [P, P, I, ctypes.c_longlong, I, I, I,
                                      D, D, I, I, P, P, P, P, P, P, P, P]
    lib.orc_branch_fork.argtypes = [P, I, P, I, I, D, I, P, P, P, P]
    lib.orc_fanout_schedule.argtypes = [I, I, D, D, P]
    lib.orc_fanout_topk.argtypes = [P, I, I, I, I, P, P, P, P]
    lib.orc_fanout_hits.argtypes = [P, P, P, P, I, I, P]
    lib.orc_verify_linear_filtered.argtypes = [P, P, I, P, P, I, I, I, D, I,
                                               D, P, P, P, P, P, P, P, P, P,
                                               P, P, P, P, P]
    for f in (lib.orc_verify_linear, lib.orc_verify_kcand,
              lib.orc_verify_tree, lib.orc_fanout_schedule,
              lib.orc_fanout_topk):
        f.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(_LIB)
    return _lib


class swapped_library:
    """Context manager for the mutation tests: route every call to another
    build of the oracle (a copy of sd_oracle.c with a planted mistake)."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        global _lib
        _load()
        self._saved = _lib
        _lib = _bind(self.path)
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def _logits(a):
    """Return (contiguous array, dtype code).  bf16 logits travel as their
    raw uint16 bit patterns; fp32 as float32."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return a, BF16
    if a.dtype == np.float32:
        return a, F32
    raise TypeError("logits must be float32 or raw bf16 bits (uint16)")


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _margins(B):
    return {"margin_acc": np.empty(B, np.float64),
            "margin_cdf": np.empty(B, np.float64),
            "cdf_lo": np.empty(B, np.int32),
            "cdf_hi": np.empty(B, np.int32),
            "acc_tests": np.empty(B, np.int32),
            "acc_flagged": np.empty(B, np.int32)}


def _margin_ptrs(m):
    return (_ptr(m["margin_acc"]), _ptr(m["margin_cdf"]), _ptr(m["cdf_lo"]),
            _ptr(m["cdf_hi"]), _ptr(m["acc_tests"]), _ptr(m["acc_flagged"]))


def _finish(out, m):
    out.update(m)
    out["margin"] = np.minimum(m["margin_acc"], m["margin_cdf"])
    return out


def verify_linear(target, draft, tokens, uniforms, T, want_resid=False):
    """Linear verify of B sequences.

    target [B, gamma+1, V], draft [B, gamma, V] (float32, or uint16 bf16 bits;
    draft may be None when T == 0), tokens [B, gamma] int32, uniforms
    [B, gamma+1] float32.  Returns a dict of numpy arrays: n, tokens, prob,
    accept, margin, status and (when asked) resid [B, V].
    """
    target, dt = _logits(target)
    B, G1, V = target.shape
    gamma = G1 - 1
    if draft is None:
        if T != 0:
            raise ValueError("draft logits are required when T > 0")
        draft_p = None
    else:
        draft, dt2 = _logits(draft)
        if dt2 != dt or draft.shape != (B, gamma, V):
            raise ValueError("draft must match target in dtype and shape")
        draft_p = _ptr(draft)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, gamma)
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B, G1)
    out = {
        "n": np.empty(B, np.int32),
        "tokens": np.empty((B, G1), np.int32),
        "prob": np.empty(B, np.float64),
        "accept": np.empty((B, max(gamma, 1)), np.float64),
        "status": np.empty(B, np.int32),
    }
    m = _margins(B)
    resid = np.empty((B, V), np.float64) if want_resid else None
    rc = _load().orc_verify_linear(
        _ptr(target), draft_p, dt, _ptr(tokens), _ptr(uniforms), B, gamma, V,
        float(T), _ptr(out["n"]), _ptr(out["tokens"]), _ptr(out["prob"]),
        _ptr(out["accept"]), *_margin_ptrs(m), _ptr(resid),
        _ptr(out["status"]))
    if rc:
        raise MemoryError("oracle allocation failed")
    out["accept"] = out["accept"][:, :gamma]
    if want_resid:
        out["resid"] = resid
    return _finish(out, m)


def verify_linear_filtered(target, draft, tokens, uniforms, T, top_k,
                           top_p=1.0, keep_forced=None, want_keep=False):
    """Linear verify with top_k / top_p filtered sampling applied to p and q
    before the ratio (same shapes as verify_linear; top_k >= V keeps every
    token).  Returns n, tokens, prob, the margins and status.

    want_keep: also return keep, keep_lo, keep_hi [B, 2 gamma + 1] (slot i
    for target row i, gamma + 1 + i for draft row i; -1 for rows not read):
    the kept count of each row and the range of counts whose nucleus cut
    lies within FLAG_MARGIN of top_p; margin_acc then covers the accept
    tests only.  Otherwise margin_acc also covers the nucleus cuts.
    keep_forced [B, 2 gamma + 1] (entries >= 1): keep that many tokens of
    the row (at most top_k) instead of the nucleus's count."""
    target, dt = _logits(target)
    B, G1, V = target.shape
    gamma = G1 - 1
    if draft is None:
        if T != 0:
            raise ValueError("draft logits are required when T > 0")
        draft_p = None
    else:
        draft, dt2 = _logits(draft)
        if dt2 != dt or draft.shape != (B, gamma, V):
            raise ValueError("draft must match target in dtype and shape")
        draft_p = _ptr(draft)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, gamma)
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B, G1)
    NS = 2 * gamma + 1
    out = {
        "n": np.empty(B, np.int32),
        "tokens": np.empty((B, G1), np.int32),
        "prob": np.empty(B, np.float64),
        "status": np.empty(B, np.int32),
    }
    kf = None if keep_forced is None else np.ascontiguousarray(
        keep_forced, np.int32).reshape(B, NS)
    kp = {k: np.empty((B, NS), np.int32) for k in ("keep", "keep_lo",
                                                   "keep_hi")} \
        if want_keep else {}
    m = _margins(B)
    rc = _load().orc_verify_linear_filtered(
        _ptr(target), draft_p, dt, _ptr(tokens), _ptr(uniforms), B, gamma, V,
        float(T), int(top_k), float(top_p), _ptr(out["n"]),
        _ptr(out["tokens"]), _ptr(out["prob"]), *_margin_ptrs(m), _ptr(kf),
        _ptr(kp.get("keep")), _ptr(kp.get("keep_lo")),
        _ptr(kp.get("keep_hi")), _ptr(out["status"]))
    if rc:
        raise MemoryError("oracle allocation failed")
    out.update(kp)
    return _finish(out, m)


def verify_kcand(target, draft, tokens, uniforms, T):
    """K-candidate verify with longest-streak self-selection.

    target [B, K, gamma+1, V], draft [B, gamma, V] shared marginals, tokens
    [B, K, gamma], uniforms [B, K, gamma+1].
    """
    target, dt = _logits(target)
    B, K, G1, V = target.shape
    gamma = G1 - 1
    draft, dt2 = _logits(draft)
    if dt2 != dt or draft.shape != (B, gamma, V):
        raise ValueError("draft must be [B, gamma, V] in the target's dtype")
    tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, K, gamma)
    uniforms = np.ascontiguousarray(uniforms, np.float32).reshape(B, K, G1)
    out = {
        "n": np.empty(B, np.int32),
        "k": np.empty(B, np.int32),
        "tokens": np.empty((B, G1), np.int32),
        "n_per_cand": np.empty((B, K), np.int32),
        "prob": np.empty(B, np.float64),
        "status": np.empty(B, np.int32),
    }
    m = _margins(B)
    rc = _load().orc_verify_kcand(
        _ptr(target), _ptr(draft), dt, _ptr(tokens), _ptr(uniforms), B, K,
        gamma, V, float(T), _ptr(out["n"]), _ptr(out["k"]),
        _ptr(out["tokens"]), _ptr(out["n_per_cand"]), _ptr(out["prob"]),
        *_margin_ptrs(m), _ptr(out["status"]))
    if rc:
        raise MemoryError("oracle allocation failed")
    return _finish(out, m)


def verify_tree(target, draft, parent, node_tokens, uniforms, T):
    """Token-tree verify with sequential sibling rejection.

    target, draft [B, N, V]; parent, node_tokens [B, N] int32; uniforms
    [B, N] float32 (slot 0 is the final draw).
    """
    target, dt = _logits(target)
    B, N, V = target.shape
    draft, dt2 = _logits(draft)
    if dt2 != dt or draft.shape != (B, N, V):
        raise ValueError("draft must match target in dtype and shape")
    parent = np.ascontiguousarray(parent, np.int32).reshape(B, N)
    node_tokens = np.ascontiguousarray(node_tokens, np.int32).reshape(B, N)
    uniforms = np.ascontiguousarray(uniforms, np.float32).reshape(B, N)
    out = {
        "n": np.empty(B, np.int32),
        "tokens": np.empty((B, N), np.int32),
        "nodes": np.empty((B, N), np.int32),
        "prob": np.empty(B, np.float64),
        "status": np.empty(B, np.int32),
    }
    m = _margins(B)
    rc = _load().orc_verify_tree(
        _ptr(target), _ptr(draft), dt, _ptr(parent), _ptr(node_tokens),
        _ptr(uniforms), B, N, V, float(T), _ptr(out["n"]),
        _ptr(out["tokens"]), _ptr(out["nodes"]), _ptr(out["prob"]),
        *_margin_ptrs(m), _ptr(out["status"]))
    if rc:
        raise MemoryError("oracle allocation failed")
    return _finish(out, m)


def verify_tree_det(target, parent, node_tokens, uniforms, T):
    """Token-tree verify with deterministic drafts: child v is accepted with
    the current p(t_v); a rejected token is removed from p, which is
    renormalised.  target [B, N, V]; the rest as verify_tree."""
    target, dt = _logits(target)
    B, N, V = target.shape
    parent = np.ascontiguousarray(parent, np.int32).reshape(B, N)
    node_tokens = np.ascontiguousarray(node_tokens, np.int32).reshape(B, N)
    uniforms = np.ascontiguousarray(uniforms, np.float32).reshape(B, N)
    out = {
        "n": np.empty(B, np.int32),
        "tokens": np.empty((B, N), np.int32),
        "nodes": np.empty((B, N), np.int32),
        "prob": np.empty(B, np.float64),
        "status": np.empty(B, np.int32),
    }
    m = _margins(B)
    rc = _load().orc_verify_tree_det(
        _ptr(target), dt, _ptr(parent), _ptr(node_tokens), _ptr(uniforms),
        B, N, V, float(T), _ptr(out["n"]), _ptr(out["tokens"]),
        _ptr(out["nodes"]), _ptr(out["prob"]), *_margin_ptrs(m),
        _ptr(out["status"]))
    if rc:
        raise MemoryError("oracle allocation failed")
    return _finish(out, m)


def kcand_trie(tokens, uniforms):
    """K candidates as one token tree (orc_kcand_trie).  tokens [B, K,
    gamma] int32, uniforms [B, K, gamma+1] float32.  Returns the tree's
    parent, node_tokens, uniforms, target_row, draft_row, node_cand and
    is_dup, each [B, 1 + K gamma]."""
    tokens = np.ascontiguousarray(tokens, np.int32)
    B, K, gamma = tokens.shape
    uniforms = np.ascontiguousarray(uniforms, np.float32).reshape(
        B, K, gamma + 1)
    N = 1 + K * gamma
    out = {k: np.empty((B, N), np.int32) for k in
           ("parent", "node_tokens", "target_row", "draft_row", "node_cand",
            "is_dup")}
    out["uniforms"] = np.empty((B, N), np.float32)
    if _load().orc_kcand_trie(
            _ptr(tokens), _ptr(uniforms), B, K, gamma, _ptr(out["parent"]),
            _ptr(out["node_tokens"]), _ptr(out["uniforms"]),
            _ptr(out["target_row"]), _ptr(out["draft_row"]),
            _ptr(out["node_cand"]), _ptr(out["is_dup"])):
        raise MemoryError("oracle allocation failed")
    return out


def verify_kcand_trie(target, draft, tokens, uniforms, T):
    """K candidates verified as one token tree: the tree of kcand_trie with
    node u's target row target[b].reshape(K (gamma+1), V)[target_row] and
    draft row draft[b][draft_row] (zeros for none), through verify_tree.
    target [B, K, gamma+1, V], draft [B, gamma, V] (None when T == 0).
    Returns verify_tree's outputs, tokens cut to [B, gamma+1], and k:
    node_cand of the last accepted node (0 when none was accepted)."""
    target, dt = _logits(target)
    B, K, G1, V = target.shape
    gamma = G1 - 1
    tr = kcand_trie(tokens, uniforms)
    N = 1 + K * gamma
    rows_b = np.arange(B)[:, None]
    tt = np.ascontiguousarray(
        target.reshape(B, K * G1, V)[rows_b, tr["target_row"]])
    dd = np.zeros((B, N, V), target.dtype)
    if draft is not None and gamma > 0:
        draft, dt2 = _logits(draft)
        if dt2 != dt or draft.shape != (B, gamma, V):
            raise ValueError("draft must be [B, gamma, V] of target's dtype")
        has = tr["draft_row"] >= 0
        dd[has] = draft[rows_b, np.maximum(tr["draft_row"], 0)][has]
    o = verify_tree(tt, dd, tr["parent"], tr["node_tokens"], tr["uniforms"],
                    T)
    o["tokens"] = np.ascontiguousarray(o["tokens"][:, :G1])
    n = o["n"]
    last = np.where(n > 0, o["nodes"][np.arange(B), np.maximum(n - 1, 0)], 0)
    o["k"] = np.where(n >= 0, tr["node_cand"][np.arange(B), last],
                          -1).astype(np.int32)
    o["trie"] = tr
    return o


class PrestoTree:
    """Host state of PRESTO trees under construction (the oracle's copy):
    node arrays [B, budget] and the frontier [B, W].  Node 0 is the root
    (parent -1, token -1, score 0) and the only frontier path."""

    def __init__(self, B, W, budget):
        self.B, self.W, self.budget = B, W, budget
        self.n_nodes = np.ones(B, np.int32)
        self.parent = np.full((B, budget), -1, np.int32)
        self.node_tokens = np.full((B, budget), -1, np.int32)
        self.node_score = np.zeros((B, budget), np.float64)
        self.frontier_node = np.full((B, W), -1, np.int32)
        self.frontier_node[:, 0] = 0
        self.frontier_score = np.zeros((B, W), np.float64)
        self.node_depth = np.zeros((B, budget), np.int32)


def presto_expand(tree, q_logits, log_rho, T, lam, b_top):
    """One depth of PRESTO's beam construction on `tree` (a PrestoTree,
    updated in place).  q_logits [B, V] the drafter's marginal at this
    depth; log_rho [B, W, V] the frontier paths' prefix signals.  Returns
    (margin [B], status [B])."""
    q_logits, dt = _logits(q_logits)
    B, V = q_logits.shape
    log_rho, dt2 = _logits(log_rho)
    if dt2 != dt or log_rho.shape != (B, tree.W, V):
        raise ValueError("log_rho must be [B, W, V] of q's dtype")
    margin = np.empty(B, np.float64)
    status = np.empty(B, np.int32)
    n_before = tree.n_nodes.copy()
    if _load().orc_presto_expand(
            _ptr(q_logits), _ptr(log_rho), dt, V, B, tree.W, V, float(T),
            float(lam), int(b_top), tree.budget, _ptr(tree.n_nodes),
            _ptr(tree.parent), _ptr(tree.node_tokens),
            _ptr(tree.node_score), _ptr(tree.frontier_node),
            _ptr(tree.frontier_score), _ptr(margin), _ptr(status)):
        raise ValueError("bad PRESTO arguments")
    for b in range(B):
        for v in range(max(n_before[b], 0), max(tree.n_nodes[b], 0)):
            tree.node_depth[b, v] = tree.node_depth[b, tree.parent[b, v]] + 1
    return margin, status


def branch_fork(draft, x_b, T, k_max):
    """SpecBranch fork: k = max(1, floor(k_max (1 - q(x_b)))) (capped at V)
    and the top-k tokens of each draft row.  draft [B, V]; x_b [B].
    Returns k [B], tokens [B, k_max] (-1 padded), margin, status."""
    draft, dt = _logits(draft)
    B, V = draft.shape
    x_b = np.ascontiguousarray(x_b, np.int32).reshape(B)
    out = {"k": np.empty(B, np.int32),
           "tokens": np.empty((B, k_max), np.int32),
           "margin": np.empty(B, np.float64),
           "status": np.empty(B, np.int32)}
    if _load().orc_branch_fork(_ptr(draft), dt, _ptr(x_b), B, V, float(T),
                               int(k_max), _ptr(out["k"]),
                               _ptr(out["tokens"]), _ptr(out["margin"]),
                               _ptr(out["status"])):
        raise ValueError("bad fork arguments")
    return out


def fanout_schedule(K, budget, a, r):
    """Geometric fan-out F[0..K] with sum == budget (Theorem 12 + largest
    remainder)."""
    F = np.zeros(K + 1, np.int32)
    if _load().orc_fanout_schedule(int(K), int(budget), float(a), float(r),
                                   _ptr(F)):
        raise ValueError("bad fan-out arguments")
    return F


def fanout_topk(draft, F):
    """Top-F_k tokens of lookahead row k; draft [B, K+1, V]."""
    draft, dt = _logits(draft)
    B, K1, V = draft.shape
    F = np.ascontiguousarray(F, np.int32)
    if F.shape != (K1,):
        raise ValueError("F must have K+1 entries")
    total = int(F.sum())
    out = {
        "tokens": np.empty((B, total), np.int32),
        "logit": np.empty((B, total), np.float64),
        "status": np.empty(B, np.int32),
    }
    rc = _load().orc_fanout_topk(_ptr(draft), dt, B, K1 - 1, V, _ptr(F),
                                 _ptr(out["tokens"]), _ptr(out["logit"]),
                                 _ptr(out["status"]))
    if rc:
        raise MemoryError("oracle allocation failed")
    return out


def fanout_hits(n, tokens, fan_tokens, F):
    """Saguaro cache hit of each sequence's outcome (n accepted, then the
    token tokens[b, n]): 1 if that token is among the F[n] fan-out tokens of
    position n, 0 if not, -1 where n < 0.  tokens [B, K+1], fan_tokens
    [B, sum F]."""
    n = np.ascontiguousarray(n, np.int32)
    tokens = np.ascontiguousarray(tokens, np.int32)
    fan_tokens = np.ascontiguousarray(fan_tokens, np.int32)
    F = np.ascontiguousarray(F, np.int32)
    B, K1 = tokens.shape
    if F.shape != (K1,) or n.shape != (B,) or \
            fan_tokens.shape != (B, int(F.sum())):
        raise ValueError("shapes: n [B], tokens [B, K+1], F [K+1], "
                         "fan_tokens [B, sum F]")
    hit = np.empty(B, np.int32)
    _load().orc_fanout_hits(_ptr(n), _ptr(tokens), _ptr(fan_tokens), _ptr(F),
                            B, K1 - 1, _ptr(hit))
    return hit


FLAG_MARGIN = 1e-5
"""A draw whose margin is below this is 'flagged': a correct fp32
implementation may land on the other side of the threshold there (for an
inverse-CDF draw it may then return any token in [cdf_lo, cdf_hi]).
Every verify result carries, per sequence, acc_tests (accept tests made,
T > 0) and acc_flagged (those whose |r - p/q| is below this margin)."""
