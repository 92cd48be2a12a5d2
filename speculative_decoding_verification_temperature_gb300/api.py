"""Thin torch binding over libsdverify.so (the C ABI of include/sd_verify.h).

Only argument marshalling happens here: shapes and dtypes are checked, raw
device pointers and the current CUDA stream are passed through ctypes, and
outputs are allocated with torch.  Every step of the verify path runs in the
library's CUDA kernels; there is no other implementation behind these
functions, and they raise if the library cannot be loaded.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

SD_OK, SD_ERR_INVALID_ARG, SD_ERR_UNSUPPORTED, SD_ERR_CUDA = 0, 1, 2, 3
SD_F32, SD_BF16 = 0, 1
DEV_BAD_TOKEN, DEV_NONFINITE, DEV_BAD_PARENT, DEV_ZERO_MASS = 1, 2, 4, 8
DEV_TIMEOUT = 16

_lock = threading.Lock()
_lib = None


class SdError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__("sd_verify error %d: %s" % (code, msg))
        self.code = code


def lib() -> ctypes.CDLL:
    """Load libsdverify.so (compiling it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            # SDV_LIB selects another build of the same library
            path = os.environ.get("SDV_LIB") or _build.build()
            if not os.path.exists(path):
                raise RuntimeError("libsdverify.so is missing: run "
                                   "__graft_entry__.build()")
            L = ctypes.CDLL(path)
            _declare(L)
            _lib = L
    return _lib


def _declare(L):
    P, I, F, D, Z = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float,
                     ctypes.c_double, ctypes.c_size_t)
    sig = {
        "sd_version": ([], ctypes.c_char_p),
        "sd_last_error": ([], ctypes.c_char_p),
        "sd_verify_linear_workspace": ([I, I, I, I], Z),
        "sd_verify_linear": ([P, P, I, P, P, I, I, I, F, P, P, P, P, P, P, P,
                              Z, P], I),
        "sd_verify_kcand_workspace": ([I, I, I, I, I], Z),
        "sd_verify_kcand": ([P, P, I, P, P, I, I, I, I, F, P, P, P, P, P, P,
                             P, Z, P], I),
        "sd_verify_kcand_trie_workspace": ([I, I, I, I, I], Z),
        "sd_verify_kcand_trie": ([P, P, I, P, P, I, I, I, I, F, P, P, P, P,
                                  P, P, Z, P], I),
        "sd_presto_init": ([I, I, I, P, P, P, P, P, P, P], I),
        "sd_presto_expand_workspace": ([I, I, I, I, I], Z),
        "sd_presto_expand": ([P, ctypes.c_longlong, P, I, I, I, I, F, F, I,
                              I, P, P, P, P, P, P, P, P, Z, P], I),
        "sd_branch_fork_workspace": ([I, I, I, I], Z),
        "sd_branch_fork": ([P, I, P, I, I, F, I, P, P, P, P, Z, P], I),
        "sd_verify_tree_workspace": ([I, I, I, I], Z),
        "sd_verify_tree": ([P, P, I, P, P, P, I, I, I, F, P, P, P, P, P, P,
                            Z, P], I),
        "sd_verify_tree_det_workspace": ([I, I, I, I], Z),
        "sd_verify_tree_det": ([P, I, P, P, P, I, I, I, F, P, P, P, P, P, P,
                                Z, P], I),
        "sd_fanout_schedule": ([I, I, D, D, P], I),
        "sd_fanout_topk_workspace": ([I, I, I, I], Z),
        "sd_fanout_topk": ([P, I, I, I, I, P, P, P, P, P, Z, P], I),
        "sd_verify_linear_static": ([P, P, I, P, P, I, I, I, F, P, P, P, P,
                                     P, P, P], I),
        "sd_fanout_hits": ([P, P, P, I, I, P, P, P], I),
        "sd_verify_linear_filtered_workspace": ([I, I, I, I], Z),
        "sd_verify_linear_filtered": ([P, P, I, P, P, I, I, I, F, I, F, P, P,
                                       P, P, P, P, Z, P], I),
        "sd_verify_linear_fanout_workspace": ([I, I, I, I], Z),
        "sd_verify_linear_fanout": ([P, P, I, P, P, I, I, I, F, P, P, P, P,
                                     P, P, P, P, Z, P], I),
        "sd_tune_set": ([I, I], I),
        "sd_selftest_bounded_wait": ([I, P, P, P], I),
        "sd_tune_get": ([I], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res


def version() -> str:
    return lib().sd_version().decode()


TUNE = {"cluster": 0, "no_tma": 1, "allrows": 2, "spec": 3, "fused": 4,
        "kcand_ring": 5, "fanout_cluster": 6, "fanout_ldg": 7,
        "fanout_maxc": 8, "fanout_l2_first": 9, "helpers": 10}
"""Tuning switches of sd_tune_set, by name (see include/sd_verify.h)."""


def tune_get(name: str) -> int:
    return lib().sd_tune_get(TUNE[name])


def tune_set(name: str, value: int) -> None:
    _check(lib().sd_tune_set(TUNE[name], int(value)))


class tuned:
    """Context manager: set tuning switches (name=value) for the block and
    restore the previous values after it."""

    def __init__(self, **switches):
        self.switches = switches

    def __enter__(self):
        self.saved = {k: tune_get(k) for k in self.switches}
        for k, v in self.switches.items():
            tune_set(k, v)
        return self

    def __exit__(self, *exc):
        for k, v in self.saved.items():
            tune_set(k, v)
        return False


def _check(rc):
    if rc != SD_OK:
        raise SdError(rc, lib().sd_last_error().decode())


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SD_F32
    if t.dtype == torch.bfloat16:
        return SD_BF16
    raise TypeError("logits must be float32 or bfloat16, got %s" % t.dtype)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(t, device, name, dtype=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor (there is no CPU path)"
                         % name)
    if t.device != device:
        raise ValueError("%s must live on %s" % (name, device))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s" % (name, dtype))
    return t


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


class Workspace:
    """Per-device scratch buffer for the library's work-queue counter.
    Reused across calls on the same stream; give each concurrent stream its
    own Workspace."""

    def __init__(self):
        self._buf = {}

    def get(self, device, nbytes):
        b = self._buf.get(device)
        if b is None or b.numel() < nbytes:
            b = torch.empty(max(nbytes, 256), dtype=torch.uint8,
                            device=device)
            self._buf[device] = b
        return b


_default_ws = Workspace()


def verify_linear(target, draft, tokens, uniforms, T, *, want_accept=False,
                  want_resid=False, status=None, workspace=None, out=None):
    """Linear verify (sd_verify_linear).

    target [B, gamma+1, V], draft [B, gamma, V] (may be None when T == 0),
    both float32 or bfloat16 on one CUDA device; tokens [B, gamma] int32;
    uniforms [B, gamma+1] float32.  Returns a dict with n [B], tokens
    [B, gamma+1], prob [B] (and accept [B, gamma], resid [B, V] on request).
    ``status``: optional int32 [1] device tensor OR-ed with SD_DEV_* bits.
    """
    dev = target.device
    _dev(target, dev, "target")
    B, G1, V = target.shape
    gamma = G1 - 1
    if draft is not None:
        _dev(draft, dev, "draft", target.dtype)
        if draft.shape[0] != B or draft.shape[2] != V or \
                draft.shape[1] != gamma:
            raise ValueError("draft must be [B, gamma, V]")
    tokens = _dev(tokens, dev, "tokens", torch.int32)
    uniforms = _dev(uniforms, dev, "uniforms", torch.float32)
    if out is None:
        out = {}
    n = out.get("n")
    if n is None:
        n = torch.empty(B, dtype=torch.int32, device=dev)
    toks = out.get("tokens")
    if toks is None:
        toks = torch.empty((B, G1), dtype=torch.int32, device=dev)
    prob = out.get("prob")
    if prob is None:
        prob = torch.empty(B, dtype=torch.float32, device=dev)
    acc = torch.empty((B, max(gamma, 1)), dtype=torch.float32,
                      device=dev) if want_accept else None
    res = torch.empty((B, V), dtype=torch.float32,
                      device=dev) if want_resid else None
    L = lib()
    nbytes = L.sd_verify_linear_workspace(B, gamma, V, _dt(target))
    ws = (workspace or _default_ws).get(dev, nbytes)
    _check(L.sd_verify_linear(
        _p(target), _p(draft), _dt(target), _p(tokens), _p(uniforms), B,
        gamma, V, float(T), _p(n), _p(toks), _p(prob), _p(acc), _p(res),
        _p(status), _p(ws), ws.numel(), _stream(dev)))
    r = {"n": n, "tokens": toks, "prob": prob}
    if want_accept:
        r["accept"] = acc[:, :gamma]
    if want_resid:
        r["resid"] = res
    return r


def verify_linear_static(target, draft, tokens, uniforms, T, *,
                         want_accept=False, status=None):
    """Linear verify with the library's static per-device scratch instead of
    a workspace (sd_verify_linear_static): same arguments and results as
    verify_linear.  Calls that overlap on the GPU race on that scratch."""
    dev = target.device
    _dev(target, dev, "target")
    B, G1, V = target.shape
    gamma = G1 - 1
    if draft is not None:
        _dev(draft, dev, "draft", target.dtype)
        if tuple(draft.shape) != (B, gamma, V):
            raise ValueError("draft must be [B, gamma, V]")
    tokens = _dev(tokens, dev, "tokens", torch.int32)
    uniforms = _dev(uniforms, dev, "uniforms", torch.float32)
    n = torch.empty(B, dtype=torch.int32, device=dev)
    toks = torch.empty((B, G1), dtype=torch.int32, device=dev)
    prob = torch.empty(B, dtype=torch.float32, device=dev)
    acc = torch.empty((B, max(gamma, 1)), dtype=torch.float32,
                      device=dev) if want_accept else None
    _check(lib().sd_verify_linear_static(
        _p(target), _p(draft), _dt(target), _p(tokens), _p(uniforms), B,
        gamma, V, float(T), _p(n), _p(toks), _p(prob), _p(acc), None,
        _p(status), _stream(dev)))
    r = {"n": n, "tokens": toks, "prob": prob}
    if want_accept:
        r["accept"] = acc[:, :gamma]
    return r


def verify_linear_filtered(target, draft, tokens, uniforms, T, top_k,
                           top_p=1.0, *, want_keep=False, status=None,
                           workspace=None):
    """Linear verify with top_k / top_p filtered sampling applied to p and q
    before the ratio (sd_verify_linear_filtered); same shapes as
    verify_linear; top_k >= V keeps every token.  Returns n, tokens, prob
    (and keep [B, 2 gamma + 1]: the kept count of each row read, -1 for the
    rest, when want_keep)."""
    dev = target.device
    _dev(target, dev, "target")
    B, G1, V = target.shape
    gamma = G1 - 1
    if draft is not None:
        _dev(draft, dev, "draft", target.dtype)
        if tuple(draft.shape) != (B, gamma, V):
            raise ValueError("draft must be [B, gamma, V]")
    tokens = _dev(tokens, dev, "tokens", torch.int32)
    uniforms = _dev(uniforms, dev, "uniforms", torch.float32)
    n = torch.empty(B, dtype=torch.int32, device=dev)
    toks = torch.empty((B, G1), dtype=torch.int32, device=dev)
    prob = torch.empty(B, dtype=torch.float32, device=dev)
    keep = torch.empty((B, 2 * gamma + 1), dtype=torch.int32,
                       device=dev) if want_keep else None
    L = lib()
    nbytes = L.sd_verify_linear_filtered_workspace(B, gamma, V, _dt(target))
    ws = (workspace or _default_ws).get(dev, nbytes)
    _check(L.sd_verify_linear_filtered(
        _p(target), _p(draft), _dt(target), _p(tokens), _p(uniforms), B,
        gamma, V, float(T), int(top_k), float(top_p), _p(n), _p(toks),
        _p(prob), _p(keep), _p(status), _p(ws), ws.numel(), _stream(dev)))
    r = {"n": n, "tokens": toks, "prob": prob}
    if want_keep:
        r["keep"] = keep
    return r


def verify_kcand(target, draft, tokens, uniforms, T, *, status=None,
                 workspace=None):
    """K-candidate verify with longest-streak selection (sd_verify_kcand).

    target [B, K, gamma+1, V], draft [B, gamma, V] shared marginals, tokens
    [B, K, gamma] int32, uniforms [B, K, gamma+1] float32.  Returns n, k,
    tokens [B, gamma+1], n_per_cand [B, K], prob."""
    dev = target.device
    _dev(target, dev, "target")
    B, K, G1, V = target.shape
    gamma = G1 - 1
    _dev(draft, dev, "draft", target.dtype)
    if tuple(draft.shape) != (B, gamma, V):
        raise ValueError("draft must be [B, gamma, V]")
    tokens = _dev(tokens, dev, "tokens", torch.int32)
    uniforms = _dev(uniforms, dev, "uniforms", torch.float32)
    n = torch.empty(B, dtype=torch.int32, device=dev)
    ks = torch.empty(B, dtype=torch.int32, device=dev)
    toks = torch.empty((B, G1), dtype=torch.int32, device=dev)
    npc = torch.empty((B, K), dtype=torch.int32, device=dev)
    prob = torch.empty(B, dtype=torch.float32, device=dev)
    L = lib()
    nbytes = L.sd_verify_kcand_workspace(B, K, gamma, V, _dt(target))
    ws = (workspace or _default_ws).get(dev, nbytes)
    _check(L.sd_verify_kcand(
        _p(target), _p(draft), _dt(target), _p(tokens), _p(uniforms), B, K,
        gamma, V, float(T), _p(n), _p(ks), _p(toks), _p(npc), _p(prob),
        _p(status), _p(ws), ws.numel(), _stream(dev)))
    return {"n": n, "k": ks, "tokens": toks, "n_per_cand": npc, "prob": prob}


def verify_kcand_trie(target, draft, tokens, uniforms, T, *, status=None,
                      workspace=None):
    """K candidates verified as one token tree (sd_verify_kcand_trie).
    Arguments as verify_kcand (draft may be None when T == 0).  Returns n,
    k (the candidate that created the last accepted node), tokens
    [B, gamma+1], prob."""
    dev = target.device
    _dev(target, dev, "target")
    B, K, G1, V = target.shape
    gamma = G1 - 1
    if draft is not None:
        _dev(draft, dev, "draft", target.dtype)
        if tuple(draft.shape) != (B, gamma, V):
            raise ValueError("draft must be [B, gamma, V]")
    tokens = _dev(tokens, dev, "tokens", torch.int32)
    uniforms = _dev(uniforms, dev, "uniforms", torch.float32)
    n = torch.empty(B, dtype=torch.int32, device=dev)
    ks = torch.empty(B, dtype=torch.int32, device=dev)
    toks = torch.empty((B, G1), dtype=torch.int32, device=dev)
    prob = torch.empty(B, dtype=torch.float32, device=dev)
    L = lib()
    nbytes = L.sd_verify_kcand_trie_workspace(B, K, gamma, V, _dt(target))
    ws = (workspace or _default_ws).get(dev, nbytes)
    _check(L.sd_verify_kcand_trie(
        _p(target), _p(draft), _dt(target), _p(tokens), _p(uniforms), B, K,
        gamma, V, float(T), _p(n), _p(ks), _p(toks), _p(prob), _p(status),
        _p(ws), ws.numel(), _stream(dev)))
    return {"n": n, "k": ks, "tokens": toks, "prob": prob}


def verify_tree(target, draft, parent, node_tokens, uniforms, T, *,
                status=None, workspace=None):
    """Token-tree verify (sd_verify_tree).  target, draft [B, N, V]; parent,
    node_tokens [B, N] int32; uniforms [B, N] float32.  Returns n, tokens
    [B, N], nodes [B, N], prob."""
    dev = target.device
    _dev(target, dev, "target")
    B, N, V = target.shape
    _dev(draft, dev, "draft", target.dtype)
    if tuple(draft.shape) != (B, N, V):
        raise ValueError("draft must be [B, N, V]")
    parent = _dev(parent, dev, "parent", torch.int32)
    node_tokens = _dev(node_tokens, dev, "node_tokens", torch.int32)
    uniforms = _dev(uniforms, dev, "uniforms", torch.float32)
    n = torch.empty(B, dtype=torch.int32, device=dev)
    toks = torch.empty((B, N), dtype=torch.int32, device=dev)
    nodes = torch.empty((B, N), dtype=torch.int32, device=dev)
    prob = torch.empty(B, dtype=torch.float32, device=dev)
    L = lib()
    nbytes = L.sd_verify_tree_workspace(B, N, V, _dt(target))
    ws = (workspace or _default_ws).get(dev, nbytes)
    _check(L.sd_verify_tree(
        _p(target), _p(draft), _dt(target), _p(parent), _p(node_tokens),
        _p(uniforms), B, N, V, float(T), _p(n), _p(toks), _p(nodes),
        _p(prob), _p(status), _p(ws), ws.numel(), _stream(dev)))
    return {"n": n, "tokens": toks, "nodes": nodes, "prob": prob}


def verify_tree_det(target, parent, node_tokens, uniforms, T, *,
                    status=None, workspace=None):
    """Token-tree verify with deterministic drafts (sd_verify_tree_det):
    child v accepted with the current p(t_v), a rejected token removed from
    p.  target [B, N, V]; the rest as verify_tree."""
    dev = target.device
    _dev(target, dev, "target")
    B, N, V = target.shape
    parent = _dev(parent, dev, "parent", torch.int32)
    node_tokens = _dev(node_tokens, dev, "node_tokens", torch.int32)
    uniforms = _dev(uniforms, dev, "uniforms", torch.float32)
    n = torch.empty(B, dtype=torch.int32, device=dev)
    toks = torch.empty((B, N), dtype=torch.int32, device=dev)
    nodes = torch.empty((B, N), dtype=torch.int32, device=dev)
    prob = torch.empty(B, dtype=torch.float32, device=dev)
    L = lib()
    nbytes = L.sd_verify_tree_det_workspace(B, N, V, _dt(target))
    ws = (workspace or _default_ws).get(dev, nbytes)
    _check(L.sd_verify_tree_det(
        _p(target), _dt(target), _p(parent), _p(node_tokens), _p(uniforms),
        B, N, V, float(T), _p(n), _p(toks), _p(nodes), _p(prob), _p(status),
        _p(ws), ws.numel(), _stream(dev)))
    return {"n": n, "tokens": toks, "nodes": nodes, "prob": prob}


class PrestoTree:
    """Device state of PRESTO trees under construction (sd_presto_init):
    node arrays [B, budget], frontier [B, W]."""

    def __init__(self, B, W, budget, device):
        if torch.device(device).type != "cuda":
            raise ValueError("PrestoTree must live on a CUDA device (there "
                             "is no CPU path)")
        self.B, self.W, self.budget = B, W, budget
        i32 = dict(dtype=torch.int32, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        self.n_nodes = torch.empty(B, **i32)
        self.parent = torch.empty((B, budget), **i32)
        self.node_tokens = torch.empty((B, budget), **i32)
        self.node_score = torch.empty((B, budget), **f32)
        self.frontier_node = torch.empty((B, W), **i32)
        self.frontier_score = torch.empty((B, W), **f32)
        _check(lib().sd_presto_init(
            B, W, budget, _p(self.n_nodes), _p(self.parent),
            _p(self.node_tokens), _p(self.node_score),
            _p(self.frontier_node), _p(self.frontier_score),
            _stream(torch.device(device))))


def presto_expand(tree, q_logits, log_rho, T, lam, b_top, *, status=None,
                  workspace=None):
    """One depth of PRESTO's beam construction (sd_presto_expand) on `tree`
    (a PrestoTree, updated in place).  q_logits [B, V] (rows may be strided,
    e.g. q[:, d] of a [B, D, V] tensor); log_rho [B, W, V] (None when
    lam == 0)."""
    dev = q_logits.device
    B, V = q_logits.shape
    if not q_logits.is_cuda or q_logits.stride(1) != 1:
        raise ValueError("q_logits must be CUDA rows with unit stride")
    if log_rho is not None:
        _dev(log_rho, dev, "log_rho", q_logits.dtype)
        if tuple(log_rho.shape) != (B, tree.W, V):
            raise ValueError("log_rho must be [B, W, V]")
    L = lib()
    nbytes = L.sd_presto_expand_workspace(B, tree.W, V, int(b_top),
                                          _dt(q_logits))
    ws = (workspace or _default_ws).get(dev, nbytes)
    _check(L.sd_presto_expand(
        _p(q_logits), q_logits.stride(0), _p(log_rho), _dt(q_logits), B,
        tree.W, V, float(T), float(lam), int(b_top), tree.budget,
        _p(tree.n_nodes), _p(tree.parent), _p(tree.node_tokens),
        _p(tree.node_score), _p(tree.frontier_node), _p(tree.frontier_score),
        _p(status), _p(ws), ws.numel(), _stream(dev)))
    return tree


def branch_fork(draft, x_b, T, k_max, *, status=None, workspace=None):
    """SpecBranch fork (sd_branch_fork): k = max(1, floor(k_max (1 -
    q(x_b)))) (capped at V) and the top-k tokens of each row.  draft
    [B, V]; x_b [B].  Returns k [B], tokens [B, k_max]."""
    dev = draft.device
    _dev(draft, dev, "draft")
    B, V = draft.shape
    x_b = _dev(x_b, dev, "x_b", torch.int32)
    k = torch.empty(B, dtype=torch.int32, device=dev)
    toks = torch.empty((B, k_max), dtype=torch.int32, device=dev)
    L = lib()
    nbytes = L.sd_branch_fork_workspace(B, V, int(k_max), _dt(draft))
    ws = (workspace or _default_ws).get(dev, nbytes)
    _check(L.sd_branch_fork(_p(draft), _dt(draft), _p(x_b), B, V, float(T),
                            int(k_max), _p(k), _p(toks), _p(status), _p(ws),
                            ws.numel(), _stream(dev)))
    return {"k": k, "tokens": toks}


def selftest_bounded_wait(polls, device="cuda"):
    """The failure-path self-test (sd_selftest_bounded_wait): a wait that
    can never complete, bounded by `polls` polls.  Returns (status word,
    threads whose wait gave up, 1 if the kernel ran to its end)."""
    dev = torch.device(device)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.zeros(2, dtype=torch.int32, device=dev)
    _check(lib().sd_selftest_bounded_wait(int(polls), _p(st), _p(out),
                                          _stream(dev)))
    torch.cuda.synchronize(dev)
    o = out.tolist()
    return int(st.item()), o[0], o[1]


def fanout_schedule(K, budget, a, r):
    """Geometric fan-out F[0..K] (sd_fanout_schedule, host only)."""
    F = (ctypes.c_int32 * (K + 1))()
    _check(lib().sd_fanout_schedule(int(K), int(budget), float(a), float(r),
                                    ctypes.cast(F, ctypes.c_void_p)))
    return [int(x) for x in F]


def fanout_topk(draft, F, *, want_logit=False, status=None, workspace=None):
    """Top-F_k tokens per lookahead row (sd_fanout_topk).  draft [B, K+1, V];
    F a list of K+1 ints.  Returns tokens [B, sum F] (and logit)."""
    dev = draft.device
    _dev(draft, dev, "draft")
    B, K1, V = draft.shape
    F = [int(x) for x in F]
    if len(F) != K1:
        raise ValueError("F must have K+1 entries")
    Fh = (ctypes.c_int32 * K1)(*F)
    total = sum(F)
    toks = torch.empty((B, max(total, 1)), dtype=torch.int32, device=dev)
    lg = torch.empty((B, max(total, 1)), dtype=torch.float32,
                     device=dev) if want_logit else None
    L = lib()
    nbytes = L.sd_fanout_topk_workspace(B, K1 - 1, V, _dt(draft))
    ws = (workspace or _default_ws).get(dev, nbytes)
    _check(L.sd_fanout_topk(
        _p(draft), _dt(draft), B, K1 - 1, V, ctypes.cast(Fh, ctypes.c_void_p),
        _p(toks), _p(lg), _p(status), _p(ws), ws.numel(), _stream(dev)))
    r = {"tokens": toks[:, :total]}
    if want_logit:
        r["logit"] = lg[:, :total]
    return r


def fanout_hits(n, tokens, fan_tokens, F):
    """Saguaro cache hit of each sequence's verification outcome
    (sd_fanout_hits): 1 if tokens[b, n[b]] is among the F[n[b]] fan-out
    tokens of position n[b], 0 if not, -1 where n[b] < 0.  n [B], tokens
    [B, K+1] and fan_tokens [B, sum F] int32 on one CUDA device."""
    dev = n.device
    n = _dev(n, dev, "n", torch.int32)
    tokens = _dev(tokens, dev, "tokens", torch.int32)
    F = [int(x) for x in F]
    B, K1 = tokens.shape
    if len(F) != K1:
        raise ValueError("F must have K+1 entries")
    fan_tokens = _dev(fan_tokens, dev, "fan_tokens", torch.int32)
    if tuple(fan_tokens.shape) != (B, sum(F)):
        raise ValueError("fan_tokens must be [B, sum F]")
    Fh = (ctypes.c_int32 * K1)(*F)
    hit = torch.empty(B, dtype=torch.int32, device=dev)
    _check(lib().sd_fanout_hits(_p(n), _p(tokens), _p(fan_tokens), B, K1 - 1,
                                ctypes.cast(Fh, ctypes.c_void_p), _p(hit),
                                _stream(dev)))
    return hit


def verify_linear_fanout(target, draft, tokens, uniforms, T, F, *,
                         status=None, workspace=None):
    """Linear verify fused with the fan-out of the same draft logits
    (sd_verify_linear_fanout).  draft [B, gamma+1, V] (K == gamma)."""
    dev = target.device
    _dev(target, dev, "target")
    B, G1, V = target.shape
    gamma = G1 - 1
    _dev(draft, dev, "draft", target.dtype)
    if tuple(draft.shape) != (B, gamma + 1, V):
        raise ValueError("draft must be [B, gamma+1, V]")
    tokens = _dev(tokens, dev, "tokens", torch.int32)
    uniforms = _dev(uniforms, dev, "uniforms", torch.float32)
    F = [int(x) for x in F]
    if len(F) != gamma + 1:
        raise ValueError("F must have gamma+1 entries")
    Fh = (ctypes.c_int32 * (gamma + 1))(*F)
    total = sum(F)
    n = torch.empty(B, dtype=torch.int32, device=dev)
    toks = torch.empty((B, G1), dtype=torch.int32, device=dev)
    prob = torch.empty(B, dtype=torch.float32, device=dev)
    ftok = torch.empty((B, max(total, 1)), dtype=torch.int32, device=dev)
    flog = torch.empty((B, max(total, 1)), dtype=torch.float32, device=dev)
    L = lib()
    nbytes = L.sd_verify_linear_fanout_workspace(B, gamma, V, _dt(target))
    ws = (workspace or _default_ws).get(dev, nbytes)
    _check(L.sd_verify_linear_fanout(
        _p(target), _p(draft), _dt(target), _p(tokens), _p(uniforms), B,
        gamma, V, float(T), ctypes.cast(Fh, ctypes.c_void_p), _p(n),
        _p(toks), _p(prob), _p(ftok), _p(flog), _p(status), _p(ws),
        ws.numel(), _stream(dev)))
    return {"n": n, "tokens": toks, "prob": prob,
            "fan_tokens": ftok[:, :total], "fan_logit": flog[:, :total]}
