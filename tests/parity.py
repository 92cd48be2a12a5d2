"""Helpers for comparing the CUDA path with the fp64 oracle.

The rule, draw by draw:
 - accept tests: the accepted counts (and everything derived from them)
   must be identical, except on sequences where some accept test has
   |r - p/q| < 1e-5 (the oracle's accept margin): an fp32 implementation may
   decide either way there, so the sequence is set aside (and counted);
 - the final inverse-CDF draw: the token must be identical when u lies more
   than 1e-5 from both CDF boundaries of the oracle's token; otherwise it
   must lie in the oracle's admissible range [cdf_lo, cdf_hi] (tokens whose
   CDF interval comes within 1e-5 of u); such draws are counted;
 - greedy (T == 0) draws are never set aside;
 - returned probabilities agree within 1e-5 absolute where the token is the
   oracle's.
"""
import numpy as np
import torch

import oracle
from speculative_decoding_verification_temperature_gb300 import synth

PROB_TOL = 1e-5


def host(t):
    return t.detach().cpu().numpy() if isinstance(t, torch.Tensor) else t


def compare(gpu, orc, extra_equal=(), prob=True):
    """Assert parity; return a dict of counts: sequences, sequences with a
    flagged accept test (acc_flagged), accept tests made (tests) and flagged
    (tests_flagged), cdf-flagged final draws and those whose token differs
    from the oracle's (cdf_diff)."""
    acc_flag = host(orc["margin_acc"]) < oracle.FLAG_MARGIN
    cdf_flag = host(orc["margin_cdf"]) < oracle.FLAG_MARGIN
    keep = ~acc_flag
    gn, on = host(gpu["n"]), host(orc["n"])
    bad = np.nonzero((gn != on) & keep)[0]
    assert bad.size == 0, "n differs on %d sequences, first %d: %s vs %s" % (
        bad.size, bad[0], gn[bad[0]], on[bad[0]])
    for k in extra_equal:
        g, o = host(gpu[k]), host(orc[k])
        d = (g != o).reshape(len(g), -1).any(axis=1) & keep
        assert not d.any(), "%s differs at %s" % (k, np.nonzero(d)[0][:5])
    gt, ot = host(gpu["tokens"]), host(orc["tokens"])
    cols = np.arange(gt.shape[1])[None, :]
    n = on[:, None]
    final = (cols == n) & (n >= 0)
    exact = ~final | ~cdf_flag[:, None]
    d = ((gt != ot) & exact).any(axis=1) & keep
    assert not d.any(), "tokens differ at %s: gpu %s oracle %s" % (
        np.nonzero(d)[0][:5], gt[d][0], ot[d][0])
    fin_rows = np.nonzero(keep & cdf_flag & (on >= 0))[0]
    lo, hi = host(orc["cdf_lo"]), host(orc["cdf_hi"])
    g_fin = gt[fin_rows, on[fin_rows]]
    inside = (g_fin >= lo[fin_rows]) & (g_fin <= hi[fin_rows])
    assert inside.all(), "near-boundary draw outside the admissible range"
    cdf_diff = int((g_fin != ot[fin_rows, on[fin_rows]]).sum())
    if prob and "prob" in gpu:
        g = host(gpu["prob"]).astype(np.float64)
        o = host(orc["prob"])
        same = keep & ~(cdf_flag & (gt[np.arange(len(gt)),
                                       np.maximum(on, 0)] !=
                                    ot[np.arange(len(ot)), np.maximum(on, 0)]))
        err = np.abs(g - o)[same]
        assert err.size == 0 or err.max() <= PROB_TOL, err.max()
    tests = int(host(orc["acc_tests"]).sum()) if "acc_tests" in orc else 0
    tflag = int(host(orc["acc_flagged"]).sum()) if "acc_flagged" in orc else 0
    return {"seqs": len(gn), "acc_flagged": int(acc_flag.sum()),
            "tests": tests, "tests_flagged": tflag,
            "cdf_flagged": int((cdf_flag & keep).sum()), "cdf_diff": cdf_diff}


FLAG_BAR = 1e-4
"""Bar on the fraction of accept tests whose |r - p/q| lies within 1e-5:
for r uniform on (0, 1) that probability is at most 2e-5 whatever p/q is,
so the fraction is binomial with a rate of at most 2e-5."""


def assert_flag_fraction(r):
    """The accept-flagged fraction of a run stays below FLAG_BAR.  With
    fewer than 1 / FLAG_BAR tests a single flagged test would already be
    above the bar, while a rate of 2e-5 leaves a second one unlikely
    (below 2e-4 at 1e4 tests): such runs may hold at most one."""
    if r["tests"] >= 1 / FLAG_BAR:
        assert r["tests_flagged"] / r["tests"] < FLAG_BAR, r
    else:
        assert r["tests_flagged"] <= 1, r


def linear_oracle(case, want_resid=False):
    return oracle.verify_linear(
        synth.host_logits(case.target),
        None if case.T == 0 else synth.host_logits(
            case.draft[:, :case.target.shape[1] - 1]),
        host(case.tokens), host(case.uniforms), case.T, want_resid=want_resid)


def to_device(case, device="cuda"):
    """Move every tensor field of a synth case to the device."""
    for k, v in list(vars(case).items()):
        if isinstance(v, torch.Tensor):
            setattr(case, k, v.to(device).contiguous())
    return case


def oracle_over_threads(fn, n, nthreads=None):
    """fn(lo, hi) -> dict of arrays over sequences lo..hi-1, run over
    contiguous chunks of range(n) in host threads (the C oracle runs with
    the interpreter lock released); the chunks' dicts are concatenated in
    sequence order."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    oracle.build()
    nt = max(1, min(n, nthreads or len(os.sched_getaffinity(0))))
    bounds = [(n * i // nt, n * (i + 1) // nt) for i in range(nt)]
    bounds = [b for b in bounds if b[1] > b[0]]
    with ThreadPoolExecutor(max_workers=len(bounds)) as pool:
        parts = list(pool.map(lambda b: fn(*b), bounds))
    out = {}
    for k, v in parts[0].items():
        if isinstance(v, np.ndarray) and v.ndim >= 1:
            out[k] = np.concatenate([p[k] for p in parts])
        else:
            out[k] = v
    return out


def linear_oracle_full(target, draft, tokens, uniforms, T):
    """The oracle's linear verify of every sequence of device tensors
    (target [B, gamma+1, V]; draft [B, >= gamma, V] or None when T == 0),
    over host threads."""
    gamma = target.shape[1] - 1
    t = synth.host_logits(target)
    d = None if T == 0 else synth.host_logits(draft)
    tk, u = host(tokens), host(uniforms)

    def part(lo, hi):
        dd = None if d is None else np.ascontiguousarray(d[lo:hi, :gamma])
        return oracle.verify_linear(t[lo:hi], dd, tk[lo:hi], u[lo:hi], T)
    return oracle_over_threads(part, target.shape[0])
