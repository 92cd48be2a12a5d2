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
    """Assert parity; return a dict of counts (sequences, accept-flagged,
    cdf-flagged, cdf-flagged draws whose token differs from the oracle's)."""
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
    return {"seqs": len(gn), "acc_flagged": int(acc_flag.sum()),
            "cdf_flagged": int((cdf_flag & keep).sum()), "cdf_diff": cdf_diff}


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
