"""Helpers for comparing the CUDA path with the fp64 oracle.

The rule: accepted counts and emitted tokens must be identical, except on
sequences where the oracle flags a draw (a margin below 1e-5 between the
uniform and an accept threshold or CDF boundary: an fp32 implementation may
legitimately land on the other side there).  Greedy (T == 0) is never
flagged.  Returned probabilities must agree within 1e-5 absolute.
"""
import numpy as np
import torch

import oracle
from speculative_decoding_verification_temperature_gb300 import synth

PROB_TOL = 1e-5


def host(t):
    return t.detach().cpu().numpy() if isinstance(t, torch.Tensor) else t


def compare(gpu, orc, keys=("n", "tokens"), extra_equal=(), prob=True):
    """Assert parity; return (flagged count, total)."""
    flagged = host(orc["margin"]) < oracle.FLAG_MARGIN
    ok = ~flagged
    for k in keys + tuple(extra_equal):
        g = host(gpu[k])
        o = host(orc[k])
        diff = (g != o).reshape(g.shape[0], -1).any(axis=1)
        bad = np.nonzero(diff & ok)[0]
        assert bad.size == 0, (
            "%s differs on %d unflagged sequences, first %d: gpu %s oracle %s"
            % (k, bad.size, bad[0], g[bad[0]], o[bad[0]]))
    if prob and "prob" in gpu:
        g = host(gpu["prob"]).astype(np.float64)
        o = host(orc["prob"])
        err = np.abs(g - o)[ok]
        assert err.size == 0 or err.max() <= PROB_TOL, err.max()
    return int(flagged.sum()), len(flagged)


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
