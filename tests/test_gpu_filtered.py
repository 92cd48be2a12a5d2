"""Parity of sd_verify_linear_filtered (top-k / top-p filtered sampling
applied to p and q before the ratio; CUDA, through the C ABI) with the fp64
oracle: small and odd sizes, gamma 0..4, top_k from 1 to 64, top_p below
and at 1, T 0.7 and 1, drafts drawn from the filtered draft distribution,
every cluster size, the large workload's shape on sampled sequences, NaN
rows, the greedy route and the refusal of misaligned rows."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_temperature_gb300 import api, synth
from tests.parity import (assert_flag_fraction, compare, host,
                          oracle_over_threads, to_device)

pytestmark = pytest.mark.gpu


def filtered_np(z, T, top_k, top_p):
    """The filtered distribution (top_k by logit desc / id asc, then the
    nucleus over the renormalised top_k), for drawing test drafts."""
    z = np.asarray(z, np.float64)
    p = np.exp((z - z.max()) / T)
    p /= p.sum()
    order = np.lexsort((np.arange(len(z)), -z))[:top_k]
    before = np.concatenate([[0.0], np.cumsum(p[order])[:-1]]) / p[order].sum()
    keep = order[before < top_p] if top_p < 1.0 else order
    out = np.zeros_like(p)
    out[keep] = p[keep] / p[keep].sum()
    return out


def case(B, gamma, V, dtype, T, top_k, top_p, seed):
    c = synth.linear_case(B, gamma, V, dtype, T, seed=seed, sigma_t=2.0,
                          sigma_d=1.0)
    d = synth.host_logits(c.draft)
    if d.dtype == np.uint16:
        d = (d.astype(np.uint32) << 16).view(np.float32)
    rng = np.random.default_rng(seed)
    toks = np.empty((B, gamma), np.int32)
    for b in range(B):
        for i in range(gamma):
            q = filtered_np(d[b, i], T, top_k, top_p)
            g = -np.log(-np.log(rng.random(V).clip(1e-300)))
            with np.errstate(divide="ignore"):
                toks[b, i] = np.argmax(np.log(q) + g)
    c.tokens = torch.from_numpy(toks)
    return c


def run(c, top_k, top_p, **kw):
    gamma = c.target.shape[1] - 1
    return api.verify_linear_filtered(
        c.target, None if c.T == 0 else c.draft[:, :gamma].contiguous(),
        c.tokens, c.uniforms, c.T, top_k, top_p, **kw)


def orc(c, top_k, top_p, idx=None):
    sel = slice(None) if idx is None else idx
    gamma = c.target.shape[1] - 1
    return oracle.verify_linear_filtered(
        synth.host_logits(c.target[sel]),
        None if c.T == 0 else np.ascontiguousarray(
            synth.host_logits(c.draft[sel])[:, :gamma]),
        host(c.tokens[sel]), host(c.uniforms[sel]), c.T, top_k, top_p)


@pytest.mark.parametrize("V,dtype", [(1000, torch.float32),
                                     (4104, torch.bfloat16),
                                     (32000, torch.bfloat16)])
@pytest.mark.parametrize("gamma", [0, 1, 4])
@pytest.mark.parametrize("top_k,top_p", [(1, 1.0), (5, 0.9), (50, 0.5),
                                         (64, 1.0)])
def test_small_cases(V, dtype, gamma, top_k, top_p):
    for T in (0.7, 1.0):
        c = to_device(case(24, gamma, V, dtype, T, top_k, top_p,
                           seed=V + gamma + top_k))
        r = compare(run(c, top_k, top_p), orc(c, top_k, top_p))
        assert r["acc_flagged"] <= 2


@pytest.mark.parametrize("cluster", ["1", "2", "8"])
def test_cluster_sizes(cluster):
    c = to_device(case(16, 3, 40000, torch.float32, 1.0, 40, 0.95,
                       seed=int(cluster)))
    with api.tuned(cluster=int(cluster)):
        g = run(c, 40, 0.95)
    compare(g, orc(c, 40, 0.95))


def test_large_workload_shape_every_sequence():
    """B=256, gamma=8, V=128256 fp32, T=1, top_k=50, top_p=0.9; drafts from
    the workload's (unfiltered) draft sampler: all 256 sequences against
    the oracle (host threads)."""
    c = synth.large(0, device="cuda")
    c.draft = c.draft[:, :8].contiguous()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = run(c, 50, 0.9, status=st)
    assert int(st.item()) & ~api.DEV_ZERO_MASS == 0
    t, d = synth.host_logits(c.target), synth.host_logits(c.draft)
    tk, u = host(c.tokens), host(c.uniforms)
    o = oracle_over_threads(lambda lo, hi: oracle.verify_linear_filtered(
        t[lo:hi], d[lo:hi], tk[lo:hi], u[lo:hi], 1.0, 50, 0.9), 256)
    r = compare(g, o)
    assert r["seqs"] == 256
    assert_flag_fraction(r)


def test_nan_rows_and_greedy_and_misaligned():
    c = case(6, 3, 2000, torch.float32, 1.0, 10, 0.9, seed=5)
    c.target[1, 2, 7] = float("nan")
    c.draft[2, 0, 3] = float("nan")
    c = to_device(c)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    compare(run(c, 10, 0.9, status=st), orc(c, 10, 0.9))
    # greedy: the same outputs as sd_verify_linear
    g = to_device(case(8, 3, 2000, torch.float32, 1.0, 10, 0.9, seed=6))
    g.T = 0.0
    a = run(g, 10, 0.9)
    b = api.verify_linear(g.target, None, g.tokens, g.uniforms, 0.0)
    assert torch.equal(a["n"], b["n"]) and torch.equal(a["tokens"],
                                                       b["tokens"])
    # misaligned rows are refused
    m = to_device(case(4, 2, 1001, torch.float32, 1.0, 5, 1.0, seed=7))
    with pytest.raises(api.SdError):
        run(m, 5, 1.0)
