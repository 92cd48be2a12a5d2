"""Parity of sd_verify_linear_filtered (top-k / top-p filtered sampling
applied to p and q before the ratio; CUDA, through the C ABI) with the fp64
oracle: small and odd sizes, gamma 0..4, top_k from 1 to 64 (exact lists)
and above it or off (the threshold select), top_p below and at 1, T 0.7
and 1, drafts drawn from the filtered draft distribution, every cluster
size, the large workload's shape on every sequence (top_k 50 with top_p
0.9, top_p alone at 0.9 and 0.95, top_k 1000), ties, masked tails and
deep cuts, NaN rows, the greedy route and the refusal of misaligned rows.

Nucleus cuts: where a prefix mass lies within 1e-5 of top_p an fp32
computation may keep one token more or fewer than the fp64 oracle (at
V = 128256 the prefix masses near the cut are ~1e-5 apart, so this is the
common case for top_p alone).  The GPU reports the kept count of every row
it read; each must lie in the oracle's admissible range, and the oracle run
again with the GPU's counts forced must then match it exactly."""
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


def orc(c, top_k, top_p, idx=None, **kw):
    sel = slice(None) if idx is None else idx
    gamma = c.target.shape[1] - 1
    return oracle.verify_linear_filtered(
        synth.host_logits(c.target[sel]),
        None if c.T == 0 else np.ascontiguousarray(
            synth.host_logits(c.draft[sel])[:, :gamma]),
        host(c.tokens[sel]), host(c.uniforms[sel]), c.T, top_k, top_p, **kw)


def check_forced(c, top_k, top_p, g=None, oracle_fn=None):
    """The forced-cut comparison: the GPU's kept count of every row it read
    lies in the oracle's admissible range, and the oracle with those counts
    forced gives the GPU's results (parity.compare's rules).  oracle_fn(**kw)
    runs the oracle (default: orc on the whole case)."""
    if g is None:
        g = run(c, top_k, top_p, want_keep=True)
    fn = oracle_fn or (lambda **kw: orc(c, top_k, top_p, **kw))
    o = fn(want_keep=True)
    gk = host(g["keep"])
    both = (gk >= 0) & (o["keep"] >= 0)
    lo, hi = o["keep_lo"], o["keep_hi"]
    out = np.nonzero(both & ((gk < lo) | (gk > hi)))
    assert out[0].size == 0, "kept count outside the admissible range at %s: " \
        "gpu %s, oracle [%s, %s]" % (out, gk[out][:5], lo[out][:5], hi[out][:5])
    of = fn(want_keep=True, keep_forced=np.where(gk >= 1, gk, -1))
    r = compare(g, of)
    same = (host(g["n"]) == of["n"]) & (of["margin_acc"] >= 1e-5)
    assert np.array_equal(gk[same] >= 0, of["keep"][same] >= 0), \
        "rows read differ"
    r["cut_differs"] = int((both & (gk != o["keep"])).sum())
    return r


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


@pytest.mark.parametrize("V,dtype", [(1000, torch.float32),
                                     (4104, torch.bfloat16),
                                     (32000, torch.bfloat16)])
@pytest.mark.parametrize("gamma", [0, 1, 4])
@pytest.mark.parametrize("top_k,top_p", [(1 << 30, 0.9), (100, 1.0),
                                         (1000, 0.95), (1 << 30, 0.5),
                                         (65, 0.8), (1 << 30, 1.0)])
def test_threshold_select_small_cases(V, dtype, gamma, top_k, top_p):
    """top_k above the exact-list limit or off (the threshold select)."""
    for T in (0.7, 1.0):
        k = min(top_k, V)
        c = to_device(case(24, gamma, V, dtype, T, k, top_p,
                           seed=V + gamma + k))
        r = check_forced(c, top_k, top_p)
        assert r["acc_flagged"] <= 2


@pytest.mark.parametrize("T,sigma,top_k,top_p", [
    (1.0, 0.0, 500, 1.0),      # constant rows: ties broken by id
    (1.0, 0.0, 1 << 30, 0.5),  # constant rows, nucleus
    (8.0, 1.0, 3000, 0.9),     # high temperature: few level-1 buckets
    (0.05, 2.0, 2000, 1.0),    # low temperature: the cut deep in the last
    (0.05, 2.0, 1 << 30, 0.999999),  # bucket, refined over keys
])
def test_threshold_select_refinement(T, sigma, top_k, top_p):
    """Cuts inside a level-1 bucket of more than 256 tokens: refined over
    the (value, id) keys before the gather."""
    B, gamma, V = 12, 3, 4096
    c = synth.linear_case(B, gamma, V, torch.float32, T, seed=31,
                          sigma_t=max(sigma, 1e-6), sigma_d=1.0)
    if sigma == 0.0:
        c.target = torch.full_like(c.target, 0.25)
        c.draft = torch.full_like(c.draft, 0.25)
    c.draft[:, :, V // 2:] = c.target[:, :gamma, V // 2:]
    c = to_device(c)
    check_forced(c, top_k, top_p)


def redraw(c, T, top_k, top_p, seed):
    """Draft tokens drawn again from the filtered draft rows of c."""
    d = synth.host_logits(c.draft)
    if d.dtype == np.uint16:
        d = (d.astype(np.uint32) << 16).view(np.float32)
    B, gamma = c.tokens.shape
    V = d.shape[-1]
    rng = np.random.default_rng(seed)
    for b in range(B):
        for i in range(gamma):
            q = filtered_np(d[b, i], T, top_k, top_p)
            g = -np.log(-np.log(rng.random(V).clip(1e-300)))
            with np.errstate(divide="ignore"):
                c.tokens[b, i] = int(np.argmax(np.log(q) + g))
    return c


@pytest.mark.parametrize("V,dtype", [(4104, torch.bfloat16),
                                     (32000, torch.float32),
                                     (128256, torch.float32)])
@pytest.mark.parametrize("top_k,top_p", [(50, 1.0), (64, 0.5), (7, 0.9)])
def test_small_k_ties_and_masked_tails(V, dtype, top_k, top_p):
    """top_k <= 64 (exact lists) on rows whose bound from the lane maxima
    admits many elements: constant rows (every element ties), rows with
    fewer finite logits than top_k (-inf tails, the bound is -inf), logits
    on a coarse grid (many ties at the bound), and ordinary rows beside
    them in the same launch."""
    B, gamma, T = 8, 3, 1.0
    c = synth.linear_case(B, gamma, V, dtype, T, seed=V + top_k,
                          sigma_t=2.0, sigma_d=1.0)
    c.target[0] = 0.25
    c.draft[0] = 0.25
    c.target[1, :, 30:] = -float("inf")
    c.draft[1, :, 30:] = -float("inf")
    c.target[2, :, :V - 5] = -float("inf")
    c.draft[2, :, 7:] = -float("inf")
    c.target[3] = torch.round(c.target[3].float() * 2).to(dtype) / 2
    c.draft[3] = torch.round(c.draft[3].float() * 2).to(dtype) / 2
    c.target[4, 1] = 0.25
    c.draft[4, :, V // 2:] = c.target[4, :gamma, V // 2:]
    c = to_device(redraw(c, T, top_k, top_p, seed=V))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = compare(run(c, top_k, top_p, status=st), orc(c, top_k, top_p))
    assert r["acc_flagged"] <= 2
    assert int(st.item()) & api.DEV_NONFINITE == 0


def test_threshold_select_edges():
    """Masked tails (-inf), a bad token, NaN and +inf rows, bf16 ties."""
    B, gamma, V = 10, 3, 8192
    c = synth.linear_case(B, gamma, V, torch.bfloat16, 1.0, seed=8,
                          sigma_t=0.3, sigma_d=0.3)
    c.target[0, :, 100:] = -float("inf")
    c.draft[0, :, 50:] = -float("inf")
    c.tokens[1, 0] = V + 3
    c.target[2, 0, 7] = float("nan")
    c.draft[3, 0, 9] = float("inf")
    c = to_device(c)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = run(c, 1 << 30, 0.9, want_keep=True, status=st)
    check_forced(c, 1 << 30, 0.9, g)
    s = int(st.item())
    assert s & api.DEV_NONFINITE and s & api.DEV_BAD_TOKEN
    assert np.all(host(g["n"])[2:4] == -1)


@pytest.mark.parametrize("top_k,top_p", [(1 << 30, 0.9), (1 << 30, 0.95),
                                         (1000, 1.0), (50, 0.9)])
def test_large_shape_general_every_sequence(top_k, top_p):
    """B=256, gamma=8, V=128256 fp32, T=1: top_p alone (0.9, 0.95), top_k
    1000 alone, and top_k 50 with top_p 0.9 through the forced-cut rule:
    every sequence against the oracle (host threads)."""
    c = synth.large(0, device="cuda")
    c.draft = c.draft[:, :8].contiguous()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = run(c, top_k, top_p, want_keep=True, status=st)
    assert int(st.item()) & ~api.DEV_ZERO_MASS == 0
    t, d = synth.host_logits(c.target), synth.host_logits(c.draft)
    tk, u = host(c.tokens), host(c.uniforms)

    def fn(keep_forced=None, **kw):
        def part(lo, hi):
            f = None if keep_forced is None else keep_forced[lo:hi]
            return oracle.verify_linear_filtered(
                t[lo:hi], d[lo:hi], tk[lo:hi], u[lo:hi], 1.0, top_k, top_p,
                keep_forced=f, **kw)
        return oracle_over_threads(part, 256)
    r = check_forced(c, top_k, top_p, g, oracle_fn=fn)
    assert r["seqs"] == 256
    assert_flag_fraction(r)


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
