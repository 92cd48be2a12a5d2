"""Parity of sd_verify_linear (CUDA, through the C ABI) with the fp64 oracle.

Covers the two small workloads at full size (tiny: B=1, gamma=4, V=1000
fp32; linear: B=32, gamma=8, V=32000 bf16 at T in {0, 0.7, 1}), ragged and
unaligned vocabularies (scalar path), gamma 0 and 1, the queue path
(B larger than the resident clusters), the large workload (B=256, gamma=8,
V=128256 fp32) on every sequence, the edge cases (bad token, NaN and
+inf rows, -inf masks, zero-mass residual), the debug outputs, and the
emitted-token law on the GPU (chi-square, 1e6 trials).
"""
import math

import numpy as np
import pytest
import torch
from scipy import stats

import oracle
from speculative_decoding_verification_temperature_gb300 import api, synth
from tests.parity import (assert_flag_fraction, compare, host,
                          linear_oracle, linear_oracle_full, to_device)

pytestmark = pytest.mark.gpu


def run(case, **kw):
    return api.verify_linear(case.target, None if case.T == 0 else
                             case.draft[:, :case.target.shape[1] - 1]
                             .contiguous(), case.tokens, case.uniforms,
                             case.T, **kw)


def test_tiny_workload_single_calls():
    """The tiny workload as separate B = 1 calls, fresh logits each round."""
    flagged = 0
    for rnd in range(40):
        c = to_device(synth.tiny(rnd))
        g = run(c, want_accept=True)
        o = linear_oracle(c)
        r = compare(g, o)
        flagged += r["acc_flagged"]
        if not r["acc_flagged"]:
            ev = o["accept"] >= 0
            np.testing.assert_allclose(host(g["accept"])[ev], o["accept"][ev],
                                       atol=1e-5)
            assert np.all(host(g["accept"])[~ev] == -1)
    assert flagged <= 1


def test_tiny_workload_batched_1000_rounds():
    """1000 independent tiny rounds in one call (queue path)."""
    c = to_device(synth.linear_case(1000, 4, 1000, torch.float32, 1.0,
                                    seed=1000, sigma_t=2.0, sigma_d=1.0))
    r = compare(run(c), linear_oracle(c))
    assert_flag_fraction(r)


@pytest.mark.parametrize("T", [0.0, 0.7, 1.0])
def test_linear_workload(T):
    """B=32, gamma=8, V=32000 bf16, spike +8, draft noise 1.5, full size."""
    c = to_device(synth.linear(T))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = run(c, want_accept=True, status=st)
    o = linear_oracle(c)
    r = compare(g, o)
    assert_flag_fraction(r)
    if T == 0:
        assert r["acc_flagged"] == 0 and r["cdf_flagged"] == 0
    assert int(st.item()) == 0
    ok = o["margin_acc"] >= oracle.FLAG_MARGIN
    ev = (o["accept"] >= 0) & ok[:, None]
    np.testing.assert_allclose(host(g["accept"])[ev], o["accept"][ev],
                               atol=1e-5)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("V", [1, 7, 33, 1001, 4099, 32003, 70001])
@pytest.mark.parametrize("T", [0.0, 1.3])
def test_ragged_vocab(dtype, V, T):
    """Vocabulary sizes that are not a multiple of the vector width (scalar
    path) or span several segments with a ragged tail."""
    for gamma in (0, 1, 3):
        c = to_device(synth.linear_case(24, gamma, V, dtype, T,
                                        seed=V * 10 + gamma, sigma_t=2.0,
                                        sigma_d=1.0))
        compare(run(c), linear_oracle(c))


def test_unaligned_pointer_uses_scalar_path():
    c = synth.linear_case(16, 3, 4096, torch.float32, 1.0, seed=5)
    big_t = torch.empty(c.target.numel() + 1, device="cuda")
    big_d = torch.empty(c.draft.numel() + 1, device="cuda")
    t = big_t[1:].view(c.target.shape)
    d = big_d[1:].view(c.draft.shape)
    t.copy_(c.target)
    d.copy_(c.draft)
    g = api.verify_linear(t, d, c.tokens.cuda(), c.uniforms.cuda(), 1.0)
    compare(g, linear_oracle(c))


def test_empty_batch():
    t = torch.empty((0, 3, 10), device="cuda")
    d = torch.empty((0, 2, 10), device="cuda")
    g = api.verify_linear(t, d, torch.empty((0, 2), dtype=torch.int32,
                                            device="cuda"),
                          torch.empty((0, 3), device="cuda"), 1.0)
    assert g["n"].numel() == 0


def test_deterministic():
    c = to_device(synth.linear(1.0))
    a = run(c)
    b = run(c)
    for k in a:
        assert torch.equal(a[k], b[k])


def test_resid_and_accept_debug_outputs():
    """out_resid is the normalised distribution of the last draw: within
    1e-5 of the oracle's (residual norm(max(0, p - q)), bonus p, or one-hot
    when greedy)."""
    for T in (0.0, 0.8, 1.0):
        c = to_device(synth.linear_case(64, 3, 500, torch.float32, T, seed=7,
                                        sigma_t=1.5, sigma_d=1.0))
        g = run(c, want_resid=True)
        o = linear_oracle(c, want_resid=True)
        compare(g, o)
        ok = (o["margin_acc"] >= oracle.FLAG_MARGIN) & \
            (host(g["tokens"]) == o["tokens"]).all(axis=1)
        np.testing.assert_allclose(host(g["resid"])[ok], o["resid"][ok],
                                   atol=1e-5)


def test_large_workload_every_sequence():
    """B=256, gamma=8, V=128256 fp32 (the benchmark's workload and launch):
    all 256 sequences against the oracle (run over host threads), and the
    accept-flagged fraction held to the bar."""
    c = synth.large(0, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    draft_v = c.draft[:, :8].contiguous()
    g = api.verify_linear(c.target, draft_v, c.tokens, c.uniforms, 1.0,
                          status=st)
    assert int(st.item()) == 0
    n = host(g["n"])
    assert n.min() >= 0 and n.max() <= 8
    o = linear_oracle_full(c.target, draft_v, c.tokens, c.uniforms, 1.0)
    r = compare(g, o)
    assert r["seqs"] == 256 and r["tests"] > 0
    assert_flag_fraction(r)


def test_edge_cases():
    """Bad token ids reject (status 1); NaN / +inf / all -inf rows make the
    sequence invalid (status 2, outputs -1); -inf entries are masked tokens;
    a rejection where p == q leaves zero residual mass: drawn from p
    (status 8)."""
    B, gamma, V = 8, 3, 300
    c = synth.linear_case(B, gamma, V, torch.float32, 1.0, seed=9)
    tg, dr, tk = c.target.clone(), c.draft.clone(), c.tokens.clone()
    tk[0, 1] = V + 5           # bad token at position 1
    tk[1, 0] = -1
    tg[2, 0, 17] = float("nan")
    dr[3, 0, 5] = float("inf")
    tg[4, 0, :] = -float("inf")
    tg[5, :, ::2] = -float("inf")   # masked half of the vocabulary
    dr[5, :, ::2] = -float("inf")
    tk[5] = 1
    dr[6] = tg[6, :gamma]      # identical rows, then a bad token
    tk[6, 0] = V
    edge = synth.LinearCase(tg, dr, tk, c.uniforms, 1.0)
    to_device(edge)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = run(edge, status=st)
    o = linear_oracle(edge)
    compare(g, o)
    assert np.array_equal(host(g["n"])[2:5], [-1, -1, -1])
    assert np.all(host(g["tokens"])[2:5] == -1)
    assert int(st.item()) == int(np.bitwise_or.reduce(o["status"]))
    assert o["status"][6] & oracle.ST_ZERO_MASS
    # greedy with a bad token: a plain mismatch
    edge.T = 0.0
    compare(run(edge), linear_oracle(edge))


def test_emitted_token_law_on_gpu():
    """Chi-square of the first emitted token against p over 1e6 GPU trials
    (V = 8, a poor drafter), the invariance of section 2.1."""
    rng = np.random.default_rng(3)
    V, B = 8, 1_000_000
    zt = rng.normal(0, 2, V).astype(np.float32)
    zd = rng.normal(0, 2, V).astype(np.float32)
    p = np.exp(zt - zt.max()); p /= p.sum()
    tg = torch.from_numpy(np.stack([zt, zt])).expand(B, 2, V).contiguous()
    dr = torch.from_numpy(zd[None]).expand(B, 1, V).contiguous()
    g = torch.Generator().manual_seed(4)
    x = synth.gumbel_argmax(dr.double(), 1.0, g)[..., 0]
    u = torch.from_numpy(synth.uniforms(5, (B, 2)))
    out = api.verify_linear(tg.cuda(), dr.cuda(), x.cuda(), u.cuda(), 1.0)
    first = host(out["tokens"][:, 0])
    cnt = np.bincount(first, minlength=V)
    stat = ((cnt - B * p) ** 2 / (B * p)).sum()
    assert stats.chi2.sf(stat, V - 1) > 1e-4


def test_flagged_fractions():
    """Over 20000 sequences of the tiny workload (about 45000 accept tests):
    accept tests within 1e-5 of their threshold stay below 1e-4 of the tests
    made; every other sequence matches exactly, and near-boundary final
    draws (counted) stay inside the oracle's admissible range and almost
    always equal its token."""
    c = to_device(synth.linear_case(20000, 4, 1000, torch.float32, 1.0,
                                    seed=77, sigma_t=2.0, sigma_d=1.0))
    r = compare(run(c), linear_oracle(c))
    assert r["tests"] > 40000
    assert r["tests_flagged"] / r["tests"] < 1e-4
    assert r["cdf_diff"] <= max(2, r["cdf_flagged"] // 20)
