"""Parity of sd_verify_kcand_trie (K candidates verified as one token tree;
CUDA, through the C ABI) with the oracle (its own tree construction, dense
node rows gathered on the host, the literal tree walk): small and odd
sizes, many repeated draws, gamma 0, K = 1 against the linear verify, the
kcand workload's shape on sampled sequences, invalid inputs, and the
emitted tokens' law on the GPU."""
import numpy as np
import pytest
import torch
from scipy import stats

import oracle
from speculative_decoding_verification_temperature_gb300 import api, synth
from tests.parity import (assert_flag_fraction, compare, host,
                          oracle_over_threads, to_device)
from tests.test_oracle_pins import _trie_law_case, softmax

pytestmark = pytest.mark.gpu


def tr_oracle(c, idx=None):
    sel = slice(None) if idx is None else idx
    return oracle.verify_kcand_trie(
        synth.host_logits(c.target[sel]),
        None if c.T == 0 else synth.host_logits(c.draft[sel]),
        host(c.tokens[sel]), host(c.uniforms[sel]), c.T)


def run(c, **kw):
    return api.verify_kcand_trie(c.target, None if c.T == 0 else c.draft,
                                 c.tokens, c.uniforms, c.T, **kw)


@pytest.mark.parametrize("T", [0.0, 0.6, 1.0])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("K,gamma,V", [(1, 5, 300), (3, 4, 1001),
                                       (8, 6, 5000), (8, 0, 700),
                                       (5, 1, 64), (32, 3, 96)])
def test_small_cases(T, dtype, K, gamma, V):
    c = to_device(synth.kcand_case(40, K, gamma, V, dtype, T,
                                   seed=K * 101 + V, sigma_t=2.0, sigma_d=1.0,
                                   sigma_k=0.7))
    compare(run(c), tr_oracle(c), extra_equal=("k",))


def test_many_repeated_draws():
    """Peaked marginals (sigma 4 over 64 tokens) and K = 16: most draws
    repeat an earlier candidate's token under the same prefix."""
    c = to_device(synth.kcand_case(64, 16, 5, 64, torch.float32, 1.0,
                                   seed=77, sigma_t=4.0, sigma_d=0.5,
                                   sigma_k=0.2))
    o = tr_oracle(c)
    assert o["trie"]["is_dup"].mean() > 0.3
    compare(run(c), o, extra_equal=("k",))


def test_one_candidate_equals_linear():
    c = to_device(synth.kcand_case(64, 1, 6, 2000, torch.bfloat16, 1.0,
                                   seed=4))
    g = run(c)
    gl = api.verify_linear(c.target[:, 0].contiguous(), c.draft,
                           c.tokens[:, 0].contiguous(),
                           c.uniforms[:, 0].contiguous(), 1.0)
    assert torch.equal(g["n"], gl["n"]) and torch.equal(g["tokens"],
                                                        gl["tokens"])
    assert torch.all(g["k"] == 0)


def test_kcand_workload_every_sequence():
    """B=64, K=8, gamma=16, V=152064 bf16, T=1, full size on the device:
    all 64 candidate trees against the oracle (host threads)."""
    c = synth.kcand(0, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = run(c, status=st)
    assert int(st.item()) & ~api.DEV_ZERO_MASS == 0
    t, d = synth.host_logits(c.target), synth.host_logits(c.draft)
    tk, u = host(c.tokens), host(c.uniforms)

    def part(lo, hi):
        o = oracle.verify_kcand_trie(t[lo:hi], d[lo:hi], tk[lo:hi],
                                     u[lo:hi], 1.0)
        o.pop("trie")
        return o
    r = compare(g, oracle_over_threads(part, 64), extra_equal=("k",))
    assert r["seqs"] == 64
    assert_flag_fraction(r)


def test_invalid_rows_and_tokens():
    c = synth.kcand_case(6, 3, 4, 500, torch.float32, 1.0, seed=31)
    c.target[1, 0, 0, 5] = float("nan")
    c.draft[2, 0, 9] = float("inf")
    c.tokens[3, 0, 0] = 10**6  # tried first under the root
    c = to_device(c)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    compare(run(c, status=st), tr_oracle(c), extra_equal=("k",))
    s = int(st.item())
    assert s & api.DEV_NONFINITE and s & api.DEV_BAD_TOKEN


def test_emitted_tokens_law_on_gpu():
    """K = 4 iid candidates, target rows depending on the prefix only: the
    first emitted token follows p_0 and the second, after an accepted first
    token a, follows P1[a] (chi-square, 3e5 sequences)."""
    B = 300_000
    z0, Z1, target, draft, x, U = _trie_law_case(B, 151)
    g = api.verify_kcand_trie(torch.from_numpy(target).cuda(),
                              torch.from_numpy(draft).cuda(),
                              torch.from_numpy(x).cuda(),
                              torch.from_numpy(U).cuda(), 1.0)
    V = len(z0)
    t0 = host(g["tokens"][:, 0])
    p0 = softmax(z0)
    stat = ((np.bincount(t0, minlength=V) - B * p0) ** 2 / (B * p0)).sum()
    assert stats.chi2.sf(stat, V - 1) > 1e-4
    n = host(g["n"])
    a, b = t0[n >= 1], host(g["tokens"][:, 1])[n >= 1]
    na = np.bincount(a, minlength=V)
    exp = (na[:, None] * np.stack([softmax(Z1[i]) for i in range(V)])).ravel()
    cnt = np.bincount(a * V + b, minlength=V * V)
    keep = exp > 0
    stat = ((cnt[keep] - exp[keep]) ** 2 / exp[keep]).sum()
    assert stats.chi2.sf(stat, keep.sum() - V) > 1e-4
