"""Pins of the fp64 oracle against what the pages and mathematics fix.

None of these re-types the oracle's arithmetic: each checks a closed form,
an invariant, a worked example, a brute-force enumeration or a statistical
law that a dropped term, a wrong sign, a wrong index or a swapped operand in
the oracle would break (tests/test_oracle_mutants.py plants such mistakes
and checks that these pins catch them).
"""
import itertools
import math

import numpy as np
import pytest
from scipy import stats

import oracle
from speculative_decoding_verification_temperature_gb300 import synth

P_MIN = 1e-4  # chi-square p-value floor (seeds are fixed: deterministic)


# ---------------------------------------------------------------- helpers
def softmax(z, T=1.0):
    z = np.asarray(z, np.float64) / T
    e = np.exp(z - z.max())
    return e / e.sum()


def draw_from(p, n, seed):
    """n iid draws from the probability vector p (Gumbel-max, numpy)."""
    rng = np.random.default_rng(seed)
    g = -np.log(-np.log(rng.random((n, len(p))).clip(1e-300)))
    with np.errstate(divide="ignore"):
        return np.argmax(np.log(p)[None, :] + g, axis=1).astype(np.int32)


def chi2_p(counts, probs):
    counts = np.asarray(counts, np.float64)
    probs = np.asarray(probs, np.float64)
    keep = probs > 0
    assert counts[~keep].sum() == 0, "mass on a zero-probability outcome"
    exp = probs[keep] * counts.sum()
    stat = ((counts[keep] - exp) ** 2 / exp).sum()
    return stats.chi2.sf(stat, keep.sum() - 1)


def f32(x):
    """The float32 value the oracle will see, back in float64."""
    return np.asarray(x, np.float32).astype(np.float64)


def tile_rows(rows, B):
    rows = np.asarray(rows, np.float32)
    return np.ascontiguousarray(np.broadcast_to(rows, (B,) + rows.shape))


# ------------------------------------------- "01 · Draft-then-verify" 2.2
def test_beta_closed_form_and_empirical_accept_rate():
    """beta = sum min(p, q) = 1 - TV (section 2.2); the oracle's empirical
    acceptance of position 0, with x ~ q, is beta within 5 sigma, and the
    residual mass equals 1 - beta (2.1 derivation)."""
    rng = np.random.default_rng(1)
    V, B = 8, 1_000_000
    zt = f32(rng.normal(0, 1.5, V))
    zd = f32(zt + rng.normal(0, 1.0, V))
    p, q = softmax(zt), softmax(zd)
    beta = np.minimum(p, q).sum()
    assert abs(beta - (1 - 0.5 * np.abs(p - q).sum())) < 1e-12
    x = draw_from(q, B, 2)[:, None]
    u = synth.uniforms(3, (B, 2))
    target = tile_rows([zt, zt], B)
    draft = tile_rows([zd], B)
    out = oracle.verify_linear(target, draft, x, u, 1.0)
    rate = (out["n"] == 1).mean()
    sd = math.sqrt(beta * (1 - beta) / B)
    assert abs(rate - beta) < 5 * sd
    # one sequence with out_resid: residual weights sum to 1 - beta before
    # normalisation, i.e. the normalised residual times (1-beta) is max(0,p-q)
    o1 = oracle.verify_linear(target[:1], draft[:1], np.array([[0]]),
                              np.array([[0.999999, 0.5]], np.float32), 1.0,
                              want_resid=True)
    if o1["n"][0] == 0:
        np.testing.assert_allclose(o1["resid"][0] * (1 - beta),
                                   np.maximum(0, p - q), atol=1e-12)


# -------------------------------- section 2.1 invariance P_alg(x) = p(x)
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_first_token_marginal_is_p(T):
    """The emitted token of a gamma = 1 round is distributed as p_1 for any
    q (section 2.1, distribution invariance).  Chi-square over 1e6 trials,
    V = 8."""
    rng = np.random.default_rng(11)
    V, B = 8, 1_000_000
    zt = rng.normal(0, 2.0, V)
    zd = rng.normal(0, 2.0, V)  # a poor drafter: q far from p
    p, q = softmax(zt, T), softmax(zd, T)
    x = draw_from(q, B, 12)[:, None]
    out = oracle.verify_linear(tile_rows([zt, zt + 5], B), tile_rows([zd], B),
                               x, synth.uniforms(13, (B, 2)), T)
    first = out["tokens"][:, 0]
    assert chi2_p(np.bincount(first, minlength=V), p) > P_MIN


def test_second_token_conditional_with_prefix_dependent_target():
    """Target rows depend on the prefix: p_2 = p(. | x_1).  Given that the
    first emitted token is a draft a that was accepted, the second emitted
    token is distributed as p(. | a) (2.1 applied at position 2, 2.3 prefix
    structure)."""
    rng = np.random.default_rng(21)
    V, B = 6, 1_000_000
    z1 = rng.normal(0, 1.5, V)
    cond = rng.normal(0, 1.5, (V, V))          # row a: logits of p(. | a)
    q1 = softmax(z1 + rng.normal(0, 0.7, V))
    zq1 = np.log(q1)
    zq2 = cond + rng.normal(0, 0.7, (V, V))    # q(. | a)
    x1 = draw_from(q1, B, 22)
    x2 = np.empty(B, np.int32)
    for a in range(V):
        idx = np.nonzero(x1 == a)[0]
        x2[idx] = draw_from(softmax(zq2[a]), len(idx), 23 + a)
    target = np.empty((B, 3, V), np.float32)
    target[:, 0] = z1
    target[:, 1] = cond[x1]
    target[:, 2] = 0.0
    draft = np.empty((B, 2, V), np.float32)
    draft[:, 0] = zq1
    draft[:, 1] = zq2[x1]
    out = oracle.verify_linear(target, draft, np.stack([x1, x2], 1),
                               synth.uniforms(24, (B, 3)), 1.0)
    assert chi2_p(np.bincount(out["tokens"][:, 0], minlength=V),
                  softmax(z1)) > P_MIN
    sel = out["n"] >= 1
    for a in range(V):
        m = sel & (out["tokens"][:, 0] == a)
        if m.sum() < 20000:
            continue
        assert chi2_p(np.bincount(out["tokens"][m, 1], minlength=V),
                      softmax(cond[a])) > P_MIN


# ------------------------------------------------ brute-force enumeration
def enumerate_first_token(zt, zq, gamma):
    """Exact distribution of the first emitted token of one round, by
    enumerating every draft x in V^gamma and every accept/reject branch.
    Rows do not depend on the prefix here.  Written from section 2.1: a
    token accepted at position 1 is emitted first; if position 1 rejects,
    the correction from norm(max(0, p1 - q1)) is emitted first."""
    p, q = softmax(zt[0]), softmax(zq[0])
    V = len(p)
    dist = np.zeros(V)
    for xs in itertools.product(range(V), repeat=gamma):
        w = np.prod([softmax(zq[i])[xs[i]] for i in range(gamma)])
        acc = min(1.0, p[xs[0]] / q[xs[0]])
        dist[xs[0]] += w * acc
        res = np.maximum(0, p - q)
        if res.sum() > 0:
            dist += w * (1 - acc) * res / res.sum()
    return dist


def enumerate_outcomes(zt, zq, gamma):
    """Exact law of (n accepted, emitted tuple) of one round (fixed rows),
    by enumeration over drafts and branches."""
    V = zt.shape[1]
    P = [softmax(zt[i]) for i in range(gamma + 1)]
    Q = [softmax(zq[i]) for i in range(gamma)]
    law = {}
    for xs in itertools.product(range(V), repeat=gamma):
        w = np.prod([Q[i][xs[i]] for i in range(gamma)])
        reach = w
        for i in range(gamma):
            acc = min(1.0, P[i][xs[i]] / Q[i][xs[i]])
            res = np.maximum(0, P[i] - Q[i])
            if res.sum() > 0 and acc < 1:
                for t in range(V):
                    key = (i, xs[:i] + (t,))
                    law[key] = law.get(key, 0) + reach * (1 - acc) * \
                        res[t] / res.sum()
            reach *= acc
        for t in range(V):
            key = (gamma, xs + (t,))
            law[key] = law.get(key, 0) + reach * P[gamma][t]
    return law


@pytest.mark.parametrize("V,gamma", [(3, 3), (5, 2), (6, 1)])
def test_bruteforce_enumeration(V, gamma):
    """Enumeration gives p_1 exactly for the first token (to 1e-12); the
    oracle's sampled (n, tokens) frequencies follow the enumerated law."""
    rng = np.random.default_rng(100 + V)
    zt = rng.normal(0, 1.2, (gamma + 1, V))
    zq = zt[:gamma] + rng.normal(0, 1.0, (gamma, V))
    first = enumerate_first_token(zt, zq, gamma)
    np.testing.assert_allclose(first, softmax(zt[0]), atol=1e-12)
    law = enumerate_outcomes(zt, zq, gamma)
    assert abs(sum(law.values()) - 1) < 1e-12
    B = 400_000
    xs = np.stack([draw_from(softmax(zq[i]), B, 200 + i)
                   for i in range(gamma)], 1)
    out = oracle.verify_linear(tile_rows(zt, B), tile_rows(zq, B), xs,
                               synth.uniforms(300 + V, (B, gamma + 1)), 1.0)
    keys = list(law)
    index = {k: i for i, k in enumerate(keys)}
    counts = np.zeros(len(keys))
    for n, toks in zip(out["n"], out["tokens"]):
        counts[index[(int(n), tuple(int(t) for t in toks[:n + 1]))]] += 1
    assert chi2_p(counts, [law[k] for k in keys]) > P_MIN


# ------------------------------- accepted-length law (iid alpha) 3 / SpecBranch
def test_truncated_geometric_length_law():
    """With identical (p, q) at every position the accepted count is
    truncated-geometric: P(n=k) = (1-a) a^k for k < gamma, a^gamma at gamma
    (SpecBranch, background); the mean emitted count is
    (1 - a^{gamma+1}) / (1 - a) ("01 · Draft-then-verify", section 3)."""
    rng = np.random.default_rng(31)
    V, gamma, B = 8, 5, 1_000_000
    zt = rng.normal(0, 1.5, V)
    zd = zt + rng.normal(0, 0.8, V)
    p, q = softmax(zt), softmax(zd)
    a = np.minimum(p, q).sum()
    xs = np.stack([draw_from(q, B, 40 + i) for i in range(gamma)], 1)
    out = oracle.verify_linear(tile_rows([zt] * (gamma + 1), B),
                               tile_rows([zd] * gamma, B), xs,
                               synth.uniforms(41, (B, gamma + 1)), 1.0)
    law = [(1 - a) * a ** k for k in range(gamma)] + [a ** gamma]
    assert chi2_p(np.bincount(out["n"], minlength=gamma + 1), law) > P_MIN
    mean = (out["n"] + 1).mean()
    expect = (1 - a ** (gamma + 1)) / (1 - a)
    sd = np.sqrt(np.sum(np.array(law) * (np.arange(gamma + 1) + 1) ** 2)
                 - expect ** 2) / np.sqrt(B)
    assert abs(mean - expect) < 5 * sd


# ------------------------------------------------------ greedy (2.2)
@pytest.mark.parametrize("T", [1.0, 0.7, 0.0])
def test_softmax_shift_invariance(T):
    """The verify reads p = softmax(z / T) and q = softmax(z_d / T) only
    ("01 · Draft-then-verify" section 1), and a softmax does not change
    when every logit of its row moves by the same constant; the greedy rule
    compares argmaxes, which do not change either.  On a 2^-10 grid the
    logits stay exact in fp32 after shifts of -1024, 1024 or 4096, and the
    shift cancels exactly in (z + c) - (m + c), so the oracle must return
    the same counts, tokens and probabilities bit for bit, row by row.  (A
    softmax without its max subtraction overflows at exp(1024).)"""
    rng = np.random.default_rng(2024)
    B, gamma, V = 48, 4, 50
    grid = lambda x: np.round(x * 1024.0) / 1024.0
    zt = grid(rng.normal(0.0, 3.0, (B, gamma + 1, V)))
    zd = grid(zt[:, :gamma] + rng.normal(0.0, 1.0, (B, gamma, V)))
    x = rng.integers(0, V, (B, gamma)).astype(np.int32)
    # draft tokens that are often accepted: the draft row's argmax
    x[::2] = np.argmax(zd[::2], axis=2)
    u = ((rng.integers(0, 2**23, (B, gamma + 1)) + 0.5) / 2**23).astype(
        np.float32)
    ct = rng.choice([-1024.0, 1024.0, 4096.0], (B, gamma + 1, 1))
    cd = rng.choice([-1024.0, 1024.0, 4096.0], (B, gamma, 1))
    f = lambda z: np.ascontiguousarray(z, np.float32)
    assert np.array_equal(f(zt + ct).astype(np.float64), zt + ct)
    assert np.array_equal(f(zd + cd).astype(np.float64), zd + cd)
    d0 = None if T == 0 else f(zd)
    d1 = None if T == 0 else f(zd + cd)
    a = oracle.verify_linear(f(zt), d0, x, u, T)
    b = oracle.verify_linear(f(zt + ct), d1, x, u, T)
    assert np.all(a["n"] >= 0) and 0 < a["n"].sum() < B * gamma
    for k in ("n", "tokens", "prob"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


def _linear_case(seed, B=40, gamma=5, V=60):
    rng = np.random.default_rng(seed)
    zt = rng.normal(0.0, 2.0, (B, gamma + 1, V)).astype(np.float32)
    zd = (zt[:, :gamma] + rng.normal(0.0, 1.0, (B, gamma, V))).astype(
        np.float32)
    x = np.argmax(zd, axis=2).astype(np.int32)
    x[::3] = rng.integers(0, V, (len(x[::3]), gamma))
    u = ((rng.integers(0, 2**23, (B, gamma + 1)) + 0.5) / 2**23).astype(
        np.float32)
    return zt, zd, x, u


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_rows_after_the_decision_are_never_read(T):
    """Algorithm 1 ("01 · Draft-then-verify" section 1) stops at the first
    rejection: what the rows after it hold cannot change the round.  Those
    rows are overwritten with NaN and +inf (which would invalidate a round
    that read them) and every output stays the same; a NaN in target row n,
    which the round does read, invalidates it (n = -1, every token -1,
    status bit 2: the reading for unusable rows)."""
    zt, zd, x, u = _linear_case(7)
    B, G1, V = zt.shape
    gamma = G1 - 1
    d = None if T == 0 else zd
    a = oracle.verify_linear(zt, d, x, u, T)
    n = a["n"]
    assert np.all(n >= 0) and np.any(n < gamma) and np.any(n > 0)
    zt2, zd2 = zt.copy(), zd.copy()
    for b in range(B):
        zt2[b, n[b] + 1:, ::2] = np.nan
        zt2[b, n[b] + 1:, 1::2] = np.inf
        zd2[b, n[b] + 1:] = np.nan
    b2 = oracle.verify_linear(zt2, None if T == 0 else zd2, x, u, T)
    for k in ("n", "tokens", "prob", "status"):
        np.testing.assert_array_equal(a[k], b2[k], err_msg=k)
    zt3 = zt.copy()
    zt3[np.arange(B), n, 3] = np.nan
    c = oracle.verify_linear(zt3, d, x, u, T)
    assert np.all(c["n"] == -1) and np.all(c["tokens"] == -1)
    assert np.all(c["status"] & 2)


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_minus_infinity_is_a_token_of_probability_zero(T):
    """A -inf logit is a masked token (the reading for masked tokens): the
    round equals the one where that logit is so low that exp underflows to
    exactly 0 in double, and a masked draft token is never accepted."""
    zt, zd, x, u = _linear_case(8)
    B, G1, V = zt.shape
    mask = np.zeros_like(zt, bool)
    mask[:, :, V // 2:] = True
    mask[:, :, 0] = False             # keep one low-id token unmasked
    x[:, 0] = V - 1                   # the first draft token is masked
    low = np.float32(-1e30)           # exp((-1e30 - m) / T) == 0.0 exactly
    zinf, zlow = zt.copy(), zt.copy()
    zinf[mask] = -np.inf
    zlow[mask] = low
    a = oracle.verify_linear(zinf, zd, x, u, T)
    b = oracle.verify_linear(zlow, zd, x, u, T)
    for k in ("n", "tokens", "prob", "status"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    assert np.all(a["n"] == 0) and np.all(a["status"] == 0)
    assert np.all(a["tokens"][:, 0] < V // 2)  # drawn among unmasked ones


def test_greedy_is_id_equality_with_argmax():
    """T = 0: accept iff the draft id equals argmax p (section 2.2), ties to
    the lowest index; the correction/bonus is argmax of row n.  Compared with
    numpy's argmax on the same bf16 values, including rows with ties."""
    rng = np.random.default_rng(51)
    B, gamma, V = 4000, 4, 40
    z = rng.integers(-6, 7, (B, gamma + 1, V)).astype(np.float32)  # ties
    import torch
    bits = synth.bf16_bits(torch.from_numpy(z).to(torch.bfloat16))
    am = np.argmax(z, axis=2)
    # drafts: the argmax with probability 0.7 each, else a random id
    xs = np.where(rng.random((B, gamma)) < 0.7, am[:, :gamma],
                  rng.integers(0, V, (B, gamma))).astype(np.int32)
    out = oracle.verify_linear(bits, None, xs,
                               np.full((B, gamma + 1), 0.5, np.float32), 0.0)
    match = xs == am[:, :gamma]
    n_ref = np.where(match.all(1), gamma, np.argmin(match, axis=1))
    np.testing.assert_array_equal(out["n"], n_ref)
    t_ref = am[np.arange(B), n_ref]
    np.testing.assert_array_equal(out["tokens"][np.arange(B), n_ref], t_ref)
    assert np.all(out["prob"] == 1.0)
    assert np.all(np.isinf(out["margin"]))


# ------------------------------------------ worked examples (golden files)
def _golden(name):
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", name)
    with open(path) as f:
        return json.load(f)


def test_worked_residual_examples():
    """Hand-worked single-step examples of section 2.1 (accept probability
    min(1, p/q), residual norm(max(0, p - q))), stored in
    tests/golden/single_step_examples.json."""
    for ex in _golden("single_step_examples.json")["cases"]:
        p = np.array(ex["p"])
        q = np.array(ex["q"])
        tgt = np.log(np.stack([p, p])).astype(np.float32)[None]
        drf = np.log(q).astype(np.float32)[None, None]
        x = np.array([[ex["x"]]], np.int32)
        for r, u, n, t in ex["draws"]:
            o = oracle.verify_linear(tgt, drf, x,
                                     np.array([[r, u]], np.float32), 1.0,
                                     want_resid=True)
            assert o["n"][0] == n and o["tokens"][0, n] == t, (ex, r, u)
            if n == 0:
                np.testing.assert_allclose(o["resid"][0], ex["residual"],
                                           atol=1e-6)
            np.testing.assert_allclose(o["accept"][0, 0], ex["accept"],
                                       atol=1e-6)


# ----------------------------------------- kcand (SpecDiff-2 self-selection)
def test_kcand_one_candidate_equals_linear():
    c = synth.kcand_case(64, 1, 5, 300, T=1.0, seed=5)
    tg = synth.host_logits(c.target)
    dr = synth.host_logits(c.draft)
    ok = oracle.verify_kcand(tg, dr, c.tokens.numpy(), c.uniforms.numpy(), 1.0)
    ol = oracle.verify_linear(tg[:, 0], dr, c.tokens.numpy()[:, 0],
                              c.uniforms.numpy()[:, 0], 1.0)
    np.testing.assert_array_equal(ok["n"], ol["n"])
    np.testing.assert_array_equal(ok["tokens"], ol["tokens"])
    np.testing.assert_array_equal(ok["prob"], ol["prob"])
    assert np.all(ok["k"] == 0)


def test_kcand_selection_is_max_streak_lowest_k():
    c = synth.kcand_case(200, 6, 6, 200, T=1.0, seed=6, sigma_k=1.0)
    o = oracle.verify_kcand(synth.host_logits(c.target),
                            synth.host_logits(c.draft), c.tokens.numpy(),
                            c.uniforms.numpy(), 1.0)
    npc = o["n_per_cand"]
    np.testing.assert_array_equal(o["n"], npc.max(1))
    np.testing.assert_array_equal(o["k"], np.argmax(npc, axis=1))
    toks = c.tokens.numpy()
    for b in range(200):
        n, k = o["n"][b], o["k"][b]
        np.testing.assert_array_equal(o["tokens"][b, :n], toks[b, k, :n])
        assert o["tokens"][b, n] >= 0 and np.all(o["tokens"][b, n + 1:] == -1)


def test_kcand_max_streak_law_bruteforce():
    """Candidates are independent given the marginals, so with fixed rows
    P(n_sel >= m) = 1 - prod_k (1 - P(n_k >= m)), P(n_k >= m) = prod_{j<m}
    beta_{k,j}, beta = sum min(p, q) (section 2.2)."""
    rng = np.random.default_rng(61)
    V, K, gamma, B = 6, 3, 3, 300_000
    zq = rng.normal(0, 1.2, (gamma, V))
    zt = zq[None, :, :] + rng.normal(0, 0.9, (K, gamma, V))
    zt = np.concatenate([zt, rng.normal(0, 1, (K, 1, V))], 1)
    beta = np.array([[np.minimum(softmax(zt[k, j]), softmax(zq[j])).sum()
                      for j in range(gamma)] for k in range(K)])
    xs = np.stack([np.stack([draw_from(softmax(zq[j]), B, 70 + 10 * k + j)
                             for j in range(gamma)], 1) for k in range(K)], 1)
    o = oracle.verify_kcand(tile_rows(zt, B), tile_rows(zq, B), xs,
                            synth.uniforms(71, (B, K, gamma + 1)), 1.0)
    for m in range(1, gamma + 1):
        pk = np.prod(beta[:, :m], axis=1)
        expect = 1 - np.prod(1 - pk)
        got = (o["n"] >= m).mean()
        assert abs(got - expect) < 5 * math.sqrt(expect * (1 - expect) / B)


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_kcand_rows_after_each_scan_are_never_read(T):
    """Each candidate is scanned with the linear rule up to its first
    rejection (SpecDiff-2, "core method"), and only the selected candidate
    draws: its row at position n, or its bonus row gamma when its streak is
    complete, and the shared draft row n.  Every other row is overwritten
    with NaN and the round stays the same."""
    import torch
    c = synth.kcand_case(16, 4, 5, 200, torch.float32, 1.0, seed=9,
                         sigma_t=1.0, sigma_d=0.4, sigma_k=0.3)
    zt, zd = synth.host_logits(c.target), synth.host_logits(c.draft)
    x, u = c.tokens.numpy(), c.uniforms.numpy()
    B, K, G1, V = zt.shape
    gamma = G1 - 1
    o = oracle.verify_kcand(zt, zd, x, u, T)
    npc, n, ks = o["n_per_cand"], o["n"], o["k"]
    assert np.all(n >= 0) and np.any(n > 0) and np.any(n < gamma)
    zt2, zd2 = np.full_like(zt, np.nan), np.full_like(zd, np.nan)
    for b in range(B):
        for k in range(K):
            last = min(int(npc[b, k]), gamma - 1)
            zt2[b, k, :last + 1] = zt[b, k, :last + 1]
        zt2[b, ks[b], n[b]] = zt[b, ks[b], n[b]]
        if T > 0:
            zd2[b, :min(int(n[b]), gamma - 1) + 1] = \
                zd[b, :min(int(n[b]), gamma - 1) + 1]
    o2 = oracle.verify_kcand(zt2, zd2, x, u, T)
    for k in ("n", "k", "n_per_cand", "tokens", "prob", "status"):
        np.testing.assert_array_equal(o[k], o2[k], err_msg=k)


def test_kcand_selection_bias_counterexample():
    """Longest-streak selection is not lossless for K > 1: V = 2,
    p = (1/2, 1/2), both candidates draft token 0 with q = delta_0.  Each
    candidate accepts with probability 1/2, the selection keeps an accepted
    one unless both reject, so the first token is 0 with probability 3/4."""
    B = 400_000
    zt = np.zeros((2, 2, 2), np.float32)             # [K, gamma+1, V]
    zq = np.array([[0.0, -np.inf]], np.float32)      # q = delta_0
    xs = np.zeros((B, 2, 1), np.int32)
    o = oracle.verify_kcand(tile_rows(zt, B), tile_rows(zq, B), xs,
                            synth.uniforms(81, (B, 2, 2)), 1.0)
    frac0 = (o["tokens"][:, 0] == 0).mean()
    assert abs(frac0 - 0.75) < 5 * math.sqrt(0.75 * 0.25 / B)


# ------------------------------------------------------------- tree
def chain_tree_from_linear(tg, dr, xs, u):
    """Rearrange a linear case as a one-child-per-node tree."""
    B, G1, V = tg.shape
    gamma = G1 - 1
    ttree = tg
    dtree = np.concatenate([dr, np.zeros((B, 1, V), dr.dtype)], 1)
    parent = np.tile(np.arange(-1, gamma, dtype=np.int32), (B, 1))
    ntok = np.concatenate([np.full((B, 1), -1, np.int32), xs], 1)
    U = np.concatenate([u[:, gamma:gamma + 1], u[:, :gamma]], 1)
    return ttree, dtree, parent, ntok, U


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_tree_chain_equals_linear(T):
    c = synth.linear_case(300, 5, 257, T=T, seed=91)
    tg, dr = synth.host_logits(c.target), synth.host_logits(c.draft)
    xs, u = c.tokens.numpy(), c.uniforms.numpy()
    ol = oracle.verify_linear(tg, dr, xs, u, T)
    ot = oracle.verify_tree(*chain_tree_from_linear(tg, dr, xs, u), T)
    np.testing.assert_array_equal(ot["n"], ol["n"])
    np.testing.assert_array_equal(ot["tokens"][:, :6], ol["tokens"])
    # the tree renormalises before drawing, the chain after: same value up
    # to the last bits
    np.testing.assert_allclose(ot["prob"], ol["prob"], rtol=1e-12)
    for b in range(300):
        np.testing.assert_array_equal(ot["nodes"][b, :ol["n"][b]],
                                      np.arange(1, ol["n"][b] + 1))


def test_tree_iid_siblings_lossless():
    """Siblings drawn iid from the parent's q, tried in turn with
    p <- norm(max(0, p - q)) after each rejection, keep the emitted token's
    marginal equal to p (the 2.1 argument applied repeatedly).  Chi-square,
    V = 8, three siblings under the root, 1e6 trials."""
    rng = np.random.default_rng(95)
    V, S, B = 8, 3, 1_000_000
    zt = rng.normal(0, 1.5, V)
    zq = zt + rng.normal(0, 1.2, V)
    N = S + 1
    tg = tile_rows([zt] + [rng.normal(0, 1, V)] * S, B)
    dr = tile_rows([zq] + [np.zeros(V)] * S, B)
    parent = np.tile(np.array([-1] + [0] * S, np.int32), (B, 1))
    kids = np.stack([draw_from(softmax(zq), B, 96 + s) for s in range(S)], 1)
    ntok = np.concatenate([np.full((B, 1), -1, np.int32), kids], 1)
    o = oracle.verify_tree(tg, dr, parent, ntok,
                           synth.uniforms(97, (B, N)), 1.0)
    assert chi2_p(np.bincount(o["tokens"][:, 0], minlength=V),
                  softmax(zt)) > P_MIN


def test_tree_scalar_c_closed_form():
    """The iterated residual p <- norm(max(0, p - q)) equals
    max(0, p - c_k q) / N_k with c_0 = 0, c_{k+1} = c_k + N_k and
    N_k = sum max(0, p - c_k q): the closed form the CUDA tree walk uses.
    Checked numerically in double against the literal iteration."""
    rng = np.random.default_rng(98)
    for _ in range(200):
        V = rng.integers(2, 60)
        p = softmax(rng.normal(0, 2, V))
        q = softmax(rng.normal(0, 2, V))
        it = p.copy()
        c = 0.0
        for _k in range(6):
            res = np.maximum(0, p - c * q)
            Nk = res.sum()
            if Nk <= 1e-12:
                break
            np.testing.assert_allclose(it, res / Nk, atol=1e-12)
            nxt = np.maximum(0, it - q)
            if nxt.sum() <= 1e-12:
                break
            it = nxt / nxt.sum()
            c = c + Nk


def test_tree_topk_sibling_counterexample():
    """Deterministic top-k siblings are not lossless: V = 2, q = (1/2, 1/2),
    p = (0.9, 0.1), children tokens 0 then 1: the first child has
    p/q = 1.8 and is always accepted, so the first token is always 0."""
    B = 10000
    zt = np.log(np.array([[0.9, 0.1], [0.5, 0.5], [0.5, 0.5]]))
    zq = np.zeros((3, 2))
    parent = np.tile(np.array([-1, 0, 0], np.int32), (B, 1))
    ntok = np.tile(np.array([-1, 0, 1], np.int32), (B, 1))
    o = oracle.verify_tree(tile_rows(zt, B), tile_rows(zq, B), parent, ntok,
                           synth.uniforms(99, (B, 3)), 1.0)
    assert np.all(o["tokens"][:, 0] == 0) and np.all(o["nodes"][:, 0] == 1)


@pytest.mark.parametrize("rule,T", [("sibling", 1.0), ("sibling", 0.0),
                                    ("det", 1.0)])
def test_tree_rows_off_the_path_are_never_read(rule, T):
    """The walk reads the target row of the root and of each accepted node
    and, under the sibling rule, the draft row of each of those that has
    children: the q their children were drafted from (PRESTO section 2.1;
    "01 · Draft-then-verify" section 2.1).  The deterministic-draft rule
    reads no draft row.  Every other row is overwritten with NaN and the
    round stays the same; a NaN in a visited node's target row makes it
    unusable (status bit 2)."""
    import torch
    c = synth.tree_case(12, 40, 300, torch.float32, 1.0, seed=5,
                        sigma_t=1.0, sigma_d=0.5, branch=4, max_depth=5)
    zt, zd = synth.host_logits(c.target), synth.host_logits(c.draft)
    par, tok, u = c.parent.numpy(), c.node_tokens.numpy(), c.uniforms.numpy()

    def run(a, d):
        if rule == "det":
            return oracle.verify_tree_det(a, par, tok, u, T)
        return oracle.verify_tree(a, d, par, tok, u, T)

    o = run(zt, zd)
    B = zt.shape[0]
    assert np.all(o["n"] >= 0) and np.any(o["n"] > 0)
    zt2, zd2 = np.full_like(zt, np.nan), np.full_like(zd, np.nan)
    for b in range(B):
        for v in [0] + [int(x) for x in o["nodes"][b, :o["n"][b]]]:
            zt2[b, v] = zt[b, v]
            if rule == "sibling" and T > 0 and np.any(par[b] == v):
                zd2[b, v] = zd[b, v]
    o2 = run(zt2, zd2)
    for k in ("n", "tokens", "nodes", "prob", "status"):
        np.testing.assert_array_equal(o[k], o2[k], err_msg=k)
    zt3 = zt.copy()
    last = [int(o["nodes"][b, o["n"][b] - 1]) if o["n"][b] else 0
            for b in range(B)]
    zt3[np.arange(B), last, 7] = np.nan
    o3 = run(zt3, zd)
    assert np.all(o3["n"] == -1) and np.all(o3["status"] & 2)


def test_tree_greedy_follows_argmax_child():
    c = synth.tree_case(20, 24, 50, dtype=__import__("torch").float32, T=0.0,
                        seed=100)
    tg = synth.host_logits(c.target)
    o = oracle.verify_tree(tg, synth.host_logits(c.draft), c.parent.numpy(),
                           c.node_tokens.numpy(), c.uniforms.numpy(), 0.0)
    par, tok = c.parent.numpy(), c.node_tokens.numpy()
    for b in range(20):
        cur, path = 0, []
        while True:
            a = int(np.argmax(tg[b, cur]))
            nxt = [v for v in range(1, 24) if par[b, v] == cur and
                   tok[b, v] == a]
            if not nxt:
                break
            cur = nxt[0]
            path.append(cur)
        assert o["n"][b] == len(path)
        np.testing.assert_array_equal(o["nodes"][b, :len(path)], path)
        assert o["tokens"][b, len(path)] == a


def test_tree_invalid_parent_flagged():
    c = synth.tree_case(3, 8, 30, dtype=__import__("torch").float32, seed=101)
    par = c.parent.numpy().copy()
    par[1, 5] = 6          # parent after child
    par[2, 0] = 0          # root with a parent
    o = oracle.verify_tree(synth.host_logits(c.target),
                           synth.host_logits(c.draft), par,
                           c.node_tokens.numpy(), c.uniforms.numpy(), 0.8)
    assert o["n"][0] >= 0 and o["status"][0] & oracle.ST_BAD_PARENT == 0
    for b in (1, 2):
        assert o["n"][b] == -1 and o["status"][b] & oracle.ST_BAD_PARENT


# ------------------------------------------------------- fan-out (Saguaro)
def bruteforce_fanout(K, budget, a, r):
    """Integer maximiser of the power-law hit rate sum_k P(k) (1 - F_k^-r),
    P(k) = (1-a) a^k for k < K and a^K for k = K (Definition 11, the capped
    geometric law of the verify length), by greedy marginal gain from
    F_k = 1 (the objective is separable and concave in each F_k)."""
    P = [(1 - a) * a ** k for k in range(K)] + [a ** K]
    F = [1] * (K + 1)
    for _ in range(budget - (K + 1)):
        gain = [P[k] * (F[k] ** -r - (F[k] + 1) ** -r) for k in range(K + 1)]
        F[int(np.argmax(gain))] += 1
    return F


def test_fanout_schedule_golden_and_theorem12():
    g = _golden("fanout_schedule.json")
    for case in g["cases"]:
        K, B, a, r = case["K"], case["budget"], case["a"], case["r"]
        F = oracle.fanout_schedule(K, B, a, r)
        assert F.sum() == B
        assert list(F) == case["F"]
        assert list(F) == bruteforce_fanout(K, B, a, r)
    # Theorem 12 ratios of the real-valued schedule: F_{k+1}/F_k =
    # a^{1/(1+r)}; the capped last position has the extra (1-a)^{-1/(1+r)}.
    # With a huge budget the rounding is negligible.
    K, a, r = 6, 0.7, 1.5
    F = oracle.fanout_schedule(K, 10 ** 7, a, r).astype(np.float64)
    ratio = a ** (1 / (1 + r))
    np.testing.assert_allclose(F[1:K] / F[:K - 1], ratio, rtol=1e-5)
    np.testing.assert_allclose(F[K] / F[K - 1],
                               ratio * (1 - a) ** (-1 / (1 + r)), rtol=1e-5)


def test_fanout_topk_against_stable_sort_and_ties():
    import torch
    rng = np.random.default_rng(111)
    B, K, V = 7, 3, 500
    z = rng.integers(-20, 20, (B, K + 1, V)).astype(np.float32) / 4  # ties
    z[0, 0, :] = 0.0
    z[0, 0, ::3] = -0.0                     # -0 equals +0
    F = np.array([5, 3, 0, 9], np.int32)
    for host in (z, synth.bf16_bits(torch.from_numpy(z).to(torch.bfloat16))):
        o = oracle.fanout_topk(host, F)
        off = 0
        for k in range(K + 1):
            for b in range(B):
                order = np.lexsort((np.arange(V), -z[b, k]))[:F[k]]
                np.testing.assert_array_equal(
                    o["tokens"][b, off:off + F[k]], order)
            off += F[k]


# --------------------------- Saguaro: cache hit of the verification outcome
def test_cache_hits_golden():
    """Hand-worked outcomes and caches (tests/golden/cache_hits.json)."""
    g = _golden("cache_hits.json")
    F = np.array(g["F"], np.int32)
    for c in g["cases"]:
        h = oracle.fanout_hits([c["n"]], [c["tokens"]], [c["fan_tokens"]], F)
        assert h[0] == c["hit"], c["why"]
    e = g["empty_position"]
    h = oracle.fanout_hits([e["n"]], [e["tokens"]], [e["fan_tokens"]],
                           np.array(e["F"], np.int32))
    assert h[0] == e["hit"], e["why"]


def test_cache_hit_rate_equals_top_f_mass_when_p_equals_q():
    """With identical target and draft rows every draft is accepted
    (p/q = 1), so the outcome is (gamma, t*) with t* ~ p_gamma, and the
    speculation cache of position gamma holds the top-F tokens of the draft
    row gamma = p_gamma's own top-F: the hit rate is the top-F mass of
    p_gamma.  The oracle's verify + fan-out + hit pipeline over 40000
    seeded rounds matches that mass within 5 sigma, for F = 1, 3 and V."""
    V, gamma, B = 12, 2, 40000
    rng = np.random.default_rng(21)
    rows = rng.normal(0.0, 1.5, (gamma + 1, V)).astype(np.float32)
    target = tile_rows(rows, B)
    draft = np.ascontiguousarray(target[:, :gamma])
    p_last = softmax(f32(rows[gamma]))
    x = np.stack([draw_from(softmax(f32(rows[j])), B, 100 + j)
                  for j in range(gamma)], axis=1)
    u = synth.uniforms(22, (B, gamma + 1))
    o = oracle.verify_linear(target, draft, x, u, 1.0)
    assert np.all(o["n"] == gamma)
    for Fl in (1, 3, V):
        F = np.array([1] * gamma + [Fl], np.int32)
        fan = oracle.fanout_topk(target, F)["tokens"]
        hit = oracle.fanout_hits(o["n"], o["tokens"], fan, F)
        mass = np.sort(p_last)[::-1][:Fl].sum()
        rate = hit.mean()
        sd = math.sqrt(max(mass * (1 - mass), 1e-12) / B)
        assert abs(rate - mass) <= 5 * sd + 1e-12, (Fl, rate, mass)


# ---------------- "01 · Draft-then-verify" 4: standardised (filtered) sampling
def filtered(z, T, top_k, top_p):
    """top_k / top_p filtered softmax(z / T) (the reading of section 4):
    top_k by (logit desc, index asc), then the smallest prefix whose mass,
    renormalised over the top_k, reaches top_p; renormalised."""
    z = np.asarray(z, np.float64)
    p = softmax(z, T)
    order = np.lexsort((np.arange(len(z)), -z))[:top_k]
    mk = p[order].sum()
    before = np.concatenate([[0.0], np.cumsum(p[order])[:-1]]) / mk
    keep = order[before < top_p] if top_p < 1.0 else order
    out = np.zeros_like(p)
    out[keep] = p[keep] / p[keep].sum()
    return out


@pytest.mark.parametrize("T,dtype", [(1.0, "f32"), (0.7, "bf16")])
def test_filtered_without_filter_equals_linear(T, dtype):
    """top_k = V and top_p = 1 keep every token: the filtered verify is the
    plain linear verify, output for output."""
    import torch
    c = synth.linear_case(300, 4, 37, torch.float32 if dtype == "f32"
                          else torch.bfloat16, T, seed=61, sigma_t=2.0,
                          sigma_d=1.0)
    t, d = synth.host_logits(c.target), synth.host_logits(c.draft)
    a = oracle.verify_linear(t, d, c.tokens.numpy(), c.uniforms.numpy(), T)
    b = oracle.verify_linear_filtered(t, d, c.tokens.numpy(),
                                      c.uniforms.numpy(), T, 37, 1.0)
    for k in ("n", "tokens", "cdf_lo", "cdf_hi"):
        np.testing.assert_array_equal(a[k], b[k], k)
    for k in ("prob", "margin_cdf"):  # the kept mass is 1 up to rounding
        np.testing.assert_allclose(a[k], b[k], rtol=1e-12, atol=1e-14)


def test_filtered_sampling_golden():
    """Hand-worked top-k / top-p cuts (tests/golden/filtered_sampling.json)
    seen through the bonus draw: with identical target and draft rows every
    draft is accepted, and uniforms placed inside each kept token's interval
    of the filtered CDF (index order) must draw that token with probability
    p_j / mass; kept-out tokens are never drawn."""
    g = _golden("filtered_sampling.json")
    p = np.array(g["p"])
    z = np.log(p).astype(np.float32)
    for c in g["cases"]:
        kept = c["kept"]
        pt = np.zeros_like(p)
        pt[kept] = p[kept] / c["mass"]
        cdf = np.cumsum(pt)
        us, want = [], []
        for j in kept:  # the middle of token j's interval
            us.append((cdf[j] - pt[j] / 2))
            want.append(j)
        B = len(us)
        rows = np.stack([z, z])  # gamma = 1: row 0 tested, row 1 bonus
        x = np.full((B, 1), kept[0], np.int32)
        u = np.zeros((B, 2), np.float32)
        u[:, 0] = 0.5
        u[:, 1] = np.array(us, np.float32)
        o = oracle.verify_linear_filtered(tile_rows(rows, B),
                                          tile_rows(rows[:1], B), x, u, 1.0,
                                          c["top_k"], c["top_p"])
        assert np.all(o["n"] == 1), c["why"]
        assert o["tokens"][:, 1].tolist() == want, c["why"]
        np.testing.assert_allclose(o["prob"], pt[want], rtol=1e-6,
                                   err_msg=c["why"])
    a = g["accept_case"]
    zt = np.log(np.array([a["p"], a["p"]])).astype(np.float32)
    zq = np.log(np.array([a["q"]])).astype(np.float32)
    o = oracle.verify_linear_filtered(zt[None], zq[None], [[a["x"]]],
                                      [[a["r"], a["u"]]], 1.0, a["top_k"],
                                      a["top_p"])
    assert o["n"][0] == a["n"] and o["tokens"][0, 0] == a["token"], a["why"]
    np.testing.assert_allclose(o["prob"][0], a["prob"], rtol=1e-6)


@pytest.mark.parametrize("top_k,top_p", [(5, 1.0), (8, 0.85), (4, 0.6)])
def test_filtered_first_token_marginal_is_filtered_p(top_k, top_p):
    """Drafts drawn from the filtered q~; the first emitted token follows
    the filtered p~ (chi-square over 400000 rounds), the lossless property
    section 4 asks of standardised sampling; tokens outside p~'s support
    never appear."""
    rng = np.random.default_rng(71 + top_k)
    V, gamma, B, T = 8, 2, 400_000, 0.8
    zt = rng.normal(0, 1.3, (gamma + 1, V))
    zq = zt[:gamma] + rng.normal(0, 0.9, (gamma, V))
    zt, zq = f32(zt), f32(zq)
    xs = np.stack([draw_from(filtered(zq[i], T, top_k, top_p), B, 80 + i)
                   for i in range(gamma)], 1)
    out = oracle.verify_linear_filtered(
        tile_rows(zt, B), tile_rows(zq, B), xs,
        synth.uniforms(90 + top_k, (B, gamma + 1)), T, top_k, top_p)
    first = out["tokens"][:, 0]
    p0 = filtered(zt[0], T, top_k, top_p)
    assert chi2_p(np.bincount(first, minlength=V), p0) > P_MIN


# ------------------------------- deterministic drafts (greedy acceptance)
def test_tree_det_golden():
    """Hand-worked trees of tests/golden/tree_deterministic_drafts.json."""
    g = _golden("tree_deterministic_drafts.json")
    rows = np.log(np.array([g["rows"][f"p{i}"] for i in range(4)]))
    for ex in g["cases"]:
        o = oracle.verify_tree_det(
            rows.astype(np.float32)[None], np.array([g["parent"]], np.int32),
            np.array([ex["node_tokens"]], np.int32),
            np.array([ex["uniforms"]], np.float32), g["T"])
        assert o["n"][0] == ex["n"], ex["why"]
        np.testing.assert_array_equal(o["tokens"][0], ex["tokens"])
        np.testing.assert_array_equal(o["nodes"][0], ex["nodes"])
        np.testing.assert_allclose(o["prob"][0], ex["prob"], atol=1e-6)


def _one_hot_logits(tok, V):
    z = np.full(V, -np.inf)
    if 0 <= tok < V:
        z[tok] = 0.0
    return z


@pytest.mark.parametrize("T", [0.6, 1.0])
def test_tree_det_chain_equals_tree_rule_with_point_mass_drafts(T):
    """On a chain (one child per node) the deterministic-draft rule is the
    sibling rule of the tree verify with q of every node the point mass on
    its child's token (logits 0 there, -inf elsewhere): accept iff
    U <= p(x)/1, residual max(0, p - delta_x) renormalised."""
    c = synth.linear_case(200, 5, 97, T=T, seed=131)
    tg, dr = synth.host_logits(c.target), synth.host_logits(c.draft)
    xs, u = c.tokens.numpy(), c.uniforms.numpy()
    target, _, parent, ntok, uni = chain_tree_from_linear(tg, dr, xs, u)
    B, N, V = target.shape
    onehot = np.zeros((B, N, V), np.float32)
    for b in range(B):
        for v in range(N - 1):  # node v's only child is node v + 1
            onehot[b, v] = _one_hot_logits(ntok[b, v + 1], V)
    ot = oracle.verify_tree(target, onehot, parent, ntok, uni, T)
    od = oracle.verify_tree_det(target, parent, ntok, uni, T)
    np.testing.assert_array_equal(od["n"], ot["n"])
    np.testing.assert_array_equal(od["tokens"], ot["tokens"])
    np.testing.assert_array_equal(od["nodes"], ot["nodes"])
    np.testing.assert_allclose(od["prob"], ot["prob"], rtol=1e-12)


def test_tree_det_topk_siblings_lossless():
    """Deterministic top-k siblings (the case the sibling rule with a fixed
    q gets wrong, above) keep the emitted token's marginal equal to p under
    the deterministic-draft rule.  V = 8, the root's children are the three
    most likely draft tokens, 1e6 trials, chi-square."""
    rng = np.random.default_rng(133)
    V, S, B = 8, 3, 1_000_000
    zt = rng.normal(0, 1.5, V)
    zq = zt + rng.normal(0, 1.2, V)
    top = np.argsort(-zq, kind="stable")[:S].astype(np.int32)
    tg = tile_rows([zt] + [rng.normal(0, 1, V)] * S, B)
    parent = np.tile(np.array([-1] + [0] * S, np.int32), (B, 1))
    ntok = np.tile(np.concatenate([[-1], top]).astype(np.int32), (B, 1))
    o = oracle.verify_tree_det(tg, parent, ntok,
                               synth.uniforms(134, (B, S + 1)), 1.0)
    assert chi2_p(np.bincount(o["tokens"][:, 0], minlength=V),
                  softmax(zt)) > P_MIN


def test_tree_det_two_level_joint_is_p():
    """Two levels of deterministic children with distinct target rows per
    node: the pair (first, second) emitted tokens has the law
    p_root(a) p_a(b), where p_a is the row of a's node when a was drafted
    and the root's row p_root(b | a) is irrelevant otherwise.  Root with
    children tokens 0, 1; each with children tokens 2, 0; V = 4; 1e6
    trials, chi-square over the 16 pairs."""
    rng = np.random.default_rng(135)
    V, B = 4, 1_000_000
    # nodes: 0 root; 1 (tok 0), 2 (tok 1) under the root; 3, 4 under 1;
    # 5, 6 under 2 (tokens 2, 0)
    parent = np.array([-1, 0, 0, 1, 1, 2, 2], np.int32)
    ntok = np.array([-1, 0, 1, 2, 0, 2, 0], np.int32)
    rows = rng.normal(0, 1.0, (7, V))
    # the row after a prefix that was not drafted: a fresh row per prefix
    # is what the target would give; rows 3..6 are leaves whose row is the
    # distribution of the token after two, irrelevant for the pair law
    o = oracle.verify_tree_det(tile_rows(rows, B), np.tile(parent, (B, 1)),
                               np.tile(ntok, (B, 1)),
                               synth.uniforms(136, (B, 7)), 1.0)
    p0 = softmax(rows[0])
    n = o["n"]
    a = o["tokens"][:, 0]
    b = o["tokens"][:, 1]
    # the second token's law given a: node 1's row for a = 0, node 2's for
    # a = 1; otherwise (a not drafted) the second token is not emitted
    drafted = np.isin(a, [0, 1])
    assert np.all((n >= 1) == drafted)
    pairs = a[drafted] * V + b[drafted]
    law = np.zeros(V * V)
    for tok, node in ((0, 1), (1, 2)):
        law[tok * V:(tok + 1) * V] = p0[tok] * softmax(rows[node])
    law /= law.sum()
    assert chi2_p(np.bincount(pairs, minlength=V * V), law) > P_MIN
    assert chi2_p(np.bincount(a, minlength=V), p0) > P_MIN


def test_tree_det_quadrature_bruteforce():
    """Exact marginal by quadrature: V = 3, two children (tokens 2, 0),
    uniforms on a G x G x G grid of cell midpoints.  Each decision is a
    threshold on one coordinate, so the grid estimate of P(first token = y)
    is within 3/G of the true value, which must be p."""
    G = 64
    p = np.array([0.5, 0.2, 0.3])
    g = (np.arange(G) + 0.5) / G
    U = np.stack(np.meshgrid(g, g, g, indexing="ij"), -1).reshape(-1, 3)
    B = U.shape[0]
    tg = tile_rows(np.log(np.stack([p, p, p])), B)
    parent = np.tile(np.array([-1, 0, 0], np.int32), (B, 1))
    ntok = np.tile(np.array([-1, 2, 0], np.int32), (B, 1))
    o = oracle.verify_tree_det(tg, parent, ntok, U.astype(np.float32), 1.0)
    est = np.bincount(o["tokens"][:, 0], minlength=3) / B
    np.testing.assert_allclose(est, p, atol=3.0 / G)


# ------------------------------ K candidates verified as one token tree
def test_kcand_trie_golden():
    """Hand-worked construction of tests/golden/kcand_trie.json."""
    g = _golden("kcand_trie.json")
    o = oracle.kcand_trie(np.array([g["tokens"]], np.int32),
                          np.array([g["uniforms"]], np.float32))
    for k in ("parent", "node_tokens", "target_row", "draft_row",
              "node_cand", "is_dup"):
        np.testing.assert_array_equal(o[k][0], g[k], err_msg=k)
    np.testing.assert_array_equal(o["uniforms"][0],
                                  np.float32(g["uniforms_out"]))


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_kcand_trie_one_candidate_equals_linear(T):
    """With K = 1 the tree is the candidate's chain, its tests use the
    candidate's uniforms and the final draw its slot gamma: the linear
    verify exactly."""
    c = synth.linear_case(200, 5, 131, T=T, seed=141)
    tg, dr = synth.host_logits(c.target), synth.host_logits(c.draft)
    xs, u = c.tokens.numpy(), c.uniforms.numpy()
    ol = oracle.verify_linear(tg, dr, xs, u, T)
    ok = oracle.verify_kcand_trie(tg[:, None], None if T == 0 else dr,
                                  xs[:, None], u[:, None], T)
    np.testing.assert_array_equal(ok["n"], ol["n"])
    np.testing.assert_array_equal(ok["tokens"], ol["tokens"])
    np.testing.assert_allclose(ok["prob"], ol["prob"], rtol=1e-12)
    assert np.all(ok["k"] == 0)


def _trie_law_case(B, seed):
    """K = 4 iid candidates from shared marginals q_0, q_1 (V = 6, gamma =
    2); target rows that depend on the prefix only: p_0 at position 0, row
    P1[a] after first token a, a fixed row at position 2."""
    rng = np.random.default_rng(seed)
    V, K, gamma = 6, 4, 2
    z0 = rng.normal(0, 1.5, V)
    Z1 = rng.normal(0, 1.5, (V, V))
    z2 = rng.normal(0, 1.0, V)
    q0 = rng.normal(0, 1.5, V)
    q1 = rng.normal(0, 1.5, V)
    x = np.stack([np.stack([draw_from(softmax(q), B, seed + 10 * k + j)
                            for j, q in enumerate((q0, q1))], 1)
                  for k in range(K)], 1)  # [B, K, gamma]
    target = np.empty((B, K, gamma + 1, V), np.float32)
    target[:, :, 0] = z0
    target[:, :, 1] = Z1[x[:, :, 0]]
    target[:, :, 2] = z2
    draft = np.ascontiguousarray(
        np.broadcast_to(np.stack([q0, q1]).astype(np.float32),
                        (B, gamma, V)))
    U = synth.uniforms(seed + 99, (B, K, gamma + 1))
    return z0, Z1, target, draft, x.astype(np.int32), U


def test_kcand_trie_lossless_first_and_second_token():
    """Lossless: the first emitted token follows p_0, and the second,
    given an accepted first token a, follows P1[a] (chi-square, 3e5
    sequences)."""
    B = 300_000
    z0, Z1, target, draft, x, U = _trie_law_case(B, 143)
    o = oracle.verify_kcand_trie(target, draft, x, U, 1.0)
    V = len(z0)
    assert chi2_p(np.bincount(o["tokens"][:, 0], minlength=V),
                  softmax(z0)) > P_MIN
    acc = o["n"] >= 1
    a, b = o["tokens"][acc, 0], o["tokens"][acc, 1]
    na = np.bincount(a, minlength=V)
    law = (na[:, None] * np.stack([softmax(Z1[i]) for i in range(V)]))
    assert chi2_p(np.bincount(a * V + b, minlength=V * V),
                  (law / law.sum()).ravel()) > P_MIN


# ------------------------------------------ PRESTO tree construction
def _presto_run(g, q, rho, depths):
    tree = oracle.PrestoTree(q.shape[0], g["W"], g["budget"])
    for d in range(depths):
        oracle.presto_expand(tree, q[:, d], rho[:, d], g["T"], g["lambda"],
                             g["b"])
        yield tree


def test_presto_golden():
    """Hand-worked two-depth construction, tests/golden/presto_tree.json."""
    g = _golden("presto_tree.json")
    q = np.log(np.array(g["q"]))[None].astype(np.float32)       # [1, D, V]
    rho = np.log(np.array(g["rho"]))[None].astype(np.float32)   # [1, D, W, V]
    for tree, want in zip(_presto_run(g, q, rho, 2), g["after_depth"]):
        n = want["n_nodes"]
        assert tree.n_nodes[0] == n, want["why"]
        np.testing.assert_array_equal(tree.parent[0, :n], want["parent"])
        np.testing.assert_array_equal(tree.node_tokens[0, :n], want["tokens"])
        np.testing.assert_allclose(tree.node_score[0, :n], want["score"],
                                   atol=1e-6)
        np.testing.assert_array_equal(tree.frontier_node[0], want["frontier"])


def test_presto_greedy_chain_is_top1_of_each_marginal():
    """lambda = 0, one path, one token per path: the tree is the chain of
    the argmax of each depth's marginal (linear diffusion drafting), and
    the path scores are the running sums of its log probabilities."""
    from scipy.special import log_softmax
    rng = np.random.default_rng(161)
    B, D, V = 30, 5, 200
    q = rng.normal(0, 2, (B, D, V)).astype(np.float32)
    rho = np.log(rng.random((B, D, 1, V))).astype(np.float32)
    tree = oracle.PrestoTree(B, 1, D + 1)
    for d in range(D):
        oracle.presto_expand(tree, q[:, d], rho[:, d], 0.8, 0.0, 1)
    np.testing.assert_array_equal(tree.n_nodes, D + 1)
    want_tok = np.argmax(q, axis=2)
    np.testing.assert_array_equal(tree.node_tokens[:, 1:], want_tok)
    np.testing.assert_array_equal(tree.parent[:, 1:],
                                  np.tile(np.arange(D), (B, 1)))
    lp = log_softmax(q.astype(np.float64) / 0.8, axis=2)
    want = np.cumsum(np.take_along_axis(lp, want_tok[:, :, None], 2)[:, :, 0],
                     axis=1)
    np.testing.assert_allclose(tree.node_score[:, 1:], want, rtol=1e-12)


def test_presto_score_is_the_kl_minimiser():
    """PRESTO section 4.4: the proxy minimising KL(p || q) - lambda
    E_p[log rho] over the simplex.  Found here by numerical minimisation
    (scipy), it must equal the oracle's scores of all V children of the
    root, normalised."""
    from scipy.optimize import minimize
    from scipy.special import logsumexp, softmax as sm
    rng = np.random.default_rng(162)
    V = 7
    for lam in (0.5, 1.0, 2.0):
        zq = rng.normal(0, 1.5, V)
        rho = rng.uniform(0.05, 1.0, V)
        q = sm(zq)

        def J(a):
            p = sm(a)
            return np.sum(p * (np.log(p) - np.log(q))) - lam * np.sum(
                p * np.log(rho))
        a = minimize(J, np.zeros(V), method="BFGS", options={"gtol": 1e-12}).x
        logp = a - logsumexp(a)
        tree = oracle.PrestoTree(1, 1, V + 1)
        oracle.presto_expand(tree, zq[None].astype(np.float32),
                             np.log(rho)[None, None].astype(np.float32), 1.0,
                             lam, V)
        s = np.empty(V)
        s[tree.node_tokens[0, 1:]] = tree.node_score[0, 1:]
        np.testing.assert_allclose(s - logsumexp(s), logp, atol=1e-5)


def test_presto_construction_invariants():
    """Several depths, W = 3 paths, b = 2 tokens each, budget 16: every
    path's children are its top-b tokens of q_d rho^lambda (probability
    products, not log sums); the nodes added at a depth are the best
    candidates of that depth; the frontier is the W best new nodes; the
    budget is respected."""
    rng = np.random.default_rng(163)
    B, D, W, V, b, budget, lam, T = 20, 5, 3, 40, 2, 16, 0.7, 1.0
    q = rng.normal(0, 1.5, (B, D, V)).astype(np.float32)
    rho = np.log(rng.uniform(0.01, 1, (B, D, W, V))).astype(np.float32)
    tree = oracle.PrestoTree(B, W, budget)
    for d in range(D):
        prev_fn = tree.frontier_node.copy()
        prev_fs = tree.frontier_score.copy()
        n0 = tree.n_nodes.copy()
        oracle.presto_expand(tree, q[:, d], rho[:, d], T, lam, b)
        qd = np.exp(q[:, d].astype(np.float64) / T)
        qd /= qd.sum(1, keepdims=True)
        for s in range(B):
            cands = []
            for w in range(W):
                if prev_fn[s, w] < 0 or n0[s] >= budget:
                    continue
                prod = qd[s] * np.exp(rho[s, d, w].astype(np.float64)) ** lam
                top = np.lexsort((np.arange(V), -prod))[:b]
                cands += [(prev_fs[s, w] + np.log(prod[t]), w, t) for t in top]
            cands.sort(key=lambda c: (-c[0], c[1], c[2]))
            add = min(len(cands), budget - n0[s])
            assert tree.n_nodes[s] == n0[s] + add
            for i in range(add):
                v = n0[s] + i
                sc, w, t = cands[i]
                assert tree.node_tokens[s, v] == t
                assert tree.parent[s, v] == prev_fn[s, w]
                np.testing.assert_allclose(tree.node_score[s, v], sc,
                                           rtol=1e-9)
            want_fn = [n0[s] + i if i < add else -1 for i in range(W)]
            if n0[s] < budget:
                np.testing.assert_array_equal(tree.frontier_node[s], want_fn)
    assert np.all(tree.n_nodes <= budget)


def test_presto_nonfinite_row_invalidates():
    q = np.zeros((3, 8), np.float32)
    rho = np.zeros((3, 2, 8), np.float32)
    q[1, 3] = np.nan
    rho[2, 0, 5] = np.inf
    tree = oracle.PrestoTree(3, 2, 6)
    _, st = oracle.presto_expand(tree, q, rho, 1.0, 1.0, 2)
    np.testing.assert_array_equal(tree.n_nodes, [3, -1, -1])
    assert st[1] & 2 and st[2] & 2 and st[0] == 0


# ------------------------------------------- SpecBranch branch resampling
def test_branch_fork_golden():
    """Hand-worked cases of tests/golden/branch_fork.json."""
    g = _golden("branch_fork.json")
    z = np.log(np.array(g["q"]))[None].astype(np.float32)
    for ex in g["cases"]:
        o = oracle.branch_fork(z, np.array([ex["x_b"]]), ex["T"], ex["k_max"])
        assert o["k"][0] == ex["k"], ex["why"]
        np.testing.assert_array_equal(o["tokens"][0], ex["tokens"])


def test_branch_fork_topk_is_a_stable_sort_and_k_law():
    """The branches are the first k of a stable descending sort of the
    logits; k is non-increasing in q(x_b) and spans 1..k_max - 1 (at T > 0
    every q(x_b) is positive, so k_max itself needs q(x_b) = 0)."""
    rng = np.random.default_rng(164)
    B, V, km = 400, 300, 16
    z = rng.normal(0, 2, (B, V)).astype(np.float32)
    z[:, 10] = z[:, 11]  # ties
    x = rng.integers(0, V, B).astype(np.int32)
    x[:100] = np.argmax(z[:100], 1)  # confident branch points
    z[:20, 0] = 30.0  # very confident: q(x_b) ~ 1, one branch
    x[:20] = 0
    o = oracle.branch_fork(z, x, 1.0, km)
    order = np.argsort(-z, axis=1, kind="stable")
    for b in range(B):
        k = o["k"][b]
        assert 1 <= k <= km
        np.testing.assert_array_equal(o["tokens"][b, :k], order[b, :k])
        assert np.all(o["tokens"][b, k:] == -1)
    from scipy.special import softmax as sm
    qx = sm(z.astype(np.float64), axis=1)[np.arange(B), x]
    srt = np.argsort(qx)
    assert np.all(np.diff(o["k"][srt]) <= 0)
    assert o["k"].max() == km - 1 and o["k"].min() == 1


def test_accept_test_counts_and_flags_planted():
    """acc_tests counts the accept tests made (min(n + 1, gamma) per valid
    sequence at T > 0, none at T == 0); acc_flagged counts those whose r lies
    within 1e-5 of p/q.  Planted: r moved to 4e-6 below the first test's
    ratio (still an accept, and flagged) on every other sequence whose first
    ratio is below 1, and to 3e-5 below it (not flagged) on the rest."""
    rng = np.random.default_rng(41)
    B, gamma, V = 400, 3, 50
    zt = rng.normal(0, 1.5, (B, gamma + 1, V)).astype(np.float32)
    zd = (zt[:, :gamma] + rng.normal(0, 1.0, (B, gamma, V))).astype(
        np.float32)
    x = rng.integers(0, V, (B, gamma)).astype(np.int32)
    u = synth.uniforms(42, (B, gamma + 1))
    o = oracle.verify_linear(zt, zd, x, u, 1.0)
    assert np.array_equal(o["acc_tests"], np.minimum(o["n"] + 1, gamma))
    # the first test's ratio from plain numpy softmaxes (not the oracle)
    def sm(z):
        e = np.exp(z.astype(np.float64) - z.max(-1, keepdims=True))
        return e / e.sum(-1, keepdims=True)
    rho = sm(zt[:, 0])[np.arange(B), x[:, 0]] / \
        sm(zd[:, 0])[np.arange(B), x[:, 0]]
    low = np.nonzero(rho < 0.9)[0]
    plant, far = low[::2], low[1::2]
    u2 = u.copy()
    u2[plant, 0] = (rho[plant] - 4e-6).astype(np.float32)
    u2[far, 0] = (rho[far] - 3e-5).astype(np.float32)
    o2 = oracle.verify_linear(zt, zd, x, u2, 1.0)
    assert np.all(o2["n"][low] >= 1)  # r <= p/q: accepted
    assert np.all(o2["acc_flagged"][plant] >= 1)
    assert np.all(o2["margin_acc"][plant] < 1e-5)
    # the far ones are not flagged unless a later test is (rare)
    assert o2["acc_flagged"][far].sum() <= 1
    assert o2["acc_flagged"].sum() >= len(plant)
    assert o2["acc_flagged"].sum() <= len(plant) + 2
    g = oracle.verify_linear(zt, None, x, u, 0.0)
    assert g["acc_tests"].sum() == 0 and g["acc_flagged"].sum() == 0


def test_filtered_keep_ranges_and_forced_cuts():
    """The kept count of each row read, its admissible range (cuts within
    1e-5 of top_p) and forced counts.  Row p = (1/2, 1/4, 1/4) by hand: with
    top_p = 0.6 the nucleus keeps 2 tokens, unambiguously; with top_p = 0.75
    the third token's prefix mass 0.75 sits on the cut, so 2 and 3 are both
    admissible.  A forced count of 1 leaves the point mass on token 0 (the
    bonus draw then returns it with probability 1)."""
    ln2 = math.log(2.0)
    zt = np.array([[[ln2, 0.0, 0.0]]], np.float32)  # gamma = 0: bonus only
    tk = np.zeros((1, 0), np.int32)
    u = np.array([[0.9]], np.float32)
    o = oracle.verify_linear_filtered(zt, np.zeros((1, 0, 3), np.float32), tk,
                                      u, 1.0, 3, 0.6, want_keep=True)
    assert o["keep"].tolist() == [[2]]
    assert o["keep_lo"].tolist() == [[2]] and o["keep_hi"].tolist() == [[2]]
    assert o["tokens"][0, 0] == 1  # u = 0.9 over (2/3, 1/3): token 1
    o = oracle.verify_linear_filtered(zt, np.zeros((1, 0, 3), np.float32), tk,
                                      u, 1.0, 3, 0.75, want_keep=True)
    assert o["keep_lo"].tolist() == [[2]] and o["keep_hi"].tolist() == [[3]]
    o = oracle.verify_linear_filtered(zt, np.zeros((1, 0, 3), np.float32), tk,
                                      u, 1.0, 3, 0.6, keep_forced=[[1]])
    assert o["tokens"][0, 0] == 0 and abs(o["prob"][0] - 1.0) < 1e-15
    # forced counts equal to the computed ones change nothing; rows not read
    # are -1; lo <= keep <= hi
    rng = np.random.default_rng(5)
    B, gamma, V = 60, 3, 400
    zt = rng.normal(0, 2, (B, gamma + 1, V)).astype(np.float32)
    zd = (zt[:, :gamma] + rng.normal(0, 1, (B, gamma, V))).astype(np.float32)
    x = rng.integers(0, 40, (B, gamma)).astype(np.int32)
    uu = synth.uniforms(6, (B, gamma + 1))
    for top_k, top_p in ((400, 0.9), (30, 0.95), (5, 1.0)):
        a = oracle.verify_linear_filtered(zt, zd, x, uu, 1.0, top_k, top_p,
                                          want_keep=True)
        b = oracle.verify_linear_filtered(zt, zd, x, uu, 1.0, top_k, top_p,
                                          keep_forced=a["keep"])
        for k in ("n", "tokens", "prob"):
            assert np.array_equal(a[k], b[k]), k
        rd = a["keep"] >= 0
        n = a["n"][:, None]
        slot = np.arange(2 * gamma + 1)[None, :]
        want = np.where(slot <= gamma, slot <= n,
                        (slot - gamma - 1 <= n) & (slot - gamma - 1 < gamma))
        assert np.array_equal(rd, want)
        assert np.all(a["keep_lo"][rd] <= a["keep"][rd])
        assert np.all(a["keep"][rd] <= a["keep_hi"][rd])
        assert np.all(a["keep"][rd] <= min(top_k, V))
        if top_p == 1.0:
            assert np.all(a["keep"][rd] == min(top_k, V))
