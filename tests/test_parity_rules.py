"""The comparison rule the GPU parity tests use (tests/parity.py), checked
on CPU: results equal to the oracle's pass; a planted disagreement fails
unless the oracle flagged that very draw (an accept test or a CDF boundary
within 1e-5 of the uniform), and even then a final token must stay inside
the oracle's admissible range.  The planted results are copies of the
oracle's own output with one entry changed; nothing here runs a GPU."""
import numpy as np
import pytest

import oracle
from tests.parity import compare


def _case(T, seed=3, B=60, gamma=4, V=40):
    rng = np.random.default_rng(seed)
    zt = rng.normal(0.0, 1.5, (B, gamma + 1, V)).astype(np.float32)
    zd = (zt[:, :gamma] + rng.normal(0.0, 0.7, (B, gamma, V))).astype(
        np.float32)
    x = np.argmax(zd, axis=2).astype(np.int32)
    x[::4] = rng.integers(0, V, (len(x[::4]), gamma))
    u = ((rng.integers(0, 2**23, (B, gamma + 1)) + 0.5) / 2**23).astype(
        np.float32)
    zt[7, 0, 5] = np.nan  # one unusable sequence (n = -1): row 0 is read
    o = oracle.verify_linear(zt, None if T == 0 else zd, x, u, T)
    g = {k: o[k].copy() for k in ("n", "tokens", "prob")}
    g["prob"] = g["prob"].astype(np.float32)
    return o, g


def _seq(o, pred):
    """A sequence satisfying pred(b) that the oracle did not flag."""
    for b in range(len(o["n"])):
        if (o["margin_acc"][b] >= oracle.FLAG_MARGIN and
                o["margin_cdf"][b] >= oracle.FLAG_MARGIN and pred(b)):
            return b
    raise AssertionError("no such sequence in the case")


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_equal_results_pass(T):
    o, g = _case(T)
    r = compare(g, o)
    assert r["seqs"] == len(o["n"]) and r["cdf_diff"] == 0
    assert o["n"][7] == -1


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_count_difference_fails(T):
    o, g = _case(T)
    b = _seq(o, lambda b: 0 <= o["n"][b] < o["tokens"].shape[1] - 1)
    g["n"][b] += 1
    with pytest.raises(AssertionError):
        compare(g, o)


def test_invalid_sequence_must_stay_invalid():
    o, g = _case(1.0)
    g["n"][7] = 0
    with pytest.raises(AssertionError):
        compare(g, o)


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_token_difference_fails(T):
    o, g = _case(T)
    b = _seq(o, lambda b: o["n"][b] >= 1)
    g["tokens"][b, 0] += 1                  # an accepted draft token
    with pytest.raises(AssertionError):
        compare(g, o)
    o, g = _case(T)
    b = _seq(o, lambda b: o["n"][b] >= 0)
    g["tokens"][b, o["n"][b]] ^= 1          # the final draw
    with pytest.raises(AssertionError):
        compare(g, o)


def test_accept_flagged_sequence_is_set_aside_and_counted():
    o, g = _case(1.0)
    b = _seq(o, lambda b: 0 <= o["n"][b] < o["tokens"].shape[1] - 1)
    o["margin_acc"][b] = 0.5 * oracle.FLAG_MARGIN
    g["n"][b] += 1
    g["tokens"][b, :] = -7
    r = compare(g, o)
    assert r["acc_flagged"] == 1


def test_cdf_flagged_draw_must_stay_in_the_admissible_range():
    o, g = _case(1.0)
    b = _seq(o, lambda b: o["n"][b] >= 0)
    n, t = o["n"][b], o["tokens"][b, o["n"][b]]
    o["margin_cdf"][b] = 0.5 * oracle.FLAG_MARGIN
    o["cdf_lo"][b], o["cdf_hi"][b] = t, t + 1
    g["tokens"][b, n] = t + 1               # inside: accepted, counted
    r = compare(g, o)
    assert r["cdf_flagged"] == 1 and r["cdf_diff"] == 1
    g["tokens"][b, n] = t + 2               # outside: rejected
    with pytest.raises(AssertionError):
        compare(g, o)


def test_greedy_draws_are_never_set_aside():
    o, g = _case(0.0)
    assert np.all(np.isinf(o["margin_acc"])) and np.all(
        np.isinf(o["margin_cdf"]))


def test_probability_tolerance():
    o, g = _case(1.0)
    b = _seq(o, lambda b: o["n"][b] >= 0)
    g["prob"][b] = o["prob"][b] + 0.5e-5
    compare(g, o)
    g["prob"][b] = o["prob"][b] + 5e-5
    with pytest.raises(AssertionError):
        compare(g, o)


def test_extra_equal_fields_are_compared():
    o, g = _case(1.0)
    o["accept"] = o["accept"].copy()
    g["accept"] = o["accept"].copy()
    compare(g, o, extra_equal=("accept",))
    b = _seq(o, lambda b: o["n"][b] >= 1)
    g["accept"][b, 0] = 0.123
    with pytest.raises(AssertionError):
        compare(g, o, extra_equal=("accept",))
