"""The byte counting behind bench.py's roofline figures, on CPU: the rows a
round needs (linear, K candidates, trees) against explicit row sets built
from the rules they count, hand-counted trees, and the schedules the bench
compares.  No GPU."""
import numpy as np
import pytest

import bench


def _linear_row_set(n, gamma, greedy):
    """Target rows 0..n (the accept tests, then the draw at n or the bonus
    at gamma); draft rows 0..min(n, gamma-1) unless greedy."""
    rows = {("t", i) for i in range(n + 1)}
    if not greedy:
        rows |= {("d", i) for i in range(min(n, gamma - 1) + 1)}
    return rows


@pytest.mark.parametrize("greedy", [False, True])
def test_linear_rows_against_row_sets(greedy):
    rng = np.random.default_rng(0)
    gamma = 8
    n = rng.integers(0, gamma + 1, size=300)
    want = sum(len(_linear_row_set(int(x), gamma, greedy)) for x in n)
    assert bench._rows_linear(n, gamma, greedy) == want
    if not greedy:
        assert bench.needed_bytes(n, gamma, 1000, 4) == want * 1000 * 4


def test_linear_rows_extremes():
    gamma, V = 8, 128256
    # every draft accepted: all 2 gamma + 1 rows, the whole tensors
    assert bench.needed_bytes([gamma], gamma, V, 4) == (2 * gamma + 1) * V * 4
    # first draft rejected: target row 0 and draft row 0
    assert bench.needed_bytes([0], gamma, V, 4) == 2 * V * 4
    assert bench._rows_linear([0, gamma], gamma, True) == 1 + gamma + 1


def _kcand_row_set(npc, gamma):
    """Candidate k's accept scan reads its target rows 0..min(n_k, gamma-1);
    the selected candidate's bonus row gamma when its streak is complete;
    the shared draft rows 0..min(n_max, gamma-1)."""
    n_max = max(npc)
    k_sel = npc.index(n_max)  # lowest k among the longest streaks
    rows = set()
    for k, nk in enumerate(npc):
        rows |= {("t", k, i) for i in range(min(nk, gamma - 1) + 1)}
    if n_max == gamma:
        rows.add(("t", k_sel, gamma))
    rows |= {("d", i) for i in range(min(n_max, gamma - 1) + 1)}
    return rows


def test_kcand_rows_against_row_sets():
    rng = np.random.default_rng(1)
    B, K, gamma = 50, 8, 16
    # streaks skewed short, with some complete ones
    npc = np.minimum(rng.geometric(0.3, size=(B, K)) - 1, gamma)
    npc[::7, 3] = gamma
    n = npc.max(1)
    want = sum(len(_kcand_row_set([int(x) for x in npc[b]], gamma))
               for b in range(B))
    assert bench._rows_kcand(npc, n, gamma) == want


def test_kcand_rows_hand_counted():
    # gamma = 4; candidates' streaks 1, 4, 0: target rows 2 + 4 + 1, the
    # bonus row of candidate 1, draft rows 0..3
    assert bench._rows_kcand([[1, 4, 0]], [4], 4) == 7 + 1 + 4
    # all rejected at once: one target row each, draft row 0
    assert bench._rows_kcand([[0, 0]], [0], 4) == 2 + 1


def test_tree_rows_hand_counted():
    #        0
    #      /   \
    #     1     2
    #    / \    |
    #   3   4   5
    parent = np.array([[-1, 0, 0, 1, 1, 2]])
    # path 0 -> 1 -> 3: target rows 0, 1, 3; draft rows 0, 1 (3 is a leaf)
    nodes = np.array([[1, 3, -1, -1, -1, -1]])
    assert bench._rows_tree(parent, nodes, np.array([2]), False) == 5
    assert bench._rows_tree(parent, nodes, np.array([2]), True) == 3
    # path 0 -> 2 stops there (5 rejected): target 0, 2; draft 0, 2
    nodes = np.array([[2, -1, -1, -1, -1, -1]])
    assert bench._rows_tree(parent, nodes, np.array([1]), False) == 4
    # nothing accepted: root's target and draft rows
    assert bench._rows_tree(parent, nodes, np.array([0]), False) == 2
    assert bench._rows_tree(parent, nodes, np.array([0]), True) == 1


@pytest.mark.parametrize("greedy", [False, True])
def test_chain_tree_rows_equal_linear_rows(greedy):
    """A chain of gamma + 1 nodes is the linear verify: the two counts, kept
    in separate code, agree for every accepted length."""
    gamma = 6
    parent = np.arange(-1, gamma)[None, :]
    for n in range(gamma + 1):
        nodes = np.full((1, gamma + 1), -1)
        nodes[0, :n] = np.arange(1, n + 1)
        assert bench._rows_tree(parent, nodes, np.array([n]), greedy) == \
            bench._rows_linear([n], gamma, greedy)


def test_uniform_schedule():
    F = bench.uniform_schedule(8, 64)
    assert F == [8, 7, 7, 7, 7, 7, 7, 7, 7]
    for K, budget in [(1, 2), (4, 17), (8, 9), (3, 100)]:
        F = bench.uniform_schedule(K, budget)
        assert sum(F) == budget and max(F) - min(F) <= 1
        assert F == sorted(F, reverse=True)


def test_traffic_constants_are_plausible():
    """The ncu traffic the roofline line scales: the fan-out reads each
    draft row once (within 1 % of a row's bytes), and the verify reads
    more than the rows it needs (the draw's second pass), but less than
    twice them."""
    fan_bytes, fan_rows = bench.TRAFFIC["fanout"]
    assert abs(fan_bytes / fan_rows - 128256 * 4) < 0.01 * 128256 * 4
    lin_traffic, lin_needed = bench.TRAFFIC["linear"]
    assert 1.0 < lin_traffic / lin_needed < 2.0


def test_flag_summary_counts_and_mismatches():
    """bench.flag_summary on oracle results: outputs equal to the oracle's
    give no mismatch; a changed count or a changed token outside a flagged
    draw is one mismatch each; a near-boundary final draw inside the
    admissible range is counted in cdf_diff, not as a mismatch."""
    import torch
    import oracle
    from speculative_decoding_verification_temperature_gb300 import synth
    c = synth.linear_case(300, 4, 200, torch.float32, 1.0, seed=3,
                          sigma_t=2.0, sigma_d=1.0)
    o = oracle.verify_linear(synth.host_logits(c.target),
                             synth.host_logits(c.draft), c.tokens.numpy(),
                             c.uniforms.numpy(), 1.0)
    g = {"n": o["n"].copy(), "tokens": o["tokens"].copy()}
    s = bench.flag_summary(o, g, 1.0)
    assert s["mismatches"] == 0 and s["sequences"] == 300
    assert s["accept_tests"] == int(np.minimum(o["n"] + 1, 4).sum())
    assert s["cdf_draws"] == 300
    clean = np.nonzero((o["margin_acc"] >= 1e-5) &
                       (o["margin_cdf"] >= 1e-5))[0]
    g["n"][clean[0]] += 1
    g["tokens"][clean[1], 0] ^= 1
    assert bench.flag_summary(o, g, 1.0)["mismatches"] == 2
    near = np.nonzero((o["margin_cdf"] < 1e-5) & (o["margin_acc"] >= 1e-5) &
                      (o["cdf_hi"] > o["cdf_lo"]))[0]
    if near.size:
        b = near[0]
        g = {"n": o["n"].copy(), "tokens": o["tokens"].copy()}
        alt = o["cdf_lo"][b] if o["tokens"][b, o["n"][b]] != o["cdf_lo"][b] \
            else o["cdf_hi"][b]
        g["tokens"][b, o["n"][b]] = alt
        s = bench.flag_summary(o, g, 1.0)
        assert s["mismatches"] == 0 and s["cdf_diff"] == 1
