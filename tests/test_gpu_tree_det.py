"""Parity of sd_verify_tree_det (deterministic drafts: child v accepted with
the current p(t_v), a rejected token removed from p; CUDA, through the C
ABI) with the oracle's literal walk: small and odd sizes, top-k trees from
the synthetic builder, wide sibling lists, repeated sibling tokens, the
plain-load path, every cluster size, the tree workload's shape, invalid
inputs, the greedy route, and the emitted token's law on the GPU."""
import numpy as np
import pytest
import torch
from scipy import stats

import oracle
from speculative_decoding_verification_temperature_gb300 import api, synth
from tests.parity import compare, host, to_device

pytestmark = pytest.mark.gpu


def det_oracle(c):
    return oracle.verify_tree_det(synth.host_logits(c.target), host(c.parent),
                                  host(c.node_tokens), host(c.uniforms), c.T)


def run(c, **kw):
    return api.verify_tree_det(c.target, c.parent, c.node_tokens, c.uniforms,
                               c.T, **kw)


@pytest.mark.parametrize("T", [0.0, 0.8, 1.0])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("N,V", [(1, 100), (8, 333), (24, 1000), (64, 4099)])
def test_small_trees(T, dtype, N, V):
    c = to_device(synth.tree_case(20, N, V, dtype, T, seed=N * 11 + V,
                                  sigma_t=1.5, sigma_d=1.0))
    compare(run(c), det_oracle(c), extra_equal=("nodes",))


def test_wide_sibling_lists():
    """Twelve children per node near the root: long runs of removals, some
    in the same 32-vector segment."""
    c = to_device(synth.tree_case(12, 60, 2000, torch.float32, 1.0, seed=6,
                                  sigma_t=1.0, sigma_d=1.5, branch=12,
                                  max_depth=3))
    compare(run(c), det_oracle(c), extra_equal=("nodes",))


def test_repeated_and_adjacent_sibling_tokens():
    """Siblings repeating a token (p(t_v) = 0 after its removal), and
    siblings on neighbouring ids (one segment recomputed for several
    removals)."""
    c = synth.tree_case(16, 12, 3000, torch.float32, 1.0, seed=8,
                        sigma_t=0.5, sigma_d=0.5, branch=6, max_depth=2)
    par = c.parent.numpy()
    for b in range(16):
        kids = [v for v in range(1, 12) if par[b, v] == 0]
        if b % 2 == 0 and len(kids) >= 3:
            c.node_tokens[b, kids[2]] = c.node_tokens[b, kids[0]]
        else:
            for i, v in enumerate(kids):
                c.node_tokens[b, v] = 40 + i
    c = to_device(c)
    compare(run(c), det_oracle(c), extra_equal=("nodes",))


@pytest.mark.parametrize("sw", [{"no_tma": 1}, {"cluster": 1},
                                {"cluster": 2}, {"cluster": 8}])
def test_load_paths_and_cluster_sizes(sw):
    c = to_device(synth.tree_case(10, 32, 20000, torch.bfloat16, 1.0,
                                  seed=9, sigma_t=1.0, sigma_d=1.0))
    with api.tuned(**sw):
        g = run(c)
    compare(g, det_oracle(c), extra_equal=("nodes",))


def test_unaligned_rows_plain_loads():
    c = to_device(synth.tree_case(10, 16, 1001, torch.float32, 0.7, seed=10,
                                  sigma_t=1.0, sigma_d=1.0))
    compare(run(c), det_oracle(c), extra_equal=("nodes",))


def test_tree_workload_shape():
    """B=16 trees of 64 nodes (top-k children, k = 4..1 with depth, depth
    <= 8), V=151936 bf16, T=0.8: every tree against the oracle."""
    c = synth.tree(0, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = run(c, status=st)
    assert int(st.item()) == 0
    compare(g, det_oracle(c), extra_equal=("nodes",))


def test_invalid_parent_rows_and_tokens():
    c = synth.tree_case(5, 10, 400, torch.float32, 1.0, seed=22)
    c.parent[1, 4] = 7
    c.parent[2, 0] = 3
    c.target[3, 0, 11] = float("nan")
    c.node_tokens[4, 1] = 10**6
    c = to_device(c)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    compare(run(c, status=st), det_oracle(c), extra_equal=("nodes",))
    s = int(st.item())
    assert s & api.DEV_BAD_PARENT and s & api.DEV_NONFINITE
    assert s & api.DEV_BAD_TOKEN


def test_greedy_equals_tree_greedy():
    c = to_device(synth.tree_case(20, 24, 5000, torch.bfloat16, 0.0, seed=23))
    a = run(c)
    b = api.verify_tree(c.target, c.draft, c.parent, c.node_tokens,
                        c.uniforms, 0.0)
    for k in ("n", "tokens", "nodes"):
        assert torch.equal(a[k], b[k])


def test_topk_children_emitted_token_law_on_gpu():
    """The root's children are the three most likely draft tokens (not
    drawn from anything): the first emitted token follows p (chi-square,
    V = 8, 1e6 trees)."""
    rng = np.random.default_rng(133)
    V, S, B = 8, 3, 1_000_000
    zt = rng.normal(0, 1.5, V).astype(np.float32)
    zq = zt + rng.normal(0, 1.2, V)
    p = np.exp(zt.astype(np.float64) - zt.max())
    p /= p.sum()
    top = np.argsort(-zq, kind="stable")[:S]
    rows = np.stack([zt] + [rng.normal(0, 1, V).astype(np.float32)] * S)
    tg = torch.from_numpy(rows).expand(B, S + 1, V).contiguous().cuda()
    parent = torch.tensor([-1] + [0] * S, dtype=torch.int32).repeat(B, 1)
    ntok = torch.tensor([-1] + list(top), dtype=torch.int32).repeat(B, 1)
    U = torch.from_numpy(synth.uniforms(134, (B, S + 1)))
    out = api.verify_tree_det(tg, parent.cuda(), ntok.cuda(), U.cuda(), 1.0)
    cnt = np.bincount(host(out["tokens"][:, 0]), minlength=V)
    stat = ((cnt - B * p) ** 2 / (B * p)).sum()
    assert stats.chi2.sf(stat, V - 1) > 1e-4
