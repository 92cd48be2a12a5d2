"""Parity of sd_verify_tree (CUDA, through the C ABI) with the oracle's
literal walk (explicit p <- norm(max(0, p - q)) after each sibling
rejection; the kernel uses the closed form max(0, p - c q) / N)."""
import numpy as np
import pytest
import torch
from scipy import stats

import oracle
from speculative_decoding_verification_temperature_gb300 import api, synth
from tests.parity import compare, host, linear_oracle, to_device

pytestmark = pytest.mark.gpu


def tr_oracle(c):
    return oracle.verify_tree(synth.host_logits(c.target),
                              synth.host_logits(c.draft), host(c.parent),
                              host(c.node_tokens), host(c.uniforms), c.T)


def run(c, **kw):
    return api.verify_tree(c.target, c.draft, c.parent, c.node_tokens,
                           c.uniforms, c.T, **kw)


@pytest.mark.parametrize("T", [0.0, 0.8, 1.0])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("N,V", [(1, 100), (8, 333), (24, 1000), (64, 4099)])
def test_small_trees(T, dtype, N, V):
    c = to_device(synth.tree_case(20, N, V, dtype, T, seed=N * 7 + V,
                                  sigma_t=1.5, sigma_d=1.0))
    compare(run(c), tr_oracle(c), extra_equal=("nodes",))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_zero_residuals_and_masked_tails(dtype):
    """Wide sibling lists on ragged slices with identical target and draft
    rows (zero residual) and masked tails."""
    c = synth.tree_case(16, 40, 8200, dtype, 0.9, seed=41,
                        sigma_t=1.0, sigma_d=1.5, branch=6, max_depth=4)
    c.draft[0] = c.target[0]                      # zero residuals
    c.target[1, :, 5000:] = -float("inf")         # masked tails
    c.draft[2, :, :4096] = -float("inf")
    c = to_device(c)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = run(c, status=st)
    compare(g, tr_oracle(c), extra_equal=("nodes",))
    assert int(st.item()) & ~(api.DEV_ZERO_MASS) == 0


def test_wide_sibling_lists():
    """Many siblings under the root and under each node (branch 12): long
    runs of residual updates."""
    c = to_device(synth.tree_case(12, 60, 2000, torch.float32, 1.0, seed=5,
                                  sigma_t=1.0, sigma_d=1.5, branch=12,
                                  max_depth=3))
    compare(run(c), tr_oracle(c), extra_equal=("nodes",))


def test_chain_tree_equals_linear():
    c = synth.linear_case(50, 5, 3000, torch.float32, 1.0, seed=12)
    B, gamma, V = 50, 5, 3000
    dtree = torch.cat([c.draft, torch.zeros(B, 1, V)], 1)
    parent = torch.arange(-1, gamma, dtype=torch.int32).repeat(B, 1)
    ntok = torch.cat([torch.full((B, 1), -1, dtype=torch.int32), c.tokens], 1)
    U = torch.cat([c.uniforms[:, gamma:], c.uniforms[:, :gamma]], 1)
    gt = api.verify_tree(c.target.cuda(), dtree.cuda(), parent.cuda(),
                         ntok.cuda(), U.cuda(), 1.0)
    gl = api.verify_linear(c.target.cuda(), c.draft.cuda(), c.tokens.cuda(),
                           c.uniforms.cuda(), 1.0)
    assert torch.equal(gt["n"], gl["n"])
    assert torch.equal(gt["tokens"][:, :gamma + 1], gl["tokens"])


def test_tree_workload():
    """B=16 trees of 64 nodes (top-k children, k = 4..1 with depth, depth
    <= 8), V=151936 bf16, T=0.8: every tree against the oracle."""
    c = synth.tree(0, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = run(c, status=st)
    assert int(st.item()) == 0
    compare(g, tr_oracle(c), extra_equal=("nodes",))


def test_iid_siblings_emitted_token_law_on_gpu():
    """Siblings drawn iid from the root's q: the first emitted token follows
    p (chi-square, V = 8, three siblings, 1e6 trees)."""
    rng = np.random.default_rng(95)
    V, S, B = 8, 3, 1_000_000
    zt = rng.normal(0, 1.5, V).astype(np.float32)
    zq = (zt + rng.normal(0, 1.2, V)).astype(np.float32)
    p = np.exp(zt - zt.max()); p /= p.sum()
    q = np.exp(zq.astype(np.float64) - zq.max()); q /= q.sum()
    rows_t = np.stack([zt] + [rng.normal(0, 1, V).astype(np.float32)] * S)
    rows_d = np.stack([zq] + [np.zeros(V, np.float32)] * S)
    tg = torch.from_numpy(rows_t).expand(B, S + 1, V).contiguous().cuda()
    dr = torch.from_numpy(rows_d).expand(B, S + 1, V).contiguous().cuda()
    parent = torch.tensor([-1] + [0] * S, dtype=torch.int32).repeat(B, 1)
    g = np.random.default_rng(96)
    kids = np.stack([np.argmax(np.log(q)[None] - np.log(-np.log(
        g.random((B, V)).clip(1e-300))), 1) for _ in range(S)], 1)
    ntok = torch.from_numpy(np.concatenate(
        [np.full((B, 1), -1), kids], 1).astype(np.int32))
    U = torch.from_numpy(synth.uniforms(97, (B, S + 1)))
    out = api.verify_tree(tg, dr, parent.cuda(), ntok.cuda(), U.cuda(), 1.0)
    cnt = np.bincount(host(out["tokens"][:, 0]), minlength=V)
    stat = ((cnt - B * p) ** 2 / (B * p)).sum()
    assert stats.chi2.sf(stat, V - 1) > 1e-4


def test_invalid_parent_and_rows():
    c = synth.tree_case(5, 10, 400, torch.float32, 1.0, seed=21)
    c.parent[1, 4] = 7            # parent after the child
    c.parent[2, 0] = 3            # root with a parent
    c.target[3, 0, 11] = float("nan")
    c.node_tokens[4, 1] = 10**6   # bad token on a child of the root
    to_device(c)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = run(c, status=st)
    o = tr_oracle(c)
    compare(g, o, extra_equal=("nodes",))
    s = int(st.item())
    assert s & api.DEV_BAD_PARENT and s & api.DEV_NONFINITE
    assert s & api.DEV_BAD_TOKEN
