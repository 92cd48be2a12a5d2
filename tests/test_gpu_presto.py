"""Parity of the device tree construction (CUDA, through the C ABI) with
the oracle: PRESTO's beam over several depths (sd_presto_init and
sd_presto_expand: score log q_d + lambda log rho, path scores, global
retention under a node budget) and SpecBranch's branch resampling
(sd_branch_fork).  Node ids, parents, tokens and frontiers must match
exactly, scores to fp32 rounding; a sequence whose outcome was decided by a
score gap below 1e-4 (the oracle's margin) is no longer compared from that
depth on, and such sequences are counted."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_temperature_gb300 import api, synth
from tests.parity import host

pytestmark = pytest.mark.gpu

MARGIN = 1e-4


def presto_inputs(B, D, W, V, dtype, seed, sigma=2.0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, D, V), generator=g) * sigma
    rho = torch.log(torch.rand((B, D, W, V), generator=g) * 0.99 + 0.01)
    return q.to(dtype), rho.to(dtype)


def run_both(q, rho, T, lam, W, b_top, budget, idx=None):
    """Build the trees depth by depth on the GPU and in the oracle; compare
    after every depth.  Returns the number of sequences set aside."""
    B, D, V = q.shape
    qd, rd = q.cuda(), rho.cuda()
    gt = api.PrestoTree(B, W, budget, "cuda")
    sel = np.arange(B) if idx is None else np.asarray(idx)
    ot = oracle.PrestoTree(len(sel), W, budget)
    qh = synth.host_logits(q[sel])
    rh = synth.host_logits(rho[sel])
    live = np.ones(len(sel), bool)
    for d in range(D):
        api.presto_expand(gt, qd[:, d],
                          None if lam == 0 else rd[:, d].contiguous(), T,
                          lam, b_top)
        margin, _ = oracle.presto_expand(
            ot, np.ascontiguousarray(qh[:, d]), np.ascontiguousarray(rh[:, d]),
            T, lam, b_top)
        live &= ~(margin < MARGIN)
        g_n = host(gt.n_nodes)[sel]
        np.testing.assert_array_equal(g_n[live], ot.n_nodes[live])
        for name in ("parent", "node_tokens", "frontier_node"):
            g = host(getattr(gt, name))[sel][live]
            np.testing.assert_array_equal(g, getattr(ot, name)[live],
                                          err_msg="%s at depth %d" % (name, d))
        gs = host(gt.node_score)[sel][live]
        os_ = ot.node_score[live]
        used = np.arange(budget)[None, :] < ot.n_nodes[live][:, None]
        np.testing.assert_allclose(gs[used], os_[used], rtol=1e-5, atol=1e-4)
    return int((~live).sum())


@pytest.mark.parametrize("V,dtype", [(1000, torch.float32),
                                     (1001, torch.float32),
                                     (4104, torch.bfloat16),
                                     (50000, torch.bfloat16)])
@pytest.mark.parametrize("lam,T", [(0.0, 1.0), (0.7, 0.8), (2.0, 1.0)])
def test_beam_construction(V, dtype, lam, T):
    q, rho = presto_inputs(12, 6, 4, V, dtype, seed=V + int(10 * lam))
    flagged = run_both(q, rho, T, lam, W=4, b_top=3, budget=30)
    assert flagged <= 2


@pytest.mark.parametrize("W,b_top,budget", [(1, 1, 7), (8, 8, 64),
                                            (2, 64, 200), (64, 2, 90)])
def test_widths_and_budgets(W, b_top, budget):
    """Up to 128 proposals per depth, every one of them added: the order of
    all of them fixes the node ids, so the logits are spread (sigma 8) to
    keep near-ties within the margin rare; at most a third of the
    sequences may be set aside."""
    q, rho = presto_inputs(12, 5, W, 3000, torch.float32, seed=W * b_top,
                           sigma=8.0)
    assert run_both(q, rho, 1.0, 0.5, W, b_top, budget) <= 4


def test_greedy_chain_is_argmax_per_depth():
    q, rho = presto_inputs(32, 8, 1, 20000, torch.bfloat16, seed=3)
    t = api.PrestoTree(32, 1, 9, "cuda")
    qd = q.cuda()
    for d in range(8):
        api.presto_expand(t, qd[:, d], None, 1.0, 0.0, 1)
    assert torch.all(t.n_nodes == 9)
    want = torch.argmax(qd.float(), dim=2).int()
    assert torch.equal(t.node_tokens[:, 1:], want)


def test_tree_workload_shape_sampled():
    """B=16 sequences, V=151936 bf16, 8 depths, W=8 paths, b=4 tokens per
    path, budget 64 nodes; 3 sequences against the oracle."""
    q, rho = presto_inputs(16, 8, 8, 151936, torch.bfloat16, seed=11)
    assert run_both(q, rho, 0.8, 1.0, 8, 4, 64, idx=[0, 7, 15]) <= 1


def test_nonfinite_rows():
    q, rho = presto_inputs(5, 2, 2, 700, torch.float32, seed=4)
    q[1, 0, 5] = float("nan")
    rho[2, 0, 0, 9] = float("inf")
    rho[3, 1, 1, 2] = float("nan")  # depth 1, path 1
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t = api.PrestoTree(5, 2, 10, "cuda")
    for d in range(2):
        api.presto_expand(t, q.cuda()[:, d], rho.cuda()[:, d].contiguous(),
                          1.0, 1.0, 2, status=st)
    n = host(t.n_nodes)
    assert n[1] == -1 and n[2] == -1 and n[3] == -1
    assert n[0] == 7 and n[4] == 7
    assert int(st.item()) & api.DEV_NONFINITE
    run_both(q[[0, 4]], rho[[0, 4]], 1.0, 1.0, 2, 2, 10)


# ---------------------------------------------------------------- fork
@pytest.mark.parametrize("V,dtype", [(1000, torch.float32),
                                     (4099, torch.float32),
                                     (32000, torch.bfloat16),
                                     (151936, torch.bfloat16)])
@pytest.mark.parametrize("T", [0.0, 0.7, 1.0])
@pytest.mark.parametrize("k_max", [1, 8, 64])
def test_branch_fork(V, dtype, T, k_max):
    g = torch.Generator().manual_seed(V + k_max)
    B = 48
    z = (torch.randn((B, V), generator=g) * 2.5).to(dtype)
    z[:4, 17] = 40.0  # confident rows
    x = torch.randint(0, V, (B,), generator=g, dtype=torch.int32)
    x[:16] = torch.argmax(z[:16].float(), 1).int()
    x[40] = V  # out of range
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gk = api.branch_fork(z.cuda(), x.cuda(), T, k_max, status=st)
    o = oracle.branch_fork(synth.host_logits(z), x.numpy(), T, k_max)
    k, tok = host(gk["k"]), host(gk["tokens"])
    near = o["margin"] < 1e-4  # relative distance of k_max q to a step
    assert near.sum() <= 2
    np.testing.assert_array_equal(k[~near], o["k"][~near])
    assert np.all(np.abs(k[near] - o["k"][near]) <= 1)
    same = k == o["k"]
    np.testing.assert_array_equal(tok[same], o["tokens"][same])
    assert k[40] == -1 and int(st.item()) & api.DEV_BAD_TOKEN


def test_branch_fork_nan_row_and_ties():
    z = torch.zeros((3, 512), dtype=torch.float32)
    z[0, 100] = float("nan")
    z[1, :] = -0.0  # every logit ties (-0 equals +0): lowest ids first
    z[2, 7] = 1.0
    z[2, 3] = 1.0
    x = torch.tensor([0, 5, 3], dtype=torch.int32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = api.branch_fork(z.cuda(), x.cuda(), 1.0, 8, status=st)
    o = oracle.branch_fork(z.numpy(), x.numpy(), 1.0, 8)
    np.testing.assert_array_equal(host(g["k"]), o["k"])
    np.testing.assert_array_equal(host(g["tokens"]), o["tokens"])
    assert host(g["k"])[0] == -1 and int(st.item()) & api.DEV_NONFINITE
