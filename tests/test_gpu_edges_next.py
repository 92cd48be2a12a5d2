"""Edge cases of the later entry points (CUDA, through the C ABI) against
the oracle: empty batches, the largest trees and tries, the largest PRESTO
proposal sets, forks wider than the vocabulary, and refused arguments."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_temperature_gb300 import api, synth
from tests.parity import compare, host, to_device

pytestmark = pytest.mark.gpu


def test_empty_batches():
    z = torch.zeros((0, 3, 64), device="cuda")
    p = torch.zeros((0, 3), dtype=torch.int32, device="cuda")
    u = torch.zeros((0, 3), device="cuda")
    o = api.verify_tree_det(z, p, p, u, 1.0)
    assert o["n"].numel() == 0
    o = api.verify_kcand_trie(torch.zeros((0, 2, 3, 64), device="cuda"),
                              torch.zeros((0, 2, 64), device="cuda"),
                              torch.zeros((0, 2, 2), dtype=torch.int32,
                                          device="cuda"),
                              torch.zeros((0, 2, 3), device="cuda"), 1.0)
    assert o["n"].numel() == 0
    f = api.branch_fork(torch.zeros((0, 64), device="cuda"),
                        torch.zeros(0, dtype=torch.int32, device="cuda"),
                        1.0, 4)
    assert f["k"].numel() == 0
    t = api.PrestoTree(0, 2, 5, "cuda")
    api.presto_expand(t, torch.zeros((0, 64), device="cuda"),
                      torch.zeros((0, 2, 64), device="cuda"), 1.0, 1.0, 2)


def test_largest_tree_deterministic_drafts():
    """1024 nodes (the cap): wide top-k trees, every level."""
    c = to_device(synth.tree_case(4, 1024, 3000, torch.float32, 1.0, seed=41,
                                  sigma_t=0.3, sigma_d=0.3, branch=40,
                                  max_depth=4))
    o = oracle.verify_tree_det(synth.host_logits(c.target), host(c.parent),
                               host(c.node_tokens), host(c.uniforms), 1.0)
    compare(api.verify_tree_det(c.target, c.parent, c.node_tokens,
                                c.uniforms, 1.0), o, extra_equal=("nodes",))


def test_largest_trie():
    """K = 32 candidates, gamma = 31: 993 nodes."""
    c = to_device(synth.kcand_case(3, 32, 31, 256, torch.float32, 1.0,
                                   seed=42, sigma_t=1.0, sigma_d=0.5,
                                   sigma_k=0.3))
    o = oracle.verify_kcand_trie(synth.host_logits(c.target),
                                 synth.host_logits(c.draft), host(c.tokens),
                                 host(c.uniforms), 1.0)
    g = api.verify_kcand_trie(c.target, c.draft, c.tokens, c.uniforms, 1.0)
    compare(g, o, extra_equal=("k",))


def test_presto_largest_proposal_set():
    """W = 64 paths x b = 16 tokens = 1024 proposals per depth (the cap).
    Their scores are dense, so the order among them (node ids, frontier
    slots) is set by near-ties; with the same log rho row for every path
    the expansion does not depend on the slot order, and the nodes of each
    depth (tokens, path scores) must match as sets."""
    B, D, W, V, b = 4, 3, 64, 5000, 16
    g = torch.Generator().manual_seed(43)
    q = torch.randn((B, D, V), generator=g) * 8.0
    rho1 = torch.log(torch.rand((D, B, 1, V), generator=g) * 0.99 + 0.01)
    rho = rho1.expand(D, B, W, V).contiguous()
    gt = api.PrestoTree(B, W, 2000, "cuda")
    ot = oracle.PrestoTree(B, W, 2000)
    for d in range(D):
        n0 = host(gt.n_nodes).copy()
        api.presto_expand(gt, q.cuda()[:, d], rho[d].cuda(), 1.0, 0.5, b)
        oracle.presto_expand(ot, np.ascontiguousarray(q[:, d].numpy()),
                             rho[d].numpy(), 1.0, 0.5, b)
        gn = host(gt.n_nodes)
        np.testing.assert_array_equal(gn, ot.n_nodes)
        for s_ in range(B):
            new = slice(int(n0[s_]), int(gn[s_]))
            np.testing.assert_array_equal(
                np.sort(host(gt.node_tokens)[s_, new]),
                np.sort(ot.node_tokens[s_, new]))
            np.testing.assert_allclose(
                np.sort(host(gt.node_score)[s_, new]),
                np.sort(ot.node_score[s_, new]), rtol=1e-5, atol=1e-4)
    assert int(gn[0]) == 1 + 16 + 256 + 1024


def test_fork_wider_than_vocabulary():
    z = torch.randn((5, 40), generator=torch.Generator().manual_seed(44))
    x = torch.tensor([0, 1, 2, 3, 39], dtype=torch.int32)
    g = api.branch_fork(z.cuda(), x.cuda(), 1.0, 64)
    o = oracle.branch_fork(z.numpy(), x.numpy(), 1.0, 64)
    np.testing.assert_array_equal(host(g["k"]), o["k"])
    np.testing.assert_array_equal(host(g["tokens"]), o["tokens"])
    assert host(g["k"]).max() <= 40


def test_refused_arguments():
    with pytest.raises(api.SdError):  # K = 33 candidates
        api.verify_kcand_trie(torch.zeros((1, 33, 2, 64), device="cuda"),
                              torch.zeros((1, 1, 64), device="cuda"),
                              torch.zeros((1, 33, 1), dtype=torch.int32,
                                          device="cuda"),
                              torch.zeros((1, 33, 2), device="cuda"), 1.0)
    t = api.PrestoTree(1, 64, 10, "cuda")
    with pytest.raises(api.SdError):  # W b = 64 x 17 > 1024
        api.presto_expand(t, torch.zeros((1, 64), device="cuda"),
                          torch.zeros((1, 64, 64), device="cuda"), 1.0, 1.0,
                          17)
    with pytest.raises(api.SdError):  # T = 0 has no log q
        api.presto_expand(t, torch.zeros((1, 64), device="cuda"),
                          torch.zeros((1, 64, 64), device="cuda"), 0.0, 1.0,
                          2)
    with pytest.raises(api.SdError):  # k_max above 64
        api.branch_fork(torch.zeros((1, 64), device="cuda"),
                        torch.zeros(1, dtype=torch.int32, device="cuda"),
                        1.0, 65)
