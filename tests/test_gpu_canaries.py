"""Out-of-bounds write checks for every entry point (a stand-in for a
memory checker): each output and workspace buffer the binding allocates is
the middle of a larger device buffer whose two guard regions hold a
sentinel byte; after each call the guards must be untouched.  Ragged
vocabularies (not a multiple of the 16-byte vector), gamma = 0, every
optional output, both linear paths and both fan-out paths."""
import numpy as np
import pytest
import torch

from speculative_decoding_verification_temperature_gb300 import api, synth
from tests.parity import compare, linear_oracle, to_device

pytestmark = pytest.mark.gpu

GUARD = 4096    # bytes on each side (keeps the payload 512-byte aligned)
SENTINEL = 0xA5


class GuardedTorch:
    """Forwards everything to torch except empty(), which returns the
    middle of a guarded byte buffer; check() verifies every guard."""

    def __init__(self):
        self.bufs = []

    def __getattr__(self, name):
        return getattr(torch, name)

    def empty(self, *shape, dtype=torch.float32, device=None, **kw):
        if len(shape) == 1 and isinstance(shape[0], (tuple, list,
                                                     torch.Size)):
            shape = tuple(shape[0])
        n = int(np.prod(shape)) if shape else 1
        esz = torch.empty((), dtype=dtype).element_size()
        nb = n * esz
        raw = torch.full((2 * GUARD + nb,), SENTINEL, dtype=torch.uint8,
                         device=device)
        self.bufs.append((raw, nb))
        return raw[GUARD:GUARD + nb].view(dtype).view(shape)

    def check(self):
        torch.cuda.synchronize()
        for raw, nb in self.bufs:
            head, tail = raw[:GUARD], raw[GUARD + nb:]
            assert bool((head == SENTINEL).all()), "write below a buffer"
            assert bool((tail == SENTINEL).all()), "write past a buffer"
        n = len(self.bufs)
        self.bufs.clear()
        return n


@pytest.fixture
def guard(monkeypatch):
    g = GuardedTorch()
    monkeypatch.setattr(api, "torch", g)
    return g


def status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("V,dtype", [(1001, torch.float32),
                                     (4099, torch.bfloat16),
                                     (4096, torch.float32)])
@pytest.mark.parametrize("gamma", [0, 3])
@pytest.mark.parametrize("T", [0.0, 1.0])
def test_linear_entries(guard, V, dtype, gamma, T):
    c = to_device(synth.linear_case(37, gamma, V, dtype, T, seed=V + gamma,
                                    sigma_t=2.0, sigma_d=1.0))
    d = None if T == 0 else c.draft
    o = linear_oracle(c)
    for allrows in (0, 2):
        with api.tuned(allrows=allrows):
            g = api.verify_linear(c.target, d, c.tokens, c.uniforms, T,
                                  want_accept=True, want_resid=True,
                                  status=status(),
                                  workspace=api.Workspace())
            assert guard.check() >= 5
            compare(g, o)
            g = api.verify_linear_static(c.target, d, c.tokens, c.uniforms,
                                         T, want_accept=True, status=status())
            assert guard.check() >= 4
            compare(g, o)


@pytest.mark.parametrize("gamma", [0, 3])
def test_filtered(guard, gamma):
    c = to_device(synth.linear_case(19, gamma, 4104, torch.float32, 1.0,
                                    seed=3 + gamma, sigma_t=2.0, sigma_d=1.0))
    for top_k in (7, 1 << 30):
        api.verify_linear_filtered(c.target, c.draft, c.tokens, c.uniforms,
                                   1.0, top_k, 0.9, want_keep=True,
                                   status=status(), workspace=api.Workspace())
        assert guard.check() >= 4


@pytest.mark.parametrize("gamma", [0, 3])
@pytest.mark.parametrize("V", [1001, 4096])
def test_kcand_entries(guard, gamma, V):
    for T in (0.0, 1.0):
        c = to_device(synth.kcand_case(11, 3, gamma, V, torch.bfloat16, T,
                                       seed=V + gamma, sigma_t=2.0,
                                       sigma_d=1.0, sigma_k=0.7))
        api.verify_kcand(c.target, c.draft, c.tokens, c.uniforms, T,
                         status=status(), workspace=api.Workspace())
        assert guard.check() >= 5
        api.verify_kcand_trie(c.target, None if T == 0 else c.draft,
                              c.tokens, c.uniforms, T, status=status(),
                              workspace=api.Workspace())
        assert guard.check() >= 4


@pytest.mark.parametrize("N", [1, 10])
@pytest.mark.parametrize("V", [1001, 4096])
def test_tree_entries(guard, N, V):
    for T in (0.0, 0.8):
        c = to_device(synth.tree_case(5, N, V, torch.float32, T, seed=N + V,
                                      sigma_t=1.0, sigma_d=1.0))
        api.verify_tree(c.target, c.draft, c.parent, c.node_tokens,
                        c.uniforms, T, status=status(),
                        workspace=api.Workspace())
        assert guard.check() >= 4
        api.verify_tree_det(c.target, c.parent, c.node_tokens, c.uniforms, T,
                            status=status(), workspace=api.Workspace())
        assert guard.check() >= 4


@pytest.mark.parametrize("V", [1001, 4096])
def test_fanout_entries(guard, V):
    g = torch.Generator().manual_seed(V)
    d = torch.randn((6, 3, V), generator=g).cuda()
    F = [3, 0, 64]
    f = api.fanout_topk(d, F, want_logit=True, status=status(),
                        workspace=api.Workspace())
    assert guard.check() >= 2
    n = torch.tensor([0, 1, 2, 2, -1, 1], dtype=torch.int32, device="cuda")
    toks = torch.randint(0, V, (6, 3), dtype=torch.int32, device="cuda")
    api.fanout_hits(n, toks, f["tokens"], F)
    assert guard.check() >= 1
    c = to_device(synth.linear_case(9, 2, V, torch.float32, 1.0, seed=V,
                                    sigma_t=2.0, sigma_d=1.0, draft_rows=3))
    for fused in (0, 1):
        with api.tuned(fused=fused):
            api.verify_linear_fanout(c.target, c.draft, c.tokens, c.uniforms,
                                     1.0, [5, 0, 3], status=status(),
                                     workspace=api.Workspace())
            assert guard.check() >= 5


@pytest.mark.parametrize("V", [1001, 4096])
def test_construction_entries(guard, V):
    g = torch.Generator().manual_seed(V)
    B, W = 3, 4
    t = api.PrestoTree(B, W, 9, "cuda")
    for _ in range(3):
        q = torch.randn((B, V), generator=g).cuda()
        rho = torch.log(torch.rand((B, W, V), generator=g) + 0.01).cuda()
        api.presto_expand(t, q, rho, 0.8, 1.0, 3, status=status(),
                          workspace=api.Workspace())
    assert guard.check() >= 6
    z = torch.randn((5, V), generator=g).cuda()
    x = torch.randint(0, V, (5,), dtype=torch.int32).cuda()
    api.branch_fork(z, x, 1.0, 8, status=status(), workspace=api.Workspace())
    assert guard.check() >= 2
