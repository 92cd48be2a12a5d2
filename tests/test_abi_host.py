"""Host-side checks of the C ABI that need no GPU: the library loads and
exports every entry point include/sd_verify.h declares, argument validation
rejects bad calls before any launch, the host-only fan-out schedule
matches the oracle, and the Python binding refuses host tensors (there is
no CPU path)."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_temperature_gb300 import api

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include",
                      "sd_verify.h")


def declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sd_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    L = api.lib()
    names = declared()
    assert len(names) >= 13
    for n in names:
        assert hasattr(L, n), n


def test_version_and_last_error():
    assert "sm_103a" in api.version()
    L = api.lib()
    rc = L.sd_verify_linear(None, None, 0, None, None, 1, 4, 0, 1.0, None,
                            None, None, None, None, None, None, 0, None)
    assert rc == api.SD_ERR_INVALID_ARG
    assert b"V=0" in L.sd_last_error()


@pytest.mark.parametrize("args", [
    dict(B=-1), dict(gamma=-1), dict(gamma=65), dict(V=0), dict(V=1 << 25),
    dict(T=-1.0), dict(T=float("nan")), dict(T=float("inf")), dict(dt=7),
    dict(target=None), dict(draft=None), dict(tokens=None), dict(uni=None),
])
def test_linear_validation(args):
    L = api.lib()
    p = ctypes.c_void_p(16)
    a = dict(target=p, draft=p, dt=0, tokens=p, uni=p, B=2, gamma=3, V=100,
             T=1.0)
    a.update(args)
    rc = L.sd_verify_linear(a["target"], a["draft"], a["dt"], a["tokens"],
                            a["uni"], a["B"], a["gamma"], a["V"], a["T"], p,
                            p, None, None, None, None, p, 256, None)
    assert rc == api.SD_ERR_INVALID_ARG, args


def test_empty_batch_is_a_no_op():
    L = api.lib()
    rc = L.sd_verify_linear(None, None, 0, None, None, 0, 3, 100, 1.0, None,
                            None, None, None, None, None, None, 0, None)
    assert rc == api.SD_OK


@pytest.mark.parametrize("K,budget,a,r", [
    (8, 64, 0.8, 1.0), (4, 20, 0.6, 0.5), (6, 40, 0.7, 1.0),
    (8, 128, 0.9, 2.0), (0, 5, 0.5, 1.0), (3, 0, 0.5, 1.0), (32, 1000, 0.95, 1.0),
    (2, 9, 0.5, 1.0), (5, 7, 0.3, 3.0)])
def test_fanout_schedule_matches_oracle(K, budget, a, r):
    F = api.fanout_schedule(K, budget, a, r)
    assert F == [int(x) for x in oracle.fanout_schedule(K, budget, a, r)]
    assert sum(F) == budget


@pytest.mark.parametrize("K,budget,a,r", [
    (-1, 5, 0.5, 1.0), (33, 5, 0.5, 1.0), (3, -1, 0.5, 1.0),
    (3, 5, 0.0, 1.0), (3, 5, 1.0, 1.0), (3, 5, 0.5, 0.0)])
def test_fanout_schedule_rejects(K, budget, a, r):
    with pytest.raises(api.SdError):
        api.fanout_schedule(K, budget, a, r)


@pytest.mark.parametrize("B,gamma,V,dt", [
    (1, 4, 1000, 0), (32, 8, 32000, 1), (7, 3, 1001, 0), (300, 2, 640, 0),
    (256, 8, 128256, 0), (64, 16, 152064, 1)])
def test_linear_workspace_covers_both_paths(B, gamma, V, dt):
    """The workspace query is host-only: it covers the all-rows path's
    slice states (B rows S AM entries) whenever that path may be taken, and
    never asks for less than 256 bytes."""
    L = api.lib()
    w = L.sd_verify_linear_workspace(B, gamma, V, dt)
    assert w >= 256
    eb = 4 if dt == 0 else 2
    rows = 2 * gamma + 1
    if B * rows * V * eb <= 64 << 20:
        smax = min(32, max(1, V // 256))
        assert w >= B * rows * smax * 12


def test_workspace_queries_cover_helping_and_records():
    """The queries size the scratch of every path a call may take: the
    linear verify's helping records (flags and 16-byte partials per
    sequence, position and CTA rank), the fused step's scan records (24
    bytes per scan thread and draft row, clusters of 8 at these sizes) and
    the K-candidate verify's helping records (none for K = 32)."""
    L = api.lib()
    B, gamma = 256, 8
    w = L.sd_verify_linear_workspace(B, gamma, 128256, 0)
    assert w >= B * (gamma + 1) * 16 * (4 + 16)
    f = L.sd_verify_linear_fanout_workspace(B, gamma, 128256, 0)
    assert f >= B * gamma * 8 * 256 * 24 and f >= w
    k = L.sd_verify_kcand_workspace(64, 8, 16, 152064, 1)
    assert k >= 64 * 16 * 9 * 16 * (4 + 8)
    assert L.sd_verify_kcand_workspace(64, 32, 16, 152064, 1) == 256


def test_later_workspace_queries_are_host_only():
    L = api.lib()
    assert L.sd_verify_kcand_trie_workspace(64, 8, 16, 152064, 1) >= \
        256 + 6 * 64 * (1 + 8 * 16) * 4
    assert L.sd_presto_expand_workspace(16, 8, 151936, 4, 1) >= 16 * 8 * 4 * 8
    assert L.sd_branch_fork_workspace(64, 152064, 8, 1) >= 64 * 8 * 8
    assert L.sd_verify_tree_det_workspace(16, 64, 151936, 1) >= 256


def test_later_entry_points_validate_before_launch():
    """Bad arguments are refused on the host (no device needed)."""
    L = api.lib()
    p = ctypes.c_void_p(16)
    # K = 33 candidates (at most 32)
    assert L.sd_verify_kcand_trie(p, p, 0, p, p, 1, 33, 2, 64, 1.0, p, p, p,
                                  None, None, p, 1 << 20, None) \
        == api.SD_ERR_INVALID_ARG
    # 1 + K gamma above the tree node cap
    assert L.sd_verify_kcand_trie(p, p, 0, p, p, 1, 32, 40, 64, 1.0, p, p, p,
                                  None, None, p, 1 << 20, None) \
        == api.SD_ERR_UNSUPPORTED
    # PRESTO: T = 0 has no log q; W b above 1024
    assert L.sd_presto_expand(p, 64, p, 0, 1, 4, 64, 0.0, 1.0, 2, 10, p, p,
                              p, p, p, p, None, p, 1 << 20, None) \
        == api.SD_ERR_INVALID_ARG
    assert L.sd_presto_expand(p, 64, p, 0, 1, 64, 64, 1.0, 1.0, 17, 10, p,
                              p, p, p, p, p, None, p, 1 << 20, None) \
        == api.SD_ERR_UNSUPPORTED
    # fork: k_max above 64
    assert L.sd_branch_fork(p, 0, p, 1, 64, 1.0, 65, p, p, None, p, 1 << 20,
                            None) == api.SD_ERR_INVALID_ARG
    # empty batches are no-ops
    assert L.sd_verify_tree_det(None, 0, None, None, None, 0, 3, 64, 1.0,
                                None, None, None, None, None, None, 0,
                                None) == api.SD_OK


def _cpu_calls():
    """One call of every Python entry point, with CPU tensors."""
    from speculative_decoding_verification_temperature_gb300 import api
    B, g, V = 2, 3, 64
    i32 = dict(dtype=torch.int32)
    t, d = torch.zeros(B, g + 1, V), torch.zeros(B, g, V)
    x, u = torch.zeros(B, g, **i32), torch.full((B, g + 1), 0.5)
    kt, kx = torch.zeros(B, 2, g + 1, V), torch.zeros(B, 2, g, **i32)
    ku = torch.full((B, 2, g + 1), 0.5)
    par = torch.tensor([[-1, 0, 0, 1]] * B, **i32)
    nt, nu = torch.zeros(B, 4, **i32), torch.full((B, 4), 0.5)
    return {
        "verify_linear": lambda: api.verify_linear(t, d, x, u, 1.0),
        "verify_linear_static":
            lambda: api.verify_linear_static(t, d, x, u, 1.0),
        "verify_linear_filtered":
            lambda: api.verify_linear_filtered(t, d, x, u, 1.0, 5),
        "verify_linear_fanout": lambda: api.verify_linear_fanout(
            t, torch.zeros(B, g + 1, V), x, u, 1.0, [2] * (g + 1)),
        "verify_kcand": lambda: api.verify_kcand(kt, d, kx, ku, 1.0),
        "verify_kcand_trie":
            lambda: api.verify_kcand_trie(kt, d, kx, ku, 1.0),
        "verify_tree": lambda: api.verify_tree(
            torch.zeros(B, 4, V), torch.zeros(B, 4, V), par, nt, nu, 1.0),
        "verify_tree_det": lambda: api.verify_tree_det(
            torch.zeros(B, 4, V), par, nt, nu, 1.0),
        "branch_fork": lambda: api.branch_fork(
            torch.zeros(B, V), torch.zeros(B, **i32), 1.0, 4),
        "fanout_topk": lambda: api.fanout_topk(torch.zeros(B, 3, V),
                                               [2, 2, 2]),
        "fanout_hits": lambda: api.fanout_hits(
            torch.zeros(B, **i32), torch.zeros(B, 3, **i32),
            torch.zeros(B, 6, **i32), [2, 2, 2]),
        "PrestoTree": lambda: api.PrestoTree(B, 2, 10, "cpu"),
    }


@pytest.mark.parametrize("name", sorted(_cpu_calls()))
def test_binding_refuses_cpu_tensors(name):
    """There is no CPU path: every entry point of the binding refuses host
    tensors with a ValueError before anything reaches the library."""
    with pytest.raises(ValueError, match="CUDA"):
        _cpu_calls()[name]()


def test_tuning_switches_set_get_and_validate():
    """sd_tune_set / sd_tune_get: defaults, a round trip, unknown keys and
    out-of-range values refused, and nothing read from the environment."""
    L = api.lib()
    defaults = {"cluster": 0, "no_tma": 0, "allrows": 1, "spec": 1,
                "fused": 1, "kcand_ring": 1, "fanout_cluster": 0,
                "fanout_ldg": 0, "fanout_maxc": 0, "fanout_l2_first": 1}
    for k, v in defaults.items():
        assert api.tune_get(k) == v, k
    with api.tuned(cluster=4, allrows=2):
        assert api.tune_get("cluster") == 4 and api.tune_get("allrows") == 2
    assert api.tune_get("cluster") == 0 and api.tune_get("allrows") == 1
    assert L.sd_tune_set(99, 1) == api.SD_ERR_INVALID_ARG
    assert L.sd_tune_get(99) == -1
    assert L.sd_tune_set(api.TUNE["cluster"], 3) == api.SD_ERR_INVALID_ARG
    assert L.sd_tune_set(api.TUNE["spec"], 3) == api.SD_ERR_INVALID_ARG
    assert L.sd_tune_set(api.TUNE["fused"], -1) == api.SD_ERR_INVALID_ARG
    assert api.tune_get("cluster") == 0
    src = "".join(open(f).read() for f in sorted(__import__("glob").glob(
        os.path.join(os.path.dirname(api.__file__), "csrc", "*.cu*"))))
    assert "getenv" not in src
