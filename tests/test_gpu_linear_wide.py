"""The position-by-position (level) path of sd_verify_linear (selected with
SDV_WIDE=1) on the small cases and the large workload, compared with the
oracle and, on the large workload, with the cluster path."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_temperature_gb300 import api, synth
from tests.parity import compare, host, linear_oracle, to_device
from tests import test_gpu_linear as base

pytestmark = pytest.mark.gpu


@pytest.fixture
def wide(monkeypatch):
    monkeypatch.setenv("SDV_WIDE", "1")


@pytest.mark.parametrize("T", [0.0, 0.7, 1.0])
def test_linear_workload_wide(wide, T):
    c = to_device(synth.linear(T))
    g = base.run(c, want_accept=True)
    o = linear_oracle(c)
    r = compare(g, o)
    if T == 0:
        assert r["acc_flagged"] == 0 and r["cdf_flagged"] == 0
    ok = o["margin_acc"] >= oracle.FLAG_MARGIN
    ev = (o["accept"] >= 0) & ok[:, None]
    np.testing.assert_allclose(host(g["accept"])[ev], o["accept"][ev],
                               atol=1e-5)
    assert np.all(host(g["accept"])[(o["accept"] < 0) & ok[:, None]] == -1)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("V", [8, 64, 4096, 32000, 70008])
@pytest.mark.parametrize("T", [0.0, 1.3])
def test_vocab_sizes_wide(wide, dtype, V, T):
    for gamma in (0, 1, 3):
        c = to_device(synth.linear_case(40, gamma, V, dtype, T,
                                        seed=V * 10 + gamma, sigma_t=2.0,
                                        sigma_d=1.0))
        compare(base.run(c), linear_oracle(c))


def test_edge_cases_wide(wide):
    base.test_edge_cases()


def test_flagged_fractions_wide(wide):
    base.test_flagged_fractions()


def test_large_workload_both_paths(monkeypatch):
    c = synth.large(0, device="cuda")
    dv = c.draft[:, :8].contiguous()
    outs = []
    for flag in ("1", "0"):
        monkeypatch.setenv("SDV_WIDE", flag)
        outs.append(api.verify_linear(c.target, dv, c.tokens, c.uniforms,
                                      1.0))
    a, b = outs
    idx = [3, 40, 99, 150, 201, 250]
    sub = synth.LinearCase(c.target[idx], c.draft[idx, :8], c.tokens[idx],
                           c.uniforms[idx], 1.0)
    o = linear_oracle(sub)
    compare({k: v[idx] for k, v in a.items()}, o)
    compare({k: v[idx] for k, v in b.items()}, o)
    # the two paths sum in different orders; they agree wherever the oracle
    # does not flag a draw
    same = (a["n"] == b["n"]).float().mean().item()
    assert same > 0.99
