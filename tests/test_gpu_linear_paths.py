"""Both paths of sd_verify_linear against the oracle on the same inputs:
the per-position cluster kernel (SD_TUNE_ALLROWS 0) and the all-rows path
for small inputs (SD_TUNE_ALLROWS 2 forces it wherever its workspace and
shared memory allow), plus the cluster kernel without its read-ahead of a
cluster's last sequence (SD_TUNE_SPEC 0) and with L2 prefetch (2), and
without helping (SD_TUNE_HELPERS 0: clusters with no sequence left compute
row statistics ahead of the running scans, which must not change a bit of
the results).  Small and odd
sizes, both dtypes, unaligned rows, gamma 0, T in {0, 0.7, 1}, bad tokens
and non-finite rows, the queue path, the accept-probability output; and
the two paths agree with each other."""
import numpy as np
import pytest
import torch

from speculative_decoding_verification_temperature_gb300 import api, synth
from tests.parity import compare, host, linear_oracle, to_device

pytestmark = pytest.mark.gpu


def run(case, **kw):
    return api.verify_linear(case.target, None if case.T == 0 else
                             case.draft[:, :case.target.shape[1] - 1]
                             .contiguous(), case.tokens, case.uniforms,
                             case.T, **kw)


def switches(mode):
    sw = {"allrows": int(mode.split("-")[0])}
    if "-spec" in mode:
        sw["spec"] = int(mode[-1])
    if "-help0" in mode:
        sw["helpers"] = 0
    return sw


@pytest.mark.parametrize("mode", ["0", "2", "0-spec0", "0-spec2", "0-help0"])
@pytest.mark.parametrize("T", [0.0, 0.7, 1.0])
@pytest.mark.parametrize("B,gamma,V,dtype", [
    (1, 4, 1000, torch.float32), (32, 8, 32000, torch.bfloat16),
    (7, 3, 1001, torch.float32), (5, 0, 4096, torch.bfloat16),
    (300, 2, 640, torch.float32), (3, 16, 50000, torch.float32)])
def test_paths_against_oracle(mode, T, B, gamma, V, dtype):
    c = to_device(synth.linear_case(B, gamma, V, dtype, T, seed=B + V + gamma,
                                    sigma_t=2.0, sigma_d=1.0))
    with api.tuned(**switches(mode)):
        g = run(c, want_accept=True)
    o = linear_oracle(c)
    r = compare(g, o)
    assert r["acc_flagged"] <= max(1, B // 50)
    if T > 0 and not r["acc_flagged"]:
        ev = o["accept"] >= 0
        np.testing.assert_allclose(host(g["accept"])[ev], o["accept"][ev],
                                   atol=1e-5)
        assert np.all(host(g["accept"])[~ev] == -1)


@pytest.mark.parametrize("mode", ["0", "2", "0-spec0", "0-spec2", "0-help0"])
def test_paths_edge_rows(mode):
    c = synth.linear_case(8, 4, 2000, torch.float32, 1.0, seed=77)
    c.tokens[1, 0] = 10**6            # bad token, tested first
    c.target[2, 1, 5] = float("nan")  # unusable target row
    c.draft[3, 0, 9] = float("inf")   # unusable draft row
    c.target[4, :, 100:] = -float("inf")  # masked tokens
    c = to_device(c)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    with api.tuned(**switches(mode)):
        g = run(c, status=st, want_accept=True)
    compare(g, linear_oracle(c))
    s = int(st.item())
    assert s & api.DEV_NONFINITE and s & api.DEV_BAD_TOKEN


def test_paths_agree():
    """Away from the flagged draws the two paths return the same tokens."""
    c = to_device(synth.linear(1.0))
    outs = []
    for mode in ("0", "2", "0-spec0", "0-spec2"):
        with api.tuned(**switches(mode)):
            outs.append(run(c))
    o = linear_oracle(c)
    keep = host(o["margin_acc"]) >= 1e-5
    keep &= host(o["margin_cdf"]) >= 1e-5
    for k in ("n", "tokens"):
        a = host(outs[0][k])
        for other in outs[1:]:
            assert np.array_equal(a[keep], host(other[k])[keep]), k


@pytest.mark.parametrize("B,gamma,V,dtype,T", [
    (300, 8, 128256, torch.float32, 1.0),    # the large workload's rows
    (300, 8, 128256, torch.float32, 0.0),
    (400, 6, 152064, torch.bfloat16, 0.7),
    (700, 6, 20000, torch.float32, 1.0),
    (700, 4, 1001, torch.float32, 1.0)])     # unaligned rows: plain loads
def test_helping_same_bits(B, gamma, V, dtype, T):
    """More sequences than resident clusters, so clusters help in the work
    counter's tail.  Partials published by helping clusters are the owner's
    own bits: the outputs with and without helping are identical, and equal
    the oracle's."""
    c = to_device(synth.linear_case(B, gamma, V, dtype, T, seed=B * gamma + V,
                                    sigma_t=2.0, sigma_d=1.0))
    outs = []
    for h in (1, 0, 1):
        with api.tuned(helpers=h, allrows=0):
            outs.append(run(c, want_accept=True))
    for g in outs[1:]:
        for k in ("n", "tokens", "prob", "accept"):
            assert torch.equal(g[k], outs[0][k]), k
    compare(outs[0], linear_oracle(c))


def test_helping_with_residual_output():
    c = to_device(synth.linear_case(200, 5, 50000, torch.float32, 1.0, seed=9,
                                    sigma_t=2.0, sigma_d=1.0))
    with api.tuned(helpers=1):
        g = run(c, want_resid=True)
    with api.tuned(helpers=0):
        h = run(c, want_resid=True)
    assert torch.equal(g["resid"], h["resid"])
    assert torch.equal(g["tokens"], h["tokens"])
    compare(g, linear_oracle(c))
