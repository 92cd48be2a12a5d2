"""Parity of sd_verify_linear_fanout (linear verify fused with the fan-out of
the same draft logits; CUDA, through the C ABI) with the fp64 oracle's
linear verify and top-F selection: the large workload (B=256, gamma=8,
V=128256 fp32, F=[10,9,8,7,6,6,5,4,9]) on sampled sequences, the linear
workload's shape with a lookahead draft row at T in {0, 0.7, 1}, small and
odd sizes, gamma 0 and 1, F with empty and 64-wide rows, every cluster
size, the work queue, NaN rows in the draft and the target, and the
two-call path taken when the fused kernel does not apply (rows not 16-byte
aligned, SD_TUNE_FUSED 0)."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_temperature_gb300 import api, synth
from tests.parity import compare, host, to_device

pytestmark = pytest.mark.gpu

F_LARGE = [10, 9, 8, 7, 6, 6, 5, 4, 9]


@pytest.fixture(autouse=True)
def fused_kernel():
    """These tests exercise the fused kernel (SD_TUNE_FUSED 1, the
    default) unless a test switches it off."""
    with api.tuned(fused=1):
        yield


def run(c, F, **kw):
    return api.verify_linear_fanout(c.target, c.draft, c.tokens, c.uniforms,
                                    c.T, F, **kw)


def check(c, F, g=None, idx=None):
    """Compare the fused outputs with the oracle (on sequences idx)."""
    if g is None:
        g = run(c, F)
    gamma = c.target.shape[1] - 1
    sel = slice(None) if idx is None else idx
    tgt = synth.host_logits(c.target[sel])
    dft = synth.host_logits(c.draft[sel])
    o = oracle.verify_linear(tgt, None if c.T == 0 else
                             np.ascontiguousarray(dft[:, :gamma]),
                             host(c.tokens[sel]), host(c.uniforms[sel]), c.T)
    gv = {k: g[k][sel] for k in ("n", "tokens", "prob")}
    r = compare(gv, o)
    fo = oracle.fanout_topk(dft, np.array(F, np.int32))
    np.testing.assert_array_equal(host(g["fan_tokens"][sel]), fo["tokens"])
    ok = fo["tokens"] >= 0
    np.testing.assert_array_equal(
        host(g["fan_logit"][sel]).astype(np.float64)[ok], fo["logit"][ok])
    return r


def test_large_workload_sampled():
    c = synth.large(0, device="cuda")
    g = run(c, F_LARGE)
    idx = torch.tensor([0, 1, 2, 3, 77, 128, 129, 200, 254, 255],
                       device="cuda")
    r = check(c, F_LARGE, g, idx)
    assert r["acc_flagged"] <= 1


@pytest.mark.parametrize("T", [0.0, 0.7, 1.0])
def test_linear_workload_shape(T):
    c = to_device(synth.linear_case(32, 8, 32000, torch.bfloat16, T,
                                    seed=1001, sigma_t=3.0, sigma_d=1.5,
                                    spike=8.0, draft_rows=9))
    r = check(c, F_LARGE)
    assert r["acc_flagged"] <= 1


@pytest.mark.parametrize("V,dtype", [(1000, torch.float32),
                                     (4100, torch.float32),
                                     (4104, torch.bfloat16),
                                     (50000, torch.bfloat16)])
@pytest.mark.parametrize("gamma", [0, 1, 5])
def test_sizes(V, dtype, gamma):
    c = to_device(synth.linear_case(24, gamma, V, dtype, 1.0, seed=V + gamma,
                                    sigma_t=2.0, sigma_d=1.0,
                                    draft_rows=gamma + 1))
    F = [min(V, f) for f in [3, 0, 64, 1, 7, 2][:gamma + 1]]
    check(c, F)


@pytest.mark.parametrize("cluster", ["1", "2", "4", "8", "16"])
def test_cluster_sizes(cluster):
    c = to_device(synth.linear_case(20, 6, 40000, torch.float32, 0.8,
                                    seed=int(cluster), sigma_t=2.0,
                                    sigma_d=1.0, draft_rows=7))
    with api.tuned(cluster=int(cluster)):
        check(c, [64, 1, 5, 0, 33, 8, 2])


def test_queue_many_sequences():
    """More sequences than resident clusters: the work counter."""
    c = to_device(synth.linear_case(1500, 4, 2048, torch.float32, 1.0,
                                    seed=5, sigma_t=2.0, sigma_d=1.0,
                                    draft_rows=5))
    r = check(c, [4, 3, 2, 2, 5])
    assert r["acc_flagged"] / r["seqs"] < 5e-3


def test_nan_rows():
    """NaN in a draft row after the rejection (fan-out flags it, the verify
    is unaffected), NaN in a target row (the verify flags it), NaN in the
    lookahead draft row."""
    c = synth.linear_case(6, 4, 3000, torch.float32, 1.0, seed=9,
                          sigma_t=2.0, sigma_d=1.0, draft_rows=5)
    c.draft[0, 4, 17] = float("nan")
    c.target[1, 0, 5] = float("nan")
    c.draft[2, 3, 2999] = float("nan")
    c = to_device(c)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = run(c, [3, 3, 3, 3, 3], status=st)
    check(c, [3, 3, 3, 3, 3], g)
    assert int(st.item()) & api.DEV_NONFINITE


def test_fallback_path_matches():
    """The two separate calls (SD_TUNE_FUSED 0, the default) and an
    unaligned vocabulary (no fused kernel); both agree with the oracle."""
    c = to_device(synth.linear_case(16, 3, 6000, torch.bfloat16, 1.0, seed=3,
                                    sigma_t=2.0, sigma_d=1.0, draft_rows=4))
    with api.tuned(fused=0):
        check(c, [5, 4, 3, 2])
    c = to_device(synth.linear_case(16, 3, 6001, torch.float32, 1.0, seed=4,
                                    sigma_t=2.0, sigma_d=1.0, draft_rows=4))
    check(c, [5, 4, 3, 2])


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_large_workload_every_sequence(T):
    """The bench's launch: all 256 sequences and all 2304 fan-out rows of the
    large workload against the oracle, at T = 1 and greedy."""
    c = synth.large(0, device="cuda")
    if T == 0:
        c.T = 0.0
    r = check(c, F_LARGE)
    assert r["acc_flagged"] <= 2


def test_fused_matches_two_calls_bitwise():
    """The fused kernel and the two calls give the same bits (verify and
    fan-out), on a queue-sized batch."""
    c = to_device(synth.linear_case(300, 8, 50000, torch.float32, 1.0,
                                    seed=12, sigma_t=2.5, sigma_d=1.0,
                                    draft_rows=9))
    F = [10, 9, 8, 7, 6, 6, 5, 4, 9]
    g = run(c, F)
    with api.tuned(fused=0):
        h = run(c, F)
    for k in ("n", "tokens", "prob", "fan_tokens", "fan_logit"):
        assert torch.equal(g[k], h[k]) or (
            k == "fan_logit" and torch.equal(g[k].isnan(), h[k].isnan())
            and torch.equal(g[k].nan_to_num(), h[k].nan_to_num())), k


@pytest.mark.parametrize("dtype,run_len", [(torch.float32, 4),
                                           (torch.bfloat16, 8)])
def test_top_run_in_one_vector(dtype, run_len):
    """A run of large, decreasing logits inside one 16-byte vector of every
    draft row: the row's best keys all come from one thread's elements.
    F wider and narrower than the run, against the oracle."""
    c = synth.linear_case(40, 4, 8192, dtype, 1.0, seed=21, sigma_t=2.0,
                          sigma_d=1.0, draft_rows=5)
    base = 64 * run_len  # the start of a vector
    for b in range(c.draft.shape[0]):
        for r in range(c.draft.shape[1]):
            for e in range(run_len):
                c.draft[b, r, base + e] = 40.0 - e
    c = to_device(c)
    check(c, [6, 6, 2, 9, 3])
    check(c, [2, 2, 2, 2, 2])
