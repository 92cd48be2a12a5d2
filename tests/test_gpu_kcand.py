"""Parity of sd_verify_kcand (CUDA, through the C ABI) with the oracle:
K candidates verified against shared draft marginals, the longest accepted
streak kept (lowest k on ties), then its correction or bonus token."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_temperature_gb300 import api, synth
from tests.parity import (assert_flag_fraction, compare, host,
                          oracle_over_threads, to_device)

pytestmark = pytest.mark.gpu


def kc_oracle(c):
    return oracle.verify_kcand(synth.host_logits(c.target),
                               synth.host_logits(c.draft), host(c.tokens),
                               host(c.uniforms), c.T)


def run(c, **kw):
    return api.verify_kcand(c.target, c.draft, c.tokens, c.uniforms, c.T, **kw)


@pytest.mark.parametrize("T", [0.0, 0.6, 1.0])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("K,gamma,V", [(1, 5, 300), (3, 4, 1001), (8, 6, 5000),
                                       (8, 0, 700), (5, 1, 64)])
def test_small_cases(T, dtype, K, gamma, V):
    c = to_device(synth.kcand_case(40, K, gamma, V, dtype, T, seed=K * 100 + V,
                                   sigma_t=2.0, sigma_d=1.0, sigma_k=0.7))
    compare(run(c), kc_oracle(c), extra_equal=("k", "n_per_cand"))


def test_one_candidate_equals_linear():
    c = to_device(synth.kcand_case(64, 1, 6, 2000, torch.bfloat16, 1.0,
                                   seed=3))
    gk = run(c)
    gl = api.verify_linear(c.target[:, 0].contiguous(), c.draft,
                           c.tokens[:, 0].contiguous(),
                           c.uniforms[:, 0].contiguous(), 1.0)
    assert torch.equal(gk["n"], gl["n"]) and torch.equal(gk["tokens"],
                                                         gl["tokens"])
    assert torch.all(gk["k"] == 0)


def test_kcand_workload_every_sequence():
    """B=64, K=8, gamma=16, V=152064 bf16, T=1 (the diffusion self-selection
    workload, full size on the device, the benchmark's launch): all 64
    sequences against the oracle (host threads), the per-candidate counts
    included, and the accept-flagged fraction held to the bar."""
    c = synth.kcand(0, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = run(c, status=st)
    assert int(st.item()) == 0
    npc = host(g["n_per_cand"])
    assert np.array_equal(host(g["n"]), npc.max(1))
    t, d = synth.host_logits(c.target), synth.host_logits(c.draft)
    tk, u = host(c.tokens), host(c.uniforms)
    o = oracle_over_threads(lambda lo, hi: oracle.verify_kcand(
        t[lo:hi], d[lo:hi], tk[lo:hi], u[lo:hi], 1.0), 64)
    r = compare(g, o, extra_equal=("k", "n_per_cand"))
    assert r["seqs"] == 64
    assert_flag_fraction(r)


def test_invalid_rows_and_bad_tokens():
    c = synth.kcand_case(6, 3, 4, 500, torch.float32, 1.0, seed=8)
    c.target[1, 2, 0, 7] = float("nan")        # candidate 2's first row
    c.draft[2, 1, 3] = float("inf")             # shared draft row 1
    c.tokens[3, 0, 0] = 500                     # bad token
    c.target[4, 0, 0, :] = -float("inf")
    to_device(c)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = run(c, status=st)
    o = kc_oracle(c)
    compare(g, o, extra_equal=("k", "n_per_cand"))
    assert int(st.item()) & api.DEV_NONFINITE
    assert int(st.item()) & api.DEV_BAD_TOKEN


@pytest.mark.parametrize("cluster", ["1", "2", "8"])
def test_streaming_kernel_cluster_sizes(cluster):
    """The streaming kernel (aligned rows) split over 1, 2 and 8 CTAs."""
    for T in (0.0, 1.0):
        c = to_device(synth.kcand_case(12, 5, 6, 40000, torch.bfloat16, T,
                                       seed=int(cluster), sigma_t=2.0,
                                       sigma_d=1.0, sigma_k=0.7))
        with api.tuned(cluster=int(cluster)):
            g = run(c)
        compare(g, kc_oracle(c), extra_equal=("k", "n_per_cand"))


def test_streaming_kernel_work_queue():
    """More sequences than resident clusters."""
    c = to_device(synth.kcand_case(700, 3, 3, 2048, torch.float32, 1.0,
                                   seed=11, sigma_t=2.0, sigma_d=1.0,
                                   sigma_k=0.7))
    r = compare(run(c), kc_oracle(c), extra_equal=("k", "n_per_cand"))
    assert r["acc_flagged"] / r["seqs"] < 5e-3


def test_plain_load_kernel_on_aligned_rows():
    """SD_TUNE_KCAND_RING 0 sends aligned rows to the plain-load kernel."""
    c = to_device(synth.kcand_case(16, 4, 5, 4096, torch.bfloat16, 0.8,
                                   seed=12, sigma_t=2.0, sigma_d=1.0,
                                   sigma_k=0.7))
    with api.tuned(kcand_ring=0):
        g = run(c)
    compare(g, kc_oracle(c), extra_equal=("k", "n_per_cand"))


@pytest.mark.parametrize("B,K,gamma,V,dtype", [
    (64, 8, 16, 152064, torch.bfloat16),  # the workload's shape: one wave
    (300, 8, 8, 20000, torch.float32),    # the work counter
    (40, 31, 6, 8192, torch.bfloat16)])   # the widest candidate mask helped
def test_helping_same_bits(B, K, gamma, V, dtype):
    """Clusters whose sequence is done compute rows of positions ahead of
    the scans still running (SD_TUNE_HELPERS): the outputs with and without
    helping are the same bits, and equal the oracle's."""
    c = to_device(synth.kcand_case(B, K, gamma, V, dtype, 1.0, seed=B + K,
                                   sigma_t=3.0, sigma_d=1.0, sigma_k=0.5))
    outs = []
    for h in (1, 0, 1):
        with api.tuned(helpers=h):
            outs.append(run(c))
    for g in outs[1:]:
        for k in outs[0]:
            assert torch.equal(g[k], outs[0][k]), k
    compare(outs[0], kc_oracle(c), extra_equal=("k", "n_per_cand"))
