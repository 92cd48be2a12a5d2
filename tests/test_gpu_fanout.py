"""Parity of sd_fanout_topk (CUDA, through the C ABI) with the oracle: the
top-F_k draft tokens of every lookahead row, ordered by (logit desc, id
asc), on the large workload's rows and on rows built to stress the exact
selection (ties, sorted rows, constant rows, NaN, F up to 64)."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_temperature_gb300 import api, synth
from tests.parity import (assert_flag_fraction, compare, host,
                          linear_oracle_full, oracle_over_threads)

pytestmark = pytest.mark.gpu


def check(draft, F):
    g = api.fanout_topk(draft, F, want_logit=True)
    o = oracle.fanout_topk(synth.host_logits(draft), np.array(F, np.int32))
    np.testing.assert_array_equal(host(g["tokens"]), o["tokens"])
    ok = o["tokens"] >= 0
    np.testing.assert_array_equal(host(g["logit"])[ok].astype(np.float64),
                                  o["logit"][ok])
    return g, o


def test_large_step_every_row():
    """The benchmark's step on the large workload (B=256, V=128256 fp32):
    the fan-out over all 2304 draft rows on a second stream beside the
    linear verify, each with its own workspace, exactly as timed; every
    row's top-F_k (F = [10,9,8,7,6,6,5,4,9]) and every sequence's verify
    against the oracle (host threads)."""
    c = synth.large(0, device="cuda")
    F = api.fanout_schedule(8, 64, 0.8, 1.0)
    assert F == [10, 9, 8, 7, 6, 6, 5, 4, 9]
    draft_v = c.draft[:, :8].contiguous()
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    ws_v, ws_f = api.Workspace(), api.Workspace()
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    fork = torch.cuda.Event()
    fork.record(main)
    side.wait_event(fork)
    with torch.cuda.stream(side):
        f = api.fanout_topk(c.draft, F, want_logit=True, status=st[1:],
                            workspace=ws_f)
    g = api.verify_linear(c.target, draft_v, c.tokens, c.uniforms, 1.0,
                          status=st[:1], workspace=ws_v)
    join = torch.cuda.Event()
    join.record(side)
    main.wait_event(join)
    torch.cuda.synchronize()
    assert host(st).tolist() == [0, 0]
    d = synth.host_logits(c.draft)
    Fa = np.array(F, np.int32)
    of = oracle_over_threads(
        lambda lo, hi: oracle.fanout_topk(d[lo:hi], Fa), d.shape[0])
    np.testing.assert_array_equal(host(f["tokens"]), of["tokens"])
    np.testing.assert_array_equal(host(f["logit"]).astype(np.float64),
                                  of["logit"])
    ov = linear_oracle_full(c.target, draft_v, c.tokens, c.uniforms, 1.0)
    r = compare(g, ov)
    assert r["seqs"] == 256
    assert_flag_fraction(r)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("V", [5, 64, 1000, 4099, 32000, 151936])
def test_random_rows(dtype, V):
    g = torch.Generator().manual_seed(V)
    d = (torch.randn((6, 4, V), generator=g) * 3).to(dtype)
    F = [min(V, f) for f in (10, 1, 0, 64)]
    check(d.cuda(), F)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_ties_sorted_and_constant_rows(dtype):
    """Integer logits (many exact ties), rows sorted ascending and
    descending (the best keys crowd into few threads: exercises the exact
    rescan), constant rows (ties everywhere) and -0 / +0."""
    V = 20000
    g = torch.Generator().manual_seed(1)
    rows = [torch.randint(-5, 6, (V,), generator=g).float(),
            torch.arange(V).float(),
            -torch.arange(V).float(),
            torch.zeros(V),
            torch.where(torch.arange(V) % 2 == 0, torch.tensor(-0.0),
                        torch.tensor(0.0))]
    d = torch.stack(rows)[:, None, :].expand(5, 3, V).contiguous().to(dtype)
    check(d.cuda(), [64, 17, 1])


def test_nan_row_and_status():
    d = torch.randn((3, 2, 3000))
    d[1, 0, 123] = float("nan")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = api.fanout_topk(d.cuda(), [5, 3], status=st)
    o = oracle.fanout_topk(d.numpy(), np.array([5, 3], np.int32))
    np.testing.assert_array_equal(host(out["tokens"]), o["tokens"])
    assert int(st.item()) & api.DEV_NONFINITE


def test_misaligned_rows_scalar_path():
    V = 1003
    d = torch.randn((4, 3, V)) * 2
    check(d.cuda(), [7, 0, 12])


def test_limits_rejected():
    d = torch.randn((2, 2, 100), device="cuda")
    with pytest.raises(api.SdError):
        api.fanout_topk(d, [65, 1])
    with pytest.raises(api.SdError):
        api.fanout_topk(torch.randn((2, 2, 10), device="cuda"), [11, 1])


def test_infinite_rows():
    """Masked (-inf) logits, a row holding both +inf and -inf (a running sum
    turns NaN there without any NaN element: must not be flagged), and a row
    that is -inf everywhere."""
    V = 9000
    g = torch.Generator().manual_seed(7)
    base = torch.randn((4, V), generator=g)
    base[0, ::3] = float("-inf")
    base[1, 17] = float("inf")
    base[1, 4000] = float("-inf")
    base[1, 8999] = float("inf")
    base[2, :] = float("-inf")
    base[3, 100:8000] = float("-inf")
    d = base[:, None, :].expand(4, 2, V).contiguous()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for dtype in (torch.float32, torch.bfloat16):
        dd = d.to(dtype).cuda()
        out = api.fanout_topk(dd, [12, 40], want_logit=True, status=st)
        o = oracle.fanout_topk(synth.host_logits(dd), np.array([12, 40], np.int32))
        np.testing.assert_array_equal(host(out["tokens"]), o["tokens"])
        np.testing.assert_array_equal(host(out["logit"]).astype(np.float64),
                                      o["logit"])
    assert int(st.item()) == 0


@pytest.mark.parametrize("mode", ["ring", "ldg"])
@pytest.mark.parametrize("cluster", ["1", "2", "16"])
def test_streaming_variants_and_clusters(mode, cluster):
    """Both streaming variants (TMA ring, 16-byte loads) with rows split
    over clusters of 1, 2 and 16 CTAs (F = 64 caps the cluster at 8)."""
    g = torch.Generator().manual_seed(int(cluster))
    with api.tuned(fanout_ldg=int(mode == "ldg"),
                   fanout_cluster=int(cluster)):
        for dtype in (torch.float32, torch.bfloat16):
            d = (torch.randn((3, 3, 50000), generator=g) * 2).to(dtype)
            d[0, 1] = torch.arange(50000).to(dtype)  # best keys: last warp
            d[1, 2] = torch.randint(-3, 3, (50000,), generator=g).to(dtype)
            check(d.cuda(), [64, 33, 10])


def test_best_keys_in_one_warp():
    """The top keys all fall in one warp's vectors (every 256th vector
    block), so that warp's list and threshold decide alone."""
    V = 65536
    d = torch.randn((2, 1, V)) - 10
    idx = torch.arange(V)
    sel = ((idx // 4) % 256) // 32 == 3
    d[:, 0, sel] += 20 + torch.rand(int(sel.sum()))
    check(d.cuda(), [64])
    check(d.cuda(), [20])


def test_cache_hits_against_oracle():
    """sd_fanout_hits on the GPU's own verify and fan-out outputs equals the
    oracle's hit function on the same integers, and the whole pipeline
    (verify, fan-out, hits) equals the oracle's pipeline on sequences whose
    draws are not near a boundary."""
    for T in (0.0, 1.0):
        c = synth.linear_case(64, 4, 3000, torch.float32, T, seed=31,
                              sigma_t=2.0, sigma_d=1.0, draft_rows=5)
        cd = synth.LinearCase(c.target.cuda(), c.draft.cuda(),
                              c.tokens.cuda(), c.uniforms.cuda(), T)
        F = [3, 0, 2, 5, 4]
        v = api.verify_linear(cd.target, None if T == 0 else
                              cd.draft[:, :4].contiguous(), cd.tokens,
                              cd.uniforms, T)
        f = api.fanout_topk(cd.draft, F)
        h = host(api.fanout_hits(v["n"], v["tokens"], f["tokens"], F))
        o = oracle.fanout_hits(host(v["n"]), host(v["tokens"]),
                               host(f["tokens"]), np.array(F, np.int32))
        np.testing.assert_array_equal(h, o)
        ov = oracle.verify_linear(
            synth.host_logits(c.target),
            None if T == 0 else np.ascontiguousarray(
                synth.host_logits(c.draft)[:, :4]),
            host(c.tokens), host(c.uniforms), T)
        of = oracle.fanout_topk(synth.host_logits(c.draft),
                                np.array(F, np.int32))
        oh = oracle.fanout_hits(ov["n"], ov["tokens"], of["tokens"],
                                np.array(F, np.int32))
        keep = (ov["margin"] >= oracle.FLAG_MARGIN) | (T == 0)
        np.testing.assert_array_equal(h[keep], oh[keep])
        assert keep.mean() > 0.8


def test_cache_hits_edge_cases():
    """Unusable rows (-1), empty positions, F = 64 wide positions."""
    n = torch.tensor([-1, 0, 1, 2, 2], dtype=torch.int32, device="cuda")
    toks = torch.tensor([[-1, -1, -1], [5, 0, 0], [1, 6, 0], [1, 2, 63],
                         [1, 2, 64]], dtype=torch.int32, device="cuda")
    F = [1, 0, 64]
    fan = torch.zeros((5, 65), dtype=torch.int32, device="cuda")
    fan[:, 0] = 5
    fan[:, 1:] = torch.arange(64, dtype=torch.int32, device="cuda")
    h = host(api.fanout_hits(n, toks, fan, F))
    o = oracle.fanout_hits(host(n), host(toks), host(fan),
                           np.array(F, np.int32))
    np.testing.assert_array_equal(h, o)
    assert h.tolist() == [-1, 1, 0, 1, 0]
