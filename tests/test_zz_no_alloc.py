"""sd_verify_linear_static (scratch in a static device array, no workspace)
against sd_verify_linear on the same inputs: identical results on two calls
in a row, with the work queue in use (more sequences than resident
clusters), on both linear paths, and the size limit rejected on the host.
The file name makes pytest collect it last, so it also runs after every
other test has used the library in the same process."""
import pytest
import torch

from speculative_decoding_verification_temperature_gb300 import api, synth


def _same(a, b):
    for k in ("n", "tokens", "prob"):
        assert torch.equal(a[k], b[k]), k
    if "accept" in a:
        assert torch.equal(a["accept"], b["accept"])


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,T", [(torch.float32, 1.0),
                                     (torch.bfloat16, 0.7),
                                     (torch.float32, 0.0)])
@pytest.mark.parametrize("wide", ["0", "1"])
def test_static_matches_workspace_entry_twice(monkeypatch, dtype, T, wide):
    monkeypatch.setenv("SDV_WIDE", wide)
    c = synth.linear_case(1024, 4, 4096, dtype=dtype, T=T, seed=11,
                          device="cuda")
    draft = None if T == 0.0 else c.draft
    ref = api.verify_linear(c.target, draft, c.tokens, c.uniforms, T,
                            want_accept=True)
    for _ in range(2):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        got = api.verify_linear_static(c.target, draft, c.tokens, c.uniforms,
                                       T, want_accept=True, status=st)
        torch.cuda.synchronize()
        _same(got, ref)
        assert int(st.item()) == 0


@pytest.mark.gpu
def test_static_large_workload_sequences():
    """64 sequences of the large workload's shape (V=128256 fp32) through
    both entry points, alternating."""
    c = synth.large(0, device="cuda")
    t, d = c.target[:64].contiguous(), c.draft[:64, :8].contiguous()
    tok, u = c.tokens[:64].contiguous(), c.uniforms[:64].contiguous()
    ref = api.verify_linear(t, d, tok, u, 1.0)
    _same(api.verify_linear_static(t, d, tok, u, 1.0), ref)
    _same(api.verify_linear(t, d, tok, u, 1.0), ref)
    _same(api.verify_linear_static(t, d, tok, u, 1.0), ref)


def test_static_scratch_limit_rejected_before_any_launch():
    """A size whose scratch exceeds SD_STATIC_WS_BYTES is refused on the
    host (null pointers: nothing may be touched)."""
    L = api.lib()
    B, gamma, V = 65536, 8, 152064
    need = L.sd_verify_linear_workspace(B, gamma, V, api.SD_BF16)
    assert need > (1 << 20)
    rc = L.sd_verify_linear_static(None, None, api.SD_BF16, None, None, B,
                                   gamma, V, 1.0, None, None, None, None, None,
                                   None, None)
    assert rc == api.SD_ERR_UNSUPPORTED
    assert b"SD_STATIC_WS_BYTES" in L.sd_last_error()
