"""sd_verify_linear_static (scratch in a static device array, no workspace)
against sd_verify_linear on the same inputs: identical results on two calls
in a row, with the work queue in use (more sequences than resident
clusters), on both linear paths; the scratch limit checked on the host.
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
@pytest.mark.parametrize("allrows", [0, 2])
def test_static_matches_workspace_entry_twice(dtype, T, allrows):
    c = synth.linear_case(1024, 4, 4096, dtype=dtype, T=T, seed=11,
                          device="cuda")
    draft = None if T == 0.0 else c.draft
    with api.tuned(allrows=allrows):
        ref = api.verify_linear(c.target, draft, c.tokens, c.uniforms, T,
                                want_accept=True)
        for _ in range(2):
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            got = api.verify_linear_static(c.target, draft, c.tokens,
                                           c.uniforms, T, want_accept=True,
                                           status=st)
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


def test_static_scratch_covers_every_size():
    """The scratch the verify needs (sd_verify_linear_workspace) stays within
    SD_STATIC_WS_BYTES at every size up to the library's limits, so the
    static entry accepts whatever the workspace entry accepts; a call is
    still validated on the host before anything is launched (null pointers
    with a bad gamma: refused without touching them)."""
    L = api.lib()
    for B in (1, 7, 256, 4096, 65536, 1 << 20):
        for gamma in (0, 1, 8, 64):
            for V in (1, 1000, 32000, 152064, 1 << 24):
                for dt in (api.SD_F32, api.SD_BF16):
                    assert L.sd_verify_linear_workspace(B, gamma, V, dt) <= \
                        (1 << 20), (B, gamma, V, dt)
    rc = L.sd_verify_linear_static(None, None, api.SD_BF16, None, None, 4,
                                   65, 1000, 1.0, None, None, None, None,
                                   None, None, None)
    assert rc == api.SD_ERR_INVALID_ARG
    assert b"gamma" in L.sd_last_error()
