"""Failure detection without a fault: a bounded wait that can never
complete (an mbarrier no copy targets, nothing in flight) gives up after
its poll limit, reports SD_DEV_TIMEOUT through the status word, and the
kernel returns; the context stays usable for the next verify."""
import pytest
import torch

from speculative_decoding_verification_temperature_gb300 import api, synth
from tests.parity import compare, linear_oracle, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("polls", [1, 1000, 100000])
def test_bounded_wait_gives_up_and_reports(polls):
    status, gave_up, finished = api.selftest_bounded_wait(polls)
    assert status == api.DEV_TIMEOUT
    assert gave_up == 256 and finished == 1
    # the context is still usable: an ordinary verify right after
    c = to_device(synth.linear_case(8, 3, 1000, torch.float32, 1.0, seed=1,
                                    sigma_t=2.0, sigma_d=1.0))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = api.verify_linear(c.target, c.draft, c.tokens, c.uniforms, 1.0,
                          status=st)
    compare(g, linear_oracle(c))
    assert int(st.item()) == 0


def test_bounded_wait_argument_checks():
    L = api.lib()
    out = torch.zeros(2, dtype=torch.int32, device="cuda")
    for polls in (0, -5, (1 << 20) + 1):
        assert L.sd_selftest_bounded_wait(polls, None, out.data_ptr(),
                                          None) == api.SD_ERR_INVALID_ARG
    assert L.sd_selftest_bounded_wait(10, None, None,
                                      None) == api.SD_ERR_INVALID_ARG
