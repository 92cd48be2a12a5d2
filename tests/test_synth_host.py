"""The seeded input generator, on CPU: its splitmix64 stream against the
published outputs of the generator (Steele, Lea and Flood, OOPSLA 2014;
the public-domain reference implementation), and the uniforms it derives
from that stream: ((s >> 41) + 0.5) * 2^-23, inside (0, 1) and exact in
fp32, so that every consumer sees the same numbers."""
import numpy as np

from speculative_decoding_verification_temperature_gb300 import synth


def test_splitmix64_published_outputs():
    # seed 0: the first three outputs of the reference implementation
    assert [int(v) for v in synth.splitmix64(0, 3)] == [
        0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    # seed 1234567: the five outputs that PRNG test suites check
    assert [int(v) for v in synth.splitmix64(1234567, 5)] == [
        6457827717110365317, 3203168211198807973, 9817491932198370423,
        4593380528125082431, 16408922859458223821]


def test_splitmix64_offsets_continue_the_stream():
    whole = synth.splitmix64(99, 10)
    np.testing.assert_array_equal(synth.splitmix64(99, 4, offset=6),
                                  whole[6:])


def test_uniforms_are_the_stream_top_23_bits_centred():
    seed, shape = 5, (7, 9)
    u = synth.uniforms(seed, shape)
    s = synth.splitmix64(seed, 63)
    assert u.dtype == np.float32 and u.shape == shape
    k = u.astype(np.float64).ravel() * 2.0**23 - 0.5
    np.testing.assert_array_equal(k, np.floor(k))       # exact in fp32
    np.testing.assert_array_equal(k.astype(np.uint64), s >> np.uint64(41))
    assert np.all(u > 0) and np.all(u < 1)
    # the extremes of the mapping stay strictly inside (0, 1) in fp32
    lo = np.float32((0 + 0.5) * 2.0**-23)
    hi = np.float32((2**23 - 1 + 0.5) * 2.0**-23)
    assert 0 < lo and hi < 1 and float(hi) == (2**23 - 0.5) / 2**23
