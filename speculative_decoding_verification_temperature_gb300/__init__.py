"""GB300-native verify step of speculative decoding.

The compute path is ``libsdverify.so`` (hand-written CUDA for sm_103a behind
the C ABI declared in ``include/sd_verify.h``); the ``api`` submodule is a
thin binding over it that takes torch tensors, and ``synth`` makes seeded
synthetic inputs.
"""
