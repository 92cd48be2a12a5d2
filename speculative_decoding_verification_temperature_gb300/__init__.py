"""GB300-native verify step of speculative decoding.

The compute path is ``libsdverify.so`` (hand-written CUDA for sm_103a behind
a C ABI declared in ``include/sd_verify.h``); :mod:`.api` is a thin binding
over it that takes torch tensors.  :mod:`.synth` makes seeded synthetic
inputs.
"""
__all__ = ["api", "synth"]


def __getattr__(name):
    if name == "api":
        from . import api
        return api
    raise AttributeError(name)
