"""GB300-native batched lossless draft verification with test-time self-selection.

The compute path is ``libsdv.so`` (hand-written CUDA for sm_103a behind a C
ABI declared in ``include/sdv.h``); ``binding`` marshals torch tensors to it.
``synth`` makes seeded synthetic inputs.
"""
__all__ = ["binding", "synth"]
