"""GB300-native FlashPrefill V2 block-sparse prefill attention with mean correction.

The compute path lives in a C-ABI shared library (``libfp.so``, declared in
``include/fp.h``) built from ``csrc/`` for sm_103a. ``binding`` marshals torch
tensors to it; ``synth`` draws seeded synthetic workloads.
"""
__all__ = ["binding", "synth"]
