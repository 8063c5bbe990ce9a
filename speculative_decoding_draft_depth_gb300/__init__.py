"""GB300-native batched DDTree draft-tree round.

The round runs as hand-written sm_103a CUDA kernels behind a C-ABI library
(``include/ddt.h``, built into ``_build/libddt.so``). ``ddt`` is the thin
ctypes binding over that library; ``synth`` draws seeded synthetic inputs.
"""
__all__ = ["ddt", "synth"]
