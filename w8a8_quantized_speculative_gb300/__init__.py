"""GB300-native (sm_103a) W8A8 verify path of Quasar quantized self-speculative decoding.

The compute lives in ``libquasar.so`` (hand-written CUDA behind a C ABI, see
``include/quasar.h``).  ``quasar`` is the thin ctypes binding; importing it
loads the library and fails loudly when it is missing.  ``synth`` draws the
seeded synthetic inputs.
"""

__all__ = ["quasar", "synth", "build"]
