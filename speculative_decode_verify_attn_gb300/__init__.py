"""GB300-native speculative-decoding verify step: paged and ring-window verify attention,
chunk-residency top-k, page-in and greedy acceptance, as hand-written sm_103a CUDA behind a
C ABI (libvfy.so). The Python side (vfy.py) only marshals arguments."""

__all__ = ["synth", "vfy"]
