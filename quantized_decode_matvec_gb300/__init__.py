"""GB300-native q4_K x q8_0 decode matvec.

The compute lives in the C-ABI library ``libmq.so`` (hand-written CUDA for
sm_103a, declared in ``include/mq.h``); ``quantized_decode_matvec_gb300.mq``
is the thin ctypes binding with the same call names.  ``synth`` holds the
seeded synthetic-input generator.  Importing the package does not load the
library; importing ``mq`` does, and fails loudly if it is missing.
"""
__all__ = ["synth"]
