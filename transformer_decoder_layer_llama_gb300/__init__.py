"""GB300-native forward pass of one Llama-style decoder layer.

The layer runs as a handful of hand-written sm_103a CUDA kernels behind the
C-ABI library `libllamalayer.so` (declared in include/llama_layer.h).  The
Python side is a thin ctypes binding (`api`) plus seeded synthetic inputs
(`synth`).  Import `transformer_decoder_layer_llama_gb300.api` for the calls.
"""
__all__ = ["api", "synth"]
