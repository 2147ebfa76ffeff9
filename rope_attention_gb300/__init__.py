"""GB300-native attention prologue: fused MXFP8 QKV projection with across-heads
RMSNorm + rotate-half RoPE, and KvRmsNormRopeCache.

The compute path is the C-ABI library ``librope_attention.so`` (CUDA, sm_103a);
``native`` is its thin ctypes binding.  ``synth`` generates seeded synthetic
inputs.  Importing this package does not load the library.
"""
__all__ = ["native", "synth"]
