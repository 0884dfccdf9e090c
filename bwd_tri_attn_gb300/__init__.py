"""GB300-native triangle attention forward and backward (sm_103a CUDA kernels).

The compute lives in ``libtriattn.so`` (built from ``csrc/``) behind a C ABI
declared in ``include/tri_attn.h``; ``binding`` marshals PyTorch device tensors
into that ABI. Nothing here computes on the CPU.
"""
