"""GB300-native Kimi Delta Attention (KDA): chunkwise prefill and single-token decode.

The compute runs in ``libkda.so`` (hand-written sm_103a CUDA kernels behind a C ABI declared in
``include/kda.h``).  ``binding`` marshals torch tensors to that ABI; it never computes anything
itself and raises if the library is missing.
"""
__all__ = ["binding", "inputs", "sharding"]
