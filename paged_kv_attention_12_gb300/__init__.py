"""Paged-KV attention for GB300 (sm_103a).

Attention read through a block-paged KV cache: decode, split-K decode with a
log-sum-exp combine, and causal chunked / mixed-batch prefill.  The compute
runs in hand-written CUDA kernels behind a C ABI (``include/paged_attn.h``);
this package holds the build step, the ctypes binding and the seeded
workload generator.  Importing it does not load the CUDA library; the first
call into :mod:`.binding` does, and fails loudly if it is missing.
"""
__all__ = ["binding", "workload"]
