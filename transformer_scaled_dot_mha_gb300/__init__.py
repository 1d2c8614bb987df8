"""GB300 (sm_103a) multi-head scaled dot-product attention forward.

The compute path is the CUDA library ``libattn_gb300.so`` behind the C ABI of
``include/attn_gb300.h``; ``transformer_scaled_dot_mha_gb300.attn`` is a thin
ctypes binding with the same entry-point names. ``workloads`` holds the seeded
input recipe shared by tests and the benchmark.
"""
