"""GB300-native (sm_103a) fused causal MHA/GQA attention, forward and backward.

The compute lives in the CUDA library built from ``csrc/`` (C ABI in
``include/attn_gb300.h``); ``binding`` is its Python binding and
``workloads`` the seeded synthetic inputs.
"""
