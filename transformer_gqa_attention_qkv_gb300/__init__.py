"""GB300 (sm_103a) forward pass of a grouped-query attention layer with an
explicit head_dim: fused QKV projection with QK-norm and RoPE, causal GQA
flash attention, o_proj with the residual add, and a split-KV decode step.

The compute lives in a C-ABI CUDA library (``libgqa_attn.so``); the binding
in :mod:`.binding` only marshals arguments.  Importing this package does not
load the library; the first call does, and fails loudly if it is missing.
"""
