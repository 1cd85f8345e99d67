"""GB300 (sm_103a) local MoE forward: route -> dispatch -> SwiGLU experts -> combine.

The compute lives in ``libmoe.so`` (hand-written CUDA kernels behind a C ABI declared in
``include/moe.h``); ``binding`` marshals torch tensors into that ABI and nothing else.
"""
