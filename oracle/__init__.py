"""fp64 CPU oracle for the local MoE forward — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import this package.  The product path (the CUDA library and its Python
binding) never imports it and has no CPU fallback.
"""
from .moe_oracle import *  # noqa: F401,F403
