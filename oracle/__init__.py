"""CPU oracle for the INT8 ConvRot W8A8 linear (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path (the CUDA library and
its Python binding) never imports it and shares no code with it.
"""
from .convrot_oracle import *  # noqa: F401,F403
