"""CPU oracle for two-stage GQA block-sparse attention (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package. It shares no code with the CUDA library.
"""
from .msa_oracle import *  # noqa: F401,F403
from . import msa_oracle  # noqa: F401
