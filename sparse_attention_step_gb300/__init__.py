"""GB300-native two-stage GQA block-sparse attention (C-ABI library + binding).

``msa`` is the ctypes binding of ``include/msa.h``; ``build`` compiles the CUDA
sources into ``_lib/libmsa.so``.
"""
from . import msa  # noqa: F401

__all__ = ["msa"]
