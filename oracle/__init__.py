"""CPU oracle for the NVFP4 / MXFP8 linear-layer arithmetic.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the product library never
does. It shares no code with the CUDA library. See ``fp4q_oracle.c`` for the
arithmetic and the page citations, and ``oracle.py`` for the numpy-level API.
"""
from .oracle import *  # noqa: F401,F403
