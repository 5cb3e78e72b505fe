"""fp64 CPU oracle for LowRAM compressed decode attention -- TEST INFRASTRUCTURE.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may import this package.
It shares no code with the CUDA library (``decode_attention_19_b300``) and never imports it.  The
arithmetic lives in ``lowram_oracle.c`` (plain C, fp64, OpenMP over (sequence, kv-head)); this module
only builds it with gcc, converts arrays to fp64 exactly, and composes the oracle's own steps.
"""
from .oracle import *  # noqa: F401,F403
from .oracle import build, lib  # noqa: F401
