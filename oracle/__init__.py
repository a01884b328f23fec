"""CPU oracle for the fine-grained-scaled FP8 GEMM family.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the package smoke check
and by the bench's CPU-baseline leg, never by the product path.  It shares no
code with the CUDA library.
"""
from .oracle import *  # noqa: F401,F403
