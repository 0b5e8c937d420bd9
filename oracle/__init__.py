"""CPU oracle of the hybrid long-context attention path (test infrastructure only).

Imported only by the tests, the smoke check and the CPU-baseline leg of the
benchmark.  The CUDA library neither imports nor links anything here.
"""
from .hybrid_attention import *  # noqa: F401,F403
