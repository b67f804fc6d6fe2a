"""CPU oracle for MLA decode (fp64, unmerged).  Test infrastructure only.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The CUDA library never depends on it.
"""
from .oracle import *  # noqa: F401,F403
