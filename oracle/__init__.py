"""CPU oracle for the same-device collective set (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this package.  It shares no code with the CUDA library.  Parity status of every
function is listed in ``oracle.py``'s module docstring.
"""
from .oracle import *  # noqa: F401,F403
