"""CPU oracle for the BF16 weight codec and its GEMV.

TEST INFRASTRUCTURE ONLY: imported by tests/, by the smoke check and by the
benchmark's CPU-baseline leg, never by the library.  See wcomp_oracle.py.
"""
from .wcomp_oracle import *  # noqa: F401,F403
