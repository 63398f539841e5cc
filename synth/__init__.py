"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This package only draws random numbers and rounds them to BF16; it holds none
of the MXFP6 method's arithmetic, so both sides may use it.
"""

from .inputs import *  # noqa: F401,F403
