"""CPU oracle for the MXFP6 MLP hot path.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its
``cpu_baseline`` leg and ``--impl reference``) may import it.
"""

from .mx_oracle import *  # noqa: F401,F403
