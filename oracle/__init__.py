"""Test infrastructure: the fp64 CPU oracle of the FASA decode step.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The library never calls it and it never calls
the library: the two share no code.
"""

from .fasa_oracle import *  # noqa: F401,F403
