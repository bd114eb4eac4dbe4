"""fp64 CPU oracle for LRKV factored-cache attention.

TEST INFRASTRUCTURE: imported only by the tests, the package smoke check and
the bench's CPU-baseline leg.  Never imported by the library or its binding.
"""
from .lrkv_oracle import *  # noqa: F401,F403
