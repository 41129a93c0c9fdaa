"""fp64 CPU oracle -- test infrastructure, never part of the product path.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU baseline
leg import this package.
"""
from .kvq_oracle import *  # noqa: F401,F403
