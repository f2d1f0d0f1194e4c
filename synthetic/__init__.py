"""Seeded synthetic workloads shared by the tests, the bench and the oracle.

This package holds input generators and workload recipes only -- shapes,
seeds, random values, context lengths, block-pool orderings and the order in
which tokens are appended -- and none of the method's arithmetic (no
attention, no quantisation, no allocation).
"""

from .workloads import *  # noqa: F401,F403
