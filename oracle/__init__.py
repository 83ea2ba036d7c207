"""CPU oracle for QSA attention over a quantised KV cache.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
CPU-baseline / reference arm may import this package.  The CUDA library never
calls it, and it shares no code with the CUDA library: the only code both sides
use is the seeded input generator in ``workloads``, which holds none of the
method's arithmetic.
"""
from .qsa_oracle import *  # noqa: F401,F403
