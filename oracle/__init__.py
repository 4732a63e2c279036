"""CPU oracle of the tensor-parallel transformer block -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it, and it
shares no code with the library: it is a plain, slow, float64 restatement of
what the block computes, written so that a reader can check it against the
pages line by line.
"""
from .tp_oracle import *  # noqa: F401,F403
