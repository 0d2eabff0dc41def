"""CPU oracle for the tensor-parallel hot path (test infrastructure only).

This package is a plain, slow, fp64 restatement of what the tensor-parallel
layers compute, written from the web pages on Megatron-style tensor
parallelism.  Only the test suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The CUDA library never imports, links or calls anything here, and nothing
here imports the CUDA library: the two sides share no code.

Every function is pinned by checks independent of it (tests/test_oracle_pins.py:
the pages' worked examples, closed forms, brute force on small integers and
library routines); a function without such a pin would say "parity unpinned"
in its docstring, and none does.
"""

from .tp_oracle import *  # noqa: F401,F403
