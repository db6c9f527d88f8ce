"""fp64 CPU oracle for FLAMIA causal microscaled-FP8 attention.

Test infrastructure only: ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` import it.  The CUDA library never does, and the
two share no code.
"""
from .flamia_oracle import *  # noqa: F401,F403
