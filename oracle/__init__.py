"""CPU oracle for the Qwen3 forward hot path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  It shares no code with the CUDA path.
"""
from .qwen3 import *  # noqa: F401,F403
