"""CPU oracle (test infrastructure only).

A plain float64 NumPy restatement of the Qwen3-style decode step, written from
the pages it cites, used to check the CUDA library. It is imported only by the
tests, by ``__graft_entry__.smoke()`` and by the CPU-baseline / reference arm
of ``bench.py``; the library never imports it, and it imports nothing from the
library.
"""
from .qwen3_decode import *  # noqa: F401,F403
