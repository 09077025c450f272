"""GB300-native Qwen3-style GQA decode step.

The compute lives in the C-ABI library ``libqd.so`` (CUDA for sm_103a, built
in-tree from ``csrc/``); ``api`` is its thin ctypes binding. ``synth`` makes
the seeded synthetic inputs. Importing the package loads nothing; the first
call into ``api`` loads the library and raises if it has not been built.
"""
