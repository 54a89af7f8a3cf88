"""GB300-native greedy DDTree tree-verify step.

The compute path is the C-ABI library ``libdfv.so`` (hand-written CUDA for
sm_103a, declared in ``include/dfv.h``); ``api`` is its thin Python binding.
``workload`` holds the seeded synthetic input generators.

Importing the package does not load the library; the first call into
``api`` does, and raises if the library is missing.
"""

__all__ = ["api", "workload"]
