"""Test infrastructure: the plain CPU oracle for the tree-verify step.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this package.  The product path (the CUDA library and its binding) never does.
"""
from .eagle_oracle import *  # noqa: F401,F403
