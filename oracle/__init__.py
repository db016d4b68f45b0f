"""CPU oracle for the diagonal linear-recurrence scan -- test infrastructure only.

Only the tests, the smoke check and the benchmark's CPU-baseline leg import
this package; the product path (the CUDA library and its binding) never does.
"""
from .oracle import Oracle, build, default, load  # noqa: F401
