"""CPU oracle for the Q1 affine g128 linear layer (test infrastructure only).

Only tests, the package's smoke entry point and the benchmark's CPU-baseline
leg may import this package; the product path never does.
"""
from . import q1_oracle  # noqa: F401
