"""CPU fp64 oracle for forget-gated causal softmax attention.

TEST INFRASTRUCTURE ONLY: imported by the tests, the package entry file's
smoke check and the benchmark's CPU-baseline / reference arm. The library and
its Python binding never import it.
"""
from .fox_oracle import *  # noqa: F401,F403
from .fox_oracle import __all__  # noqa: F401
