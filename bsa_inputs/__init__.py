"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the bench.

This package holds shapes and random draws only: no step of the selected-block
attention method (pooling, scoring, selection, softmax) is computed here.
"""

from .synthetic import (  # noqa: F401
    CONFIGS,
    WORKLOAD_CONFIGS,
    Config,
    make_inputs,
    derived_sizes,
)
