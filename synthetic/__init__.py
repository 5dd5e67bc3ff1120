"""Seeded synthetic workloads: shapes, value distributions and generators.

This package holds NO arithmetic of the method (no norm, clip, sum or
noise).  It only describes the five workloads and draws their inputs A and E
with a seeded torch generator, on whatever device the caller names.  Both the
CUDA path (through its tests and ``bench.py``) and the CPU oracle (through the
tests) receive the same bytes from here; neither imports the other.
"""

from .workloads import (  # noqa: F401
    LayerSpec,
    Workload,
    WORKLOADS,
    by_index,
    by_name,
    generate_layer,
    record_scales,
)
