"""Synthetic workloads shared by the tests, the bench and the oracle's callers.

`configs` holds the tensor lists and settings of the five workloads; `gen` holds
the counter-based input generator.  Neither computes any part of the
synchronisation step.
"""
from . import configs, gen  # noqa: F401
