"""Seeded synthetic inputs for the tests and the benchmark.

This package holds input generators only -- no attention, pool or page-table
arithmetic -- so that the oracle and the CUDA library can both be fed from it
without sharing any of the method's code.
"""
from .gate_lcg import GATE_SEED, LcgStream, lcg_next, gate_inputs  # noqa: F401
from . import workloads  # noqa: F401
