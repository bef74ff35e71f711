"""Seeded synthetic inputs shared by the tests and the benchmark.

Holds geometry and bound-matrix construction only; no smoothing arithmetic.
"""
from .molecules import (CONFIGS, Q, make_config, random_bounds, to_f32,  # noqa: F401
                        chain_bounds, globule_bounds, sentinel_q, blank_bounds)
