"""Workload shapes and seeded synthetic input generators.

This package holds no arithmetic of the method (no scores, no selection, no
attention).  It only describes the five workloads and draws their inputs from
seeded torch generators, so that the CUDA path and the CPU oracle can be fed
the very same bytes.
"""
from .configs import CONFIGS, Config, get_config  # noqa: F401
from .gen import (  # noqa: F401
    make_indexer_inputs,
    make_attn_inputs,
    seed_for,
    TORCH_DTYPE,
)
