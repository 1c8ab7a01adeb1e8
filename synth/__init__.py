"""Seeded synthetic inputs for the LOCKS decode step.

This package only draws random numbers and lays them out; it holds none of the
method's arithmetic (no SVD, no log-sum-exp, no selection, no attention).  Both
the fp64 oracle (``oracle/``) and the CUDA path (``sparse_kv_page_rank_gb300``)
are fed from it, so that the two see bit-identical bf16 inputs.
"""

from .generator import (  # noqa: F401
    CONFIGS,
    PAGE_SIZE,
    HEAD_DIM,
    LocksCase,
    bf16_bits,
    bf16_to_f32,
    make_case,
    make_config_case,
)
