"""Seeded synthetic inputs for block-sparse decode attention.

This package is the only code shared by the float64 oracle (``oracle/``) and the
CUDA path (``long_context_serving_gb300/``). It holds none of the method's
arithmetic: it draws random numbers, plants the attention-sink and needle
structure, rounds to bf16 and assigns logical KV pages to physical pages.
"""

from .synthetic import (  # noqa: F401
    CONFIG_IDS,
    STREAMING,
    RETRIEVAL,
    DUAL,
    Workload,
    bf16_bits_to_f32,
    make_workload,
    to_bf16_bits,
)
