"""Seeded synthetic inputs for ring attention.

This package holds the workload definitions (shapes, document lengths,
per-document ring sizes) and the seeded random draws that feed both the
CUDA path and the CPU oracle.  It contains none of the attention
arithmetic: only random numbers, integer bookkeeping of document lengths,
and the bf16 rounding of the drawn values.
"""

from .synth import (  # noqa: F401
    CONFIGS,
    Workload,
    custom,
    draw_qkvdo,
    varlen_doc_lengths,
    workload,
)
