"""Seeded synthetic inputs for the DSA lightning-indexer decode step.

This package is the only code shared by the CPU oracle (``oracle/``) and the
CUDA path (``sparse_attention_indexer_score_gb300``).  It draws raw inputs
(BF16 query and key projections, head-weight logits, LayerNorm affine
parameters, sequence and query lengths, block tables, cache slots) and holds
none of the method's arithmetic: no quantisation, no normalisation, no
scoring and no selection.
"""

from .workloads import (  # noqa: F401
    CONFIGS,
    Workload,
    bf16_bits_to_f32,
    make_workload,
)
