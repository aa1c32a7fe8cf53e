"""GB300-native DSA lightning-indexer decode step.

The compute lives in ``libdsa.so`` (hand-written CUDA for sm_103a, C ABI in
``include/dsa.h``); ``dsa`` is its Python binding.  PyTorch only provides
device memory and streams.
"""

from . import dsa  # noqa: F401
from .dsa import (  # noqa: F401
    FORMATS,
    decode_layout,
    insert_key,
    quantize_queries_rg,
    quantize_query,
    score_paged,
    topk,
    topk_workspace_size,
    workspace_size,
)
