"""CPU oracle of the DSA lightning-indexer decode step.

TEST INFRASTRUCTURE ONLY.  This package is imported by ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``; nothing
on the product path (the ``sparse_attention_indexer_score_gb300`` package and
its CUDA library) imports, links or runs it, and it shares no code with that
path.  It is a plain, slow restatement of what the indexer pages define: the
number formats (``codecs``) and the five steps of the decode step
(``indexer``: query quantisation, key LayerNorm + quantise + insert, row
bounds, paged logits, top-k).

Parity unpinned: the pages' claim that the MXFP4 scale is bit-exact with a
particular compiled ``log2`` sequence (page *cutedsl.dsa.index*,
``mxfp4_scale``) is not reproduced; the exact mathematical definition printed
there is used instead (a reading of ours).
"""

from . import codecs, indexer  # noqa: F401
