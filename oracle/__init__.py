"""Float64 CPU oracle (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  It is independent of the CUDA library:
neither imports the other.  See ``oracle/attention.py`` (attention, merge,
gates, indexer) and ``oracle/mla.py`` (the MLA value up-projection and the
K/V materialisation from latents) for the passages each function follows.
"""

from . import mla  # noqa: F401

from .attention import (  # noqa: F401
    NEG_INF,
    Layout,
    block_means,
    chunk_summary,
    dense_attention,
    dense_attention_backward,
    dsa_indexer_topk,
    finalise,
    logical_positions,
    lse_merge,
    make_layout,
    merge_summaries,
    moba_attention,
    moba_block_gate,
    neutral_summary,
    sequence_index,
    sparse_attention,
    sparse_key_list,
    summarised_attention,
)
