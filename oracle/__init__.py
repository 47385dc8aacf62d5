"""Plain fp64 CPU oracle for the DeepSeek Sparse Attention (DSA) forward pass.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code, table or constant generator with the CUDA library, and imports nothing
from it.

Every function restates a definition from the source pages (cited in each
docstring) in the most direct way: no blocking, no fusion, no reordering beyond
what the definition states.  Library primitives used as single steps: numpy
matmul, exp/log, and lexsort.
"""

from .dsa_oracle import (  # noqa: F401
    decode_e4m3,
    encode_e4m3,
    quantize_e4m3_groups,
    decode_bf16,
    query_positions,
    index_scores_row,
    index_scores,
    topk_indices,
    sparse_mla_row,
    sparse_mla,
    lse_merge,
    forward_rows,
)
from .indexer_loss import (  # noqa: F401
    dense_attention_target_row,
    kl_to_softmax_row,
    indexer_scores_backward_row,
    indexer_warmup_loss,
)
