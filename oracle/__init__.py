"""FP64 CPU oracle for context-parallel causal GQA attention over packed THD.

TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path imports,
calls or links this package: only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It
shares no code, constants or helpers with the CUDA path.

The subject is the TransformerEngine pull request "Optimize context parallel
attention layouts and gradient accumulation" (BF16 causal GQA attention over
packed THD sequences, context parallelism with AllGather / P2P / A2A
exchange, first dK/dV contribution reused as the accumulator, A2A
pack/unpack layout copies).  The pages name the operation but print no
formulas, so the plain textbook definition of causal scaled-dot-product
attention is taken as what is computed; every place where that reading
fills a gap is listed in the module that makes it.

Modules
-------
attention  plain per-(sequence, head) definition: forward (O, LSE) and
           backward (dQ, dK, dV), GQA head map, THD padding.
cp         the context-parallel decomposition: 2*CP load-balanced chunks,
           ring-step partials with LSE stats, K-way LSE merge, and the
           canonical fixed-order gradient accumulation with the first
           contribution used as the accumulator.
layout     the A2A head-split pack / unpack index maps and the O.dO row dot.

Parity pins: every function here is pinned in ``tests/test_oracle*.py``
against closed forms, brute-force scalar loops, finite differences, a library
routine (torch CPU fp64 SDPA), a hand-worked golden example and structural
identities.  No function is "parity unpinned".
"""

from .attention import (attention_forward, attention_backward, head_forward,
                        head_backward, kv_head_of)
from .cp import (chunk_table, chunk_owner, ring_source, rank_chunks,
                 visible_kv_chunks, cp_forward_partials, lse_merge,
                 cp_attention_forward, cp_attention_backward, dkdv_contribution_order,
                 dq_contribution_order, partial_steps_for_chunk)
from .layout import (rank_major_token_index, thd_pack, thd_unpack, bwd_dot)

__all__ = [
    "attention_forward", "attention_backward", "head_forward", "head_backward",
    "kv_head_of", "chunk_table", "chunk_owner", "ring_source", "rank_chunks",
    "visible_kv_chunks", "cp_forward_partials", "lse_merge",
    "cp_attention_forward", "cp_attention_backward", "dkdv_contribution_order",
    "dq_contribution_order", "partial_steps_for_chunk",
    "rank_major_token_index", "thd_pack", "thd_unpack", "bwd_dot",
]
