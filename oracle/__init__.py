"""Plain, slow CPU oracle for exact ring attention.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports, calls or links
anything in this package: only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it. It shares no code, table or helper
with the CUDA library; the two meet only through the seeded input generators,
which hold none of the method's arithmetic.

Everything here is float64 NumPy, written to be read against the pages:

* ``attention_naive``   - full softmax attention from its definition
  (the exact result ring attention is said to equal, glossary
  "sequence parallelism transformers", §Ring Attention, "Computation").
* ``ring_schedule``     - which key/value chunk each virtual rank holds at
  each ring step (same glossary, §Ring Attention, "Ring Communication";
  §Sequence Parallelism Fundamentals, "Sequence Dimension Splitting").
* ``ring_attention``    - the ring restated step by step: per-step partial
  attention over one chunk, folded with the log-sum-exp merge.
* ``lse_merge`` / ``lse_merge_n`` - the exact merge of partial softmax results
  (same glossary, §Implementation Considerations, "Numerical Stability").
* ``attention_backward`` - dq, dk, dv from the chain rule through the
  forward definition (same glossary, §Implementation Considerations: the
  backward pass runs over the same ring); ``ring_attention_backward``
  restates it per (rank, step); ``backward_rows`` evaluates sampled rows.
* ``attention_varlen`` / ``attention_backward_varlen`` - packed batches of
  sequences of different lengths, each its own problem.
* ``ulysses_attention`` - the Ulysses steps (all-to-all to heads, full
  attention per head group, all-to-all back) on sequence-sharded tensors.
* ``tile_visits``       - expands the chunk-level schedule into the sequence of
  fixed-size key tiles a tiled kernel must visit, classifying every tile by
  brute force over its (query, key) pairs.

Pins: every function above is checked in ``tests/test_oracle.py`` against
brute force, closed forms, invariants and hand-derived fixtures under
``tests/golden/``; none is "parity unpinned".
"""

from .attention import attention_naive, attention_rows, partial_attention
from .merge import lse_merge, lse_merge_n
from .schedule import (
    SKIP, FULL, PARTIAL,
    ORDER_CONTIGUOUS, ORDER_ZIGZAG,
    rank_segments, ring_schedule, schedule_table, tile_visits,
)
from .ring import ring_attention
from .backward import attention_backward, ring_attention_backward, backward_rows
from .varlen import attention_varlen, attention_backward_varlen
from .ulysses import (ulysses_attention, to_sequence_shards, from_sequence_shards,
                      all_to_all_seq_to_head, all_to_all_head_to_seq)

__all__ = [
    "attention_naive", "attention_rows", "partial_attention",
    "lse_merge", "lse_merge_n",
    "SKIP", "FULL", "PARTIAL", "ORDER_CONTIGUOUS", "ORDER_ZIGZAG",
    "rank_segments", "ring_schedule", "schedule_table", "tile_visits",
    "ring_attention",
    "attention_backward", "ring_attention_backward", "backward_rows",
    "attention_varlen", "attention_backward_varlen",
    "ulysses_attention", "to_sequence_shards", "from_sequence_shards",
    "all_to_all_seq_to_head", "all_to_all_head_to_seq",
]
