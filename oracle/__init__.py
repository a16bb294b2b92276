"""fp64 CPU oracle for the structured-mask attention forward and backward.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``, never by the library itself.  It
shares no code with the CUDA path.
"""
from .core import (EMPTY, FULL, KINDS, PARTIAL, attention, attention_backward, attention_backward_sampled,  # noqa: F401
                   block_lists, block_lists_transposed, label_totals, lpt_order,
                   masked_attention, masked_attention_backward, predicate, sequence_mask,
                   tile_labels, unmasked_pairs)
