"""fp64 CPU oracle for the structured-mask attention forward.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``, never by the library itself.  It
shares no code with the CUDA path.
"""
from .core import (EMPTY, FULL, KINDS, PARTIAL, attention, block_lists,  # noqa: F401
                        label_totals, lpt_order, masked_attention, predicate,
                        sequence_mask, tile_labels, unmasked_pairs)
