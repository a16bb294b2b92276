"""GB300 (sm_103a) structured-mask attention, forward and backward.

The computation lives in the CUDA library ``libattnmask.so`` (C ABI declared
in ``include/attn_block_mask.h``); this package is its thin Python binding
plus the seeded synthetic workloads used by the tests and the benchmark.
"""
from .api import (AttnError, BlockMask, MASK_KINDS, TILE_EMPTY, TILE_FULL,  # noqa: F401
                  TILE_PARTIAL, attn_block_mask_build, attn_block_mask_build_noalloc,
                  attn_block_mask_workspace_size,
                  attn_bwd, attn_bwd_workspace_size, attn_fwd, attn_get_status, attn_last_error_message, attn_status_string,
                  attn_version)
