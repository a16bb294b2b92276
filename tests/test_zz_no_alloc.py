"""attn_block_mask_build_noalloc: the builder for callers that cannot allocate.

Some callers cannot call cudaMalloc (a host memory manager that owns every
device byte, or a loop where an allocation and the synchronisation it may
bring are not allowed).  The no-allocation builder keeps its temporaries in a
fixed array inside the library, so such a caller only passes the metadata and
the output buffer it owns.  These tests call it through the C ABI twice in a
row, on different masks that share that array, and check that its output
equals the regular builder's (the lists bit-exact, as every block-mask test
requires) and that the forward gives the same O and LSE from either mask
(within the forward tolerances, O 2e-2 and LSE 1e-3).

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test; it also passes when run alone.
"""
import ctypes

import numpy as np
import pytest
import torch

from block_sparse_masked_mask_gb300 import _native, api
from block_sparse_masked_mask_gb300 import workloads as W

OUTPUT_ARRAYS = ["header", "qt_seq", "qt_idx", "kcount", "koff", "kidx", "klabel", "order",
                 "pair_q0", "pair_order", "qcount", "qoff", "qidx", "qlabel", "korder"]


def _both_masks(w):
    dm = w.device_meta()
    args = dict(seg_id=dm["seg_id"], role=dm["role"], turn=dm["turn"], role_think=w.role_think)
    ref = api.attn_block_mask_build(w.kind, dm["cu_seqlens"], w.total_tokens, w.max_seqlen, **args)
    ws = torch.empty(api.attn_block_mask_workspace_size(w.batch, w.total_tokens, w.max_seqlen),
                     dtype=torch.uint8, device="cuda")
    na = api.attn_block_mask_build_noalloc(w.kind, dm["cu_seqlens"], w.total_tokens, w.max_seqlen,
                                           ws, **args)
    assert api.attn_get_status(ref) == api.ATTN_OK
    assert api.attn_get_status(na) == api.ATTN_OK
    return dm, ref, na


@pytest.mark.gpu
def test_noalloc_build_matches_regular_build_twice_in_a_row():
    cases = [
        W.random_workload(31, "shared_prefix", [700, 129, 1000], num_heads=2, head_dim=128),
        W.random_workload(32, "strip_thinking", [1500, 257], num_heads=2, head_dim=128),
    ]
    for w in cases:
        dm, ref, na = _both_masks(w)
        got, want = na.lists(), ref.lists()
        for name in OUTPUT_ARRAYS:
            assert torch.equal(got[name], want[name]), name
        q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
        fwd = dict(seg_id=dm["seg_id"], role=dm["role"], turn=dm["turn"], role_think=w.role_think)
        o_ref, l_ref = api.attn_fwd(q, k, v, ref, w.kind, dm["cu_seqlens"], w.max_seqlen, **fwd)
        o_na, l_na = api.attn_fwd(q, k, v, na, w.kind, dm["cu_seqlens"], w.max_seqlen, **fwd)
        assert api.attn_get_status(na) == api.ATTN_OK
        assert (o_na.float() - o_ref.float()).abs().max().item() <= 2e-2
        assert (l_na - l_ref).abs().max().item() <= 1e-3


def test_noalloc_rejects_problems_larger_than_its_scratch(native_lib):
    """The label matrix of one 300k-token sequence needs more than the 4 MiB
    scratch; the call is refused before anything is launched."""
    lib = native_lib
    out = _native.AttnBlockMask()
    prm = _native.AttnMaskParams(1)
    T = 300_000
    ws_bytes = api.attn_block_mask_workspace_size(1, T, T)
    status = lib.attn_block_mask_build_noalloc(0, ctypes.byref(prm), ctypes.c_void_p(0x10000), 1, T, T,
                                               None, None, None, 128, 128, ctypes.c_void_p(0x100000),
                                               ws_bytes, ctypes.byref(out), None)
    assert status == 2  # ATTN_ERR_UNSUPPORTED
    assert out.magic == 0
