"""attn_block_mask_build_noalloc: the builder for callers that cannot allocate.

Some callers cannot call cudaMalloc (a host memory manager that owns every
device byte, or a loop where an allocation and the synchronisation it may
bring are not allowed).  The no-allocation builder keeps its temporaries in a
fixed array inside the library, so such a caller only passes the metadata and
the output buffer it owns.  These tests call it through the C ABI twice in a
row, on different masks that share that array, and check that its output
equals the regular builder's (the lists bit-exact, as every block-mask test
requires) and that the forward and backward give the same results from
either mask (bit for bit, as the same lists drive the same deterministic
kernels, so well within the forward tolerances, O 2e-2 and LSE 1e-3).

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
    args = w.api_kwargs(dm)
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
    """Back-to-back no-allocation builds (sharing the scratch) of different
    kinds, among them a caller-supplied dense mask: the same lists as the
    regular builder, and the same forward and backward results from either
    mask (the backward reads the transposed lists this builder writes)."""
    cases = [
        W.random_workload(31, "shared_prefix", [700, 129, 1000], num_heads=2, head_dim=128),
        W.random_workload(32, "strip_thinking", [1500, 257], num_heads=2, head_dim=128),
        W.random_workload(33, "dense", [600, 300, 1], num_heads=2, head_dim=64),
        W.random_workload(34, "causal_document", [1200, 140], num_heads=2, head_dim=128),
    ]
    for w in cases:
        dm, ref, na = _both_masks(w)
        got, want = na.lists(), ref.lists()
        for name in api.BlockMask.NOALLOC_UNWRITTEN:
            assert name not in got, name
        for name in OUTPUT_ARRAYS:
            assert torch.equal(got[name], want[name]), name
        q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
        kw = w.api_kwargs(dm)
        o_ref, l_ref = api.attn_fwd(q, k, v, ref, w.kind, dm["cu_seqlens"], w.max_seqlen, **kw)
        o_na, l_na = api.attn_fwd(q, k, v, na, w.kind, dm["cu_seqlens"], w.max_seqlen, **kw)
        assert api.attn_get_status(na) == api.ATTN_OK
        # identical lists drive the same deterministic kernels: the outputs are
        # equal bit for bit (well inside the forward tolerances, O 2e-2 and LSE
        # 1e-3; rows that see no key have LSE = -inf on both sides)
        assert torch.equal(o_na, o_ref)
        assert torch.equal(l_na, l_ref)
        do = W.grad_output(w, seed=3).cuda()
        g_ref = api.attn_bwd(q, k, v, o_ref, l_ref, do, ref, w.kind, dm["cu_seqlens"], w.max_seqlen, **kw)
        g_na = api.attn_bwd(q, k, v, o_ref, l_ref, do, na, w.kind, dm["cu_seqlens"], w.max_seqlen, **kw)
        assert api.attn_get_status(na) == api.ATTN_OK
        for x, y in zip(g_na, g_ref):
            assert torch.equal(x, y)


@pytest.mark.gpu
def test_noalloc_serves_the_largest_problem_its_scratch_holds():
    """One 259,968-token sequence (2031 tiles) is the largest the 4 MiB scratch
    holds: it is built, with the same lists as the regular builder."""
    T = 259_968
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    ref = api.attn_block_mask_build("causal", cu, T, T)
    ws = torch.empty(api.attn_block_mask_workspace_size(1, T, T), dtype=torch.uint8, device="cuda")
    na = api.attn_block_mask_build_noalloc("causal", cu, T, T, ws)
    assert api.attn_get_status(na) == api.ATTN_OK
    got, want = na.lists(), ref.lists()
    for name in OUTPUT_ARRAYS:
        assert torch.equal(got[name], want[name]), name


@pytest.mark.parametrize("T", [259_969, 262_144, 300_000])
def test_noalloc_rejects_problems_larger_than_its_scratch(native_lib, T):
    """Past 259,968 tokens in one sequence (2032 tiles and more) the label
    matrix and summaries need more than the 4 MiB scratch; the call is refused
    on the host before any CUDA call or launch (the pointers are never used)."""
    lib = native_lib
    out = _native.AttnBlockMask()
    prm = _native.AttnMaskParams(1)
    ws_bytes = api.attn_block_mask_workspace_size(1, T, T)
    status = lib.attn_block_mask_build_noalloc(0, ctypes.byref(prm), ctypes.c_void_p(0x10000), 1, T, T,
                                               None, None, None, 128, 128, ctypes.c_void_p(0x100000),
                                               ws_bytes, ctypes.byref(out), None)
    assert status == 2  # ATTN_ERR_UNSUPPORTED
    assert out.magic == 0
