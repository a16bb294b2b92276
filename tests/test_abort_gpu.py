"""The device-side abort path, exercised on the GPU without a fault.

Every pipeline wait in the tcgen05 kernels is bounded: past the bound the
waiting thread sets the CTA's abort flag and ATTN_ERR_DEVICE_TIMEOUT (with the
wait's site) in the block mask's error word, every other role leaves its loop
at its next wait, copies and products already in flight are drained (with a
bound of their own), tensor memory is freed and the kernel returns.

A copy of the library built with a 100 ns bound (instead of 1 s) runs the
forward and the backward on an ordinary workload: ordinary waits run out.
The launches must return, the status must read ATTN_ERR_DEVICE_TIMEOUT, the
CUDA context must stay usable, and the regular library, after a rebuild of the
mask (which clears the error word), must give a correct forward and backward.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_masked_mask_gb300 import _native, api
from block_sparse_masked_mask_gb300 import build as B
from block_sparse_masked_mask_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def short_wait_library():
    return B.build_variant("waitshort", {"ATTN_WAIT_TIMEOUT_NS": "100ull"})


def _setup():
    w = W.random_workload(41, "causal_document", [4096, 3000, 900], num_heads=8, head_dim=128)
    dm = w.device_meta()
    return w, dm, w.api_kwargs(dm)


def _mask(w, dm, kw):
    return api.attn_block_mask_build(w.kind, dm["cu_seqlens"], w.total_tokens, w.max_seqlen, **kw)


def test_short_waits_run_out_and_the_launch_returns(short_wait_library):
    w, dm, kw = _setup()
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    do = W.grad_output(w, seed=41).cuda()
    # O and LSE for the backward from the regular library
    bm = _mask(w, dm, kw)
    o, lse = api.attn_fwd(q, k, v, bm, w.kind, dm["cu_seqlens"], w.max_seqlen, **kw)
    assert api.attn_get_status(bm) == api.ATTN_OK

    with _native.use_library(short_wait_library):
        bm_f = _mask(w, dm, kw)
        api.attn_fwd(q, k, v, bm_f, w.kind, dm["cu_seqlens"], w.max_seqlen, **kw)
        torch.cuda.synchronize()  # the forward's kernels have returned
        assert api.attn_get_status(bm_f) == api.ATTN_ERR_DEVICE_TIMEOUT

        bm_b = _mask(w, dm, kw)
        assert api.attn_get_status(bm_b) == api.ATTN_OK  # a rebuild clears the error word
        api.attn_bwd(q, k, v, o, lse, do, bm_b, w.kind, dm["cu_seqlens"], w.max_seqlen, **kw)
        torch.cuda.synchronize()
        assert api.attn_get_status(bm_b) == api.ATTN_ERR_DEVICE_TIMEOUT

        # a mask whose error word holds a timeout makes later kernels on it
        # return at once (they see the abort at their start)
        api.attn_fwd(q, k, v, bm_f, w.kind, dm["cu_seqlens"], w.max_seqlen, **kw)
        torch.cuda.synchronize()
        assert api.attn_get_status(bm_f) == api.ATTN_ERR_DEVICE_TIMEOUT

    # the context is usable and the regular library is correct again
    x = torch.arange(1 << 20, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == float((1 << 20) * ((1 << 20) - 1) / 2)
    bm = _mask(w, dm, kw)
    o2, lse2 = api.attn_fwd(q, k, v, bm, w.kind, dm["cu_seqlens"], w.max_seqlen, **kw)
    assert api.attn_get_status(bm) == api.ATTN_OK
    O, L = oracle.attention(w.q, w.k, w.v, w.kind, w.cu_seqlens, w.meta())
    assert np.abs(o2.float().cpu().numpy() - O).max() <= 2e-2
    assert np.abs(lse2.cpu().numpy() - L).max() <= 1e-3
    dq, dk, dv = api.attn_bwd(q, k, v, o2, lse2, do, bm, w.kind, dm["cu_seqlens"], w.max_seqlen, **kw)
    assert api.attn_get_status(bm) == api.ATTN_OK
    rows = np.arange(0, w.total_tokens, 97)
    ref = oracle.attention_backward_sampled(w.q, w.k, w.v, do.cpu(), w.kind, w.cu_seqlens, w.meta(),
                                            heads=[0, 7], q_rows=rows, k_rows=rows)
    for g, r in zip((dq, dk, dv), ref):
        got = g.float().cpu().numpy()[rows][:, [0, 7]]
        want = r[rows][:, [0, 7]]
        assert np.abs(got - want).max() <= 2.0 ** -6 * np.abs(want).max()
