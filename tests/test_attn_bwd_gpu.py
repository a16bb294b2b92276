"""GPU attention backward (dQ, dK, dV) vs the fp64 oracle on the same seeded inputs.

Tolerance, derived from the arithmetic (no figure is fixed for the backward):
P and dS are rounded to bf16 (unit roundoff u = 2^-8) before the tensor-core
products, which accumulate in fp32, and each output is rounded to bf16 once
more.  Each output element is a sum of many such terms with independent
rounding errors, so its error is a few u relative to the size of the terms,
not of the (often cancelling) sum.  The bar for every output tensor X:
  * max |X - X_ref| <= 2^-6 * max |X_ref|      (two bf16 ULPs of the largest)
  * sum |X - X_ref| <= 2^-8 * sum |X_ref|      (mean error within one u)
Where X_ref is exactly zero (dQ of a one-token sequence), the bar is an
absolute 1e-5: the fp32 rounding left over when dP - D cancels.
The forward that produces O and LSE for the backward is the library's own, as
a caller would run it; the oracle computes everything from Q, K, V, dO alone.
"""
import functools

import numpy as np
import pytest
import torch

import oracle
from block_sparse_masked_mask_gb300 import api
from block_sparse_masked_mask_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_REL = 2.0 ** -6
MEAN_REL = 2.0 ** -8


def build_mask(w, dm):
    return api.attn_block_mask_build(w.kind, dm["cu_seqlens"], w.total_tokens, w.max_seqlen,
                                     **w.api_kwargs(dm))


def run_bwd(w, do, q=None, k=None, v=None, bm=None, scale=0.0):
    dm = w.device_meta()
    bm = bm or build_mask(w, dm)
    q = (w.q if q is None else q).cuda()
    k = (w.k if k is None else k).cuda()
    v = (w.v if v is None else v).cuda()
    kw = dict(w.api_kwargs(dm), scale=scale)
    o, lse = api.attn_fwd(q, k, v, bm, w.kind, dm["cu_seqlens"], w.max_seqlen, **kw)
    dq, dk, dv = api.attn_bwd(q, k, v, o, lse, do.cuda(), bm, w.kind, dm["cu_seqlens"],
                              w.max_seqlen, **kw)
    assert api.attn_get_status(bm) == api.ATTN_OK
    return dq.cpu(), dk.cpu(), dv.cpu()


def check(name, got, ref, rows=None, heads=None):
    got = got.float().numpy()
    if rows is not None:
        got, ref = got[rows], ref[rows]
    if heads is not None:
        got, ref = got[:, heads], ref[:, heads]
    assert np.isfinite(ref).all()
    err = np.abs(got - ref)
    assert np.isfinite(err).all(), f"{name}: non-finite output"
    scale = np.abs(ref).max()
    if scale == 0:
        # an exact zero, e.g. dQ of a one-token sequence, where dP - D cancels:
        # the kernel forms dP on the tensor cores and D in its own fp32 sum, so
        # what is left is their fp32 rounding difference, times scale and K
        assert err.max() <= 1e-5, f"{name}: expected zeros, max abs {err.max()}"
        return 0.0, 0.0
    mx = err.max() / scale
    mean = err.sum() / np.abs(ref).sum()
    assert mx <= MAX_REL, f"{name}: max abs err {err.max()} = {mx:.3g} of max|ref|"
    assert mean <= MEAN_REL, f"{name}: mean rel err {mean:.3g}"
    return mx, mean


def compare_all(w, do, grads):
    ref = oracle.attention_backward(w.q, w.k, w.v, do, w.kind, w.cu_seqlens, w.meta())
    for name, g, r in zip(("dQ", "dK", "dV"), grads, ref):
        check(f"{w.name} {name}", g, r)


SMALL_LENGTHS = [300, 1, 129, 517, 0, 128]


@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("kind", oracle.KINDS)
def test_small_all_elements(kind, D):
    w = W.random_workload(5 + D, kind, SMALL_LENGTHS, num_heads=2, head_dim=D)
    do = W.grad_output(w, seed=D)
    compare_all(w, do, run_bwd(w, do))


@pytest.mark.parametrize("kind", ["causal_document", "shared_prefix", "strip_thinking",
                                  "strip_thinking_dup"])
def test_small_repeating_ids_all_elements(kind):
    """Ids and turns from a small alphabet: keys of one warp often hold different
    codes, so the dK/dV side takes the per-key predicate path."""
    w = W.random_workload(71, kind, [700, 255, 1000], num_heads=2, head_dim=128, id_alphabet=4)
    do = W.grad_output(w, seed=7)
    compare_all(w, do, run_bwd(w, do))


@pytest.mark.parametrize("lens", [[1], [2], [127], [128], [129], [255, 257], [1000]])
def test_ragged_shapes_causal(lens):
    w = W.random_workload(sum(lens) + 1, "causal", lens, num_heads=3, head_dim=128)
    do = W.grad_output(w, seed=len(lens))
    compare_all(w, do, run_bwd(w, do))


def test_scale_argument_is_used():
    w = W.random_workload(4, "causal", [300], num_heads=1, head_dim=64)
    do = W.grad_output(w)
    got = run_bwd(w, do, scale=0.37)
    ref = oracle.attention_backward(w.q, w.k, w.v, do, w.kind, w.cu_seqlens, scale=0.37)
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        check(name, g, r)


@functools.lru_cache(maxsize=None)
def full_workload(c, form="mask"):
    return W.make_workload(c, tensors=True, document_form=form)


def sample_rows(w, n=48, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(rng.integers(0, w.total_tokens, n).tolist())
    for b in range(w.batch):
        s0, s1 = int(w.cu_seqlens[b]), int(w.cu_seqlens[b + 1])
        if s1 > s0:
            rows.update([s0, s1 - 1, min(s1 - 1, s0 + 127), min(s1 - 1, s0 + 128)])
    return sorted(rows)


@pytest.mark.parametrize("c,form,heads", [(2, "mask", (0, 15)),
                                          (3, "mask", (0, 31)), (4, "mask", (0, 31)),
                                          (5, "cu_seqlens", (0, 31)), (5, "mask", (31,)),
                                          (6, "mask", (0, 31)), (7, "mask", (0, 15)),
                                          (8, "mask", (31,))])
def test_full_size_workloads_sampled(c, form, heads):
    """The bf16 workloads at full size, on sampled query rows (dQ) and key rows
    (dK, dV) that the oracle computes one by one."""
    w = full_workload(c, form)
    do = W.grad_output(w, seed=100 + c)
    got = run_bwd(w, do)
    for g in got:
        assert torch.isfinite(g.float()).all()
    rows = sample_rows(w, seed=c)
    ref = oracle.attention_backward_sampled(w.q, w.k, w.v, do, w.kind, w.cu_seqlens, w.meta(),
                                            heads=heads, q_rows=rows, k_rows=rows)
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        check(f"{w.name} {name}", g, r, rows=rows, heads=list(heads))


def test_longest_single_sequence_sampled():
    """The largest backward case: one 65536-token causal sequence (512 k-tiles,
    131328 tile pairs; the last q-tile's dQ sums 512 k-tiles); dQ on sampled query rows, dK and
    dV on sampled keys of the last eight k-tiles (few rows see those, which
    keeps the oracle quick)."""
    L = 65536
    w = W.random_workload(12, "causal", [L], num_heads=1, head_dim=128)
    do = W.grad_output(w, seed=12)
    got = run_bwd(w, do)
    for g in got:
        assert torch.isfinite(g.float()).all()
    q_rows = sample_rows(w, seed=12)
    rng = np.random.default_rng(12)
    k_rows = sorted(set(rng.integers(L - 1024, L, 24).tolist()) | {L - 1024, L - 897, L - 896, L - 1})
    ref = oracle.attention_backward_sampled(w.q, w.k, w.v, do, w.kind, w.cu_seqlens, w.meta(),
                                            heads=[0], q_rows=q_rows, k_rows=k_rows)
    check(f"{w.name} dQ", got[0], ref[0], rows=q_rows, heads=[0])
    check(f"{w.name} dK", got[1], ref[1], rows=k_rows, heads=[0])
    check(f"{w.name} dV", got[2], ref[2], rows=k_rows, heads=[0])


def test_small_config_fp32_inputs_rounded_to_bf16():
    """The 64-token fp32 workload, rounded to bf16 for the backward (the
    backward has no fp32 path): every element against the oracle on the
    rounded inputs."""
    w = full_workload(1)
    wb = W.Workload(w.name, w.kind, w.cu_seqlens, w.num_heads, w.head_dim, torch.bfloat16,
                    q=w.q.bfloat16(), k=w.k.bfloat16(), v=w.v.bfloat16())
    do = W.grad_output(wb, seed=11)
    compare_all(wb, do, run_bwd(wb, do))


def test_dq_follows_each_rows_upstream_scale():
    """dO rows spanning twenty binary orders of magnitude, and a tenth of them
    zero (as under a loss mask): the dQ of the smallest rows meets the bar
    relative to their own size, not to the largest row's (the fixed-point
    quantum follows each row's ||dO_i||), and zero rows get exactly zero."""
    w = W.random_workload(91, "causal_document", [700, 1300, 129], num_heads=2, head_dim=128)
    rng = np.random.default_rng(91)
    e = rng.integers(0, 21, w.total_tokens)
    f = 2.0 ** -e.astype(np.float64)
    f[rng.random(w.total_tokens) < 0.1] = 0.0
    do = (W.grad_output(w, seed=91).float() * torch.from_numpy(f).float()[:, None, None]).bfloat16()
    got = run_bwd(w, do)
    ref = oracle.attention_backward(w.q, w.k, w.v, do, w.kind, w.cu_seqlens, w.meta())
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        check(name, g, r)
    small = np.flatnonzero((e >= 16) & (f > 0)).tolist()
    zero = np.flatnonzero(f == 0).tolist()
    assert len(small) > 50 and len(zero) > 50
    check("dQ of the rows scaled by 2^-16 .. 2^-20", got[0], ref[0], rows=small)
    assert torch.count_nonzero(got[0][zero]).item() == 0


def test_deterministic_repeats_bit_identical():
    w = full_workload(3)
    do = W.grad_output(w, seed=3)
    a = run_bwd(w, do)
    b = run_bwd(w, do)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_packing_invariance_bit_exact():
    """The same sequence packed at different batch positions gets bit-identical
    gradients (xorl issue, "Batch / packing invariance")."""
    H, D, A = 2, 128, 517
    g = torch.Generator().manual_seed(12)
    qa, ka, va, da = (torch.randn(A, H, D, generator=g).bfloat16() for _ in range(4))
    ref = None
    for pre in ([], [300], [1, 129], [1000, 64]):
        lens = pre + [A] + [77]
        T = sum(lens)
        q, k, v, do = (torch.randn(T, H, D).bfloat16() for _ in range(4))
        s = sum(pre)
        q[s:s + A], k[s:s + A], v[s:s + A], do[s:s + A] = qa, ka, va, da
        w = W.Workload("pack", "causal", W._cu(lens), H, D, torch.bfloat16, q=q, k=k, v=v)
        got = tuple(x[s:s + A] for x in run_bwd(w, do))
        if ref is None:
            ref = got
        else:
            for x, y in zip(ref, got):
                assert torch.equal(x, y)


def test_neighbour_sequence_nonfinite_does_not_leak():
    """Ragged last tiles load rows of the next packed sequence; inf and NaN
    there must not reach this sequence's gradients."""
    lens = [200, 300]
    w = W.random_workload(9, "causal", lens, num_heads=2, head_dim=128)
    do = W.grad_output(w, seed=9)
    clean = run_bwd(w, do)
    qp, kp, vp, dp = w.q.clone(), w.k.clone(), w.v.clone(), do.clone()
    qp[200:] = float("inf")
    kp[200:] = float("inf")
    vp[200:] = float("nan")
    dp[200:] = float("nan")
    dirty = run_bwd(w, dp, q=qp, k=kp, v=vp)
    for x, y in zip(clean, dirty):
        assert torch.equal(x[:200], y[:200])


def test_empty_tiles_are_never_used():
    """With a causal mask the last k-tile is EMPTY for every earlier q-tile: NaN
    keys and values there must leave the dQ of every earlier query exact (a
    skipped tile is never loaded, Ch. 9, Section 9.2)."""
    w = W.random_workload(43, "causal", [1000], num_heads=2, head_dim=128)
    do = W.grad_output(w, seed=43)
    kp, vp = w.k.clone(), w.v.clone()
    kp[896:] = float("nan")
    vp[896:] = float("nan")
    dq, _, _ = run_bwd(w, do, k=kp, v=vp)
    ref = oracle.attention_backward_sampled(w.q, w.k, w.v, do, w.kind, w.cu_seqlens,
                                            q_rows=range(896))
    check("dQ rows before the NaN k-tile", dq, ref[0], rows=list(range(896)))


def test_invalid_dtype_and_mask_mismatch():
    w = W.random_workload(2, "shared_prefix", [300], num_heads=1, head_dim=64)
    dm = w.device_meta()
    bm = build_mask(w, dm)
    q = w.q.cuda()
    lse = torch.zeros((1, 300), device="cuda")
    with pytest.raises(api.AttnError) as e:
        api.attn_bwd(q.float(), q.float(), q.float(), q.float(), lse, q.float(), bm, w.kind,
                     dm["cu_seqlens"], w.max_seqlen, seg_id=dm["seg_id"])
    assert e.value.status == 2
    with pytest.raises(api.AttnError) as e:
        api.attn_bwd(q, q, q, q, lse, q, bm, "causal", dm["cu_seqlens"], w.max_seqlen)
    assert e.value.status == 4


def test_workspace_is_linear_in_tokens_heads_and_dims():
    """The backward's workspace holds per-row side values (LSE, D, the
    fixed-point multiplier) and ||dO_i||, the int32 dQ accumulator and
    per-sequence bound words, O(T H D); no storage per tile pair (the 32k
    workload's 32 heads take about 0.56 GB)."""
    w = full_workload(5)
    dm = w.device_meta()
    bm = build_mask(w, dm)
    T, H, D = w.total_tokens, w.num_heads, w.head_dim
    size = api.attn_bwd_workspace_size(bm, H, D)
    side = 4 * H * bm.struct.max_qtiles * 3 * 128
    assert side + 4 * T * H * (D + 1) <= size < side + 4 * T * H * (D + 1) + (1 << 20)
    # a too small workspace is refused before any launch
    with pytest.raises(api.AttnError) as e:
        api.attn_bwd(w.q.cuda(), w.k.cuda(), w.v.cuda(), w.q.cuda(), torch.zeros((H, T), device="cuda"),
                     w.q.cuda(), bm, w.kind, dm["cu_seqlens"], w.max_seqlen,
                     workspace=torch.empty(size - 256, dtype=torch.uint8, device="cuda"), **w.api_kwargs(dm))
    assert e.value.status == 3


def test_dq_is_bit_identical_under_other_work():
    """dQ is the same bit for bit when the backward shares the GPU with other
    kernels (its CTAs then start at other times, take other items and add
    into the accumulator in another order): the fixed-point sums do not
    depend on the order of the adds."""
    w = W.random_workload(82, "causal_document", [3000, 2500, 700], num_heads=8, head_dim=128)
    do = W.grad_output(w, seed=82)
    ref = run_bwd(w, do)
    dm = w.device_meta()
    bm = build_mask(w, dm)
    kw = w.api_kwargs(dm)
    q, k, v, dod = w.q.cuda(), w.k.cuda(), w.v.cuda(), do.cuda()
    o, lse = api.attn_fwd(q, k, v, bm, w.kind, dm["cu_seqlens"], w.max_seqlen, **kw)
    side = torch.cuda.Stream()
    big = torch.randn(4096, 4096, device="cuda")
    for _ in range(3):
        with torch.cuda.stream(side):
            for _ in range(4):
                big = big @ big * 1e-3
        got = api.attn_bwd(q, k, v, o, lse, dod, bm, w.kind, dm["cu_seqlens"], w.max_seqlen, **kw)
        torch.cuda.synchronize()
        assert api.attn_get_status(bm) == api.ATTN_OK
        for x, y in zip(got, ref):
            assert torch.equal(x.cpu(), y)


def test_one_mask_serves_overlapping_forward_and_backward():
    """One block mask, built once, serves forwards on one stream while backwards
    run on another (the reuse across layers the xorl issue asks for, Proposed
    work, item 3): the kernels only read the mask, their work counters belong
    to each launch.  Every result matches the oracle and equals the serial run
    bit for bit."""
    w = W.random_workload(81, "strip_thinking", [1500, 700, 257], num_heads=4, head_dim=128)
    do = W.grad_output(w, seed=81)
    dm = w.device_meta()
    bm = build_mask(w, dm)
    kw = w.api_kwargs(dm)
    q, k, v, dod = w.q.cuda(), w.k.cuda(), w.v.cuda(), do.cuda()
    o, lse = api.attn_fwd(q, k, v, bm, w.kind, dm["cu_seqlens"], w.max_seqlen, **kw)
    g_ser = api.attn_bwd(q, k, v, o, lse, dod, bm, w.kind, dm["cu_seqlens"], w.max_seqlen, **kw)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    fwd_out, bwd_out = [], []
    for _ in range(4):
        with torch.cuda.stream(sa):
            fwd_out.append(api.attn_fwd(q, k, v, bm, w.kind, dm["cu_seqlens"], w.max_seqlen, **kw))
        with torch.cuda.stream(sb):
            bwd_out.append(api.attn_bwd(q, k, v, o, lse, dod, bm, w.kind, dm["cu_seqlens"],
                                        w.max_seqlen, **kw))
    torch.cuda.synchronize()
    assert api.attn_get_status(bm) == api.ATTN_OK
    for o2, l2 in fwd_out:
        assert torch.equal(o2, o) and torch.equal(l2, lse)
    for g in bwd_out:
        for x, y in zip(g, g_ser):
            assert torch.equal(x, y)
    O, L = oracle.attention(w.q, w.k, w.v, w.kind, w.cu_seqlens, w.meta())
    assert np.abs(o.float().cpu().numpy() - O).max() <= 2e-2
    assert np.abs(lse.cpu().numpy() - L).max() <= 1e-3
    compare_all(w, do, tuple(x.cpu() for x in g_ser))
