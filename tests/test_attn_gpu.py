"""GPU attention forward vs the fp64 oracle on the same seeded inputs.

Tolerances (from the target statement): bf16 in / fp32 accumulate, O max-abs
error <= 2e-2 and LSE max-abs error <= 1e-3.  The fp32 path is held to a
tighter 1e-4 on both.  Small cases are compared element by element; the five
full-size workloads run in the launch configuration the benchmark times and
are compared on sampled rows the oracle computes one by one.
"""
import functools

import numpy as np
import pytest
import torch

import oracle
from block_sparse_masked_mask_gb300 import api
from block_sparse_masked_mask_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: (2e-2, 1e-3), torch.float32: (1e-4, 1e-4)}


def run_gpu(w, q=None, k=None, v=None, bm=None, dm=None):
    dm = dm or w.device_meta()
    if bm is None:
        bm = api.attn_block_mask_build(w.kind, dm["cu_seqlens"], w.total_tokens, w.max_seqlen,
                                       **w.api_kwargs(dm))
    q = (w.q if q is None else q).cuda()
    k = (w.k if k is None else k).cuda()
    v = (w.v if v is None else v).cuda()
    o, lse = api.attn_fwd(q, k, v, bm, w.kind, dm["cu_seqlens"], w.max_seqlen, **w.api_kwargs(dm))
    assert api.attn_get_status(bm) == api.ATTN_OK
    return o, lse


def compare(w, o, lse, rows=None, heads=None, q=None, k=None, v=None):
    q = w.q if q is None else q
    k = w.k if k is None else k
    v = w.v if v is None else v
    O, L = oracle.attention(q, k, v, w.kind, w.cu_seqlens, w.meta(), rows=rows, heads=heads)
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    sel_r = np.arange(w.total_tokens) if rows is None else np.unique(np.asarray(rows))
    sel_h = list(range(w.num_heads)) if heads is None else list(heads)
    eo = np.abs(o[sel_r][:, sel_h] - O[sel_r][:, sel_h]).max() if len(sel_r) else 0.0
    lg, lw = lse[sel_h][:, sel_r], L[sel_h][:, sel_r]
    # a row that sees no key has LSE = -inf on both sides (and O = 0)
    empty = lw == -np.inf
    assert (lg[empty] == -np.inf).all(), "a row with no visible key needs LSE = -inf"
    el = np.abs(lg[~empty] - lw[~empty]).max(initial=0.0) if len(sel_r) else 0.0
    to, tl = TOL[w.dtype]
    assert np.isfinite(eo) and np.isfinite(el)
    assert eo <= to, f"{w.name}: O max abs err {eo}"
    assert el <= tl, f"{w.name}: LSE max abs err {el}"
    return eo, el


SMALL_LENGTHS = [300, 1, 129, 517, 0, 128]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("kind", oracle.KINDS)
def test_small_all_elements(kind, D, dtype):
    w = W.random_workload(5 + D, kind, SMALL_LENGTHS, num_heads=2, head_dim=D, dtype=dtype)
    o, lse = run_gpu(w)
    compare(w, o, lse)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("kind", ["causal_document", "shared_prefix", "strip_thinking",
                                  "strip_thinking_dup"])
def test_small_repeating_ids_all_elements(kind, D):
    """Ids and turns drawn from a small alphabet: the rows of a warp often hold
    different query codes, so PARTIAL tiles take the per-row predicate path
    rather than the per-warp ballot."""
    w = W.random_workload(70 + D, kind, [700, 255, 1000], num_heads=2, head_dim=D, id_alphabet=4)
    o, lse = run_gpu(w)
    compare(w, o, lse)


@pytest.mark.parametrize("lens", [[1], [2], [127], [128], [129], [255, 257], [1000]])
def test_ragged_shapes_causal(lens):
    w = W.random_workload(sum(lens), "causal", lens, num_heads=3, head_dim=128)
    o, lse = run_gpu(w)
    compare(w, o, lse)


def test_scale_argument_is_used():
    w = W.random_workload(3, "causal", [300], num_heads=1, head_dim=64)
    dm = w.device_meta()
    bm = api.attn_block_mask_build(w.kind, dm["cu_seqlens"], w.total_tokens, w.max_seqlen)
    o, lse = api.attn_fwd(w.q.cuda(), w.k.cuda(), w.v.cuda(), bm, w.kind, dm["cu_seqlens"],
                          w.max_seqlen, scale=0.37)
    O, L = oracle.attention(w.q, w.k, w.v, w.kind, w.cu_seqlens, scale=0.37)
    assert np.abs(o.float().cpu().numpy() - O).max() <= 2e-2
    assert np.abs(lse.cpu().numpy() - L).max() <= 1e-3


@functools.lru_cache(maxsize=None)
def full_workload(c, form="mask"):
    return W.make_workload(c, tensors=True, document_form=form)


def sample_rows(w, n=96, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(rng.integers(0, w.total_tokens, n).tolist())
    for b in range(w.batch):
        s0, s1 = int(w.cu_seqlens[b]), int(w.cu_seqlens[b + 1])
        if s1 > s0:
            rows.update([s0, s1 - 1, min(s1 - 1, s0 + 127), min(s1 - 1, s0 + 128)])
    return sorted(rows)


@pytest.mark.parametrize("c,form", [(1, "mask"), (2, "mask"), (3, "mask"), (4, "mask"),
                                    (5, "mask"), (5, "cu_seqlens"), (6, "mask"), (7, "mask"),
                                    (8, "mask")])
def test_full_size_workloads_sampled(c, form):
    w = full_workload(c, form)
    o, lse = run_gpu(w)
    if c == 1:
        compare(w, o, lse)  # small enough for every element
        return
    rows = sample_rows(w)
    heads = [0, w.num_heads - 1]
    compare(w, o, lse, rows=rows, heads=heads)
    # every output is finite; every LSE too, except -inf on rows that see no
    # key (the padding of the dense workload)
    assert torch.isfinite(o.float()).all()
    assert torch.isfinite(lse).all() or w.kind == "dense"
    assert not torch.isnan(lse).any() and not (lse == float("inf")).any()


def test_longest_single_sequence_sampled():
    """The largest case: one 131072-token causal sequence (1024 q-tiles, 524800
    listed tile pairs per head), compared on sampled rows; the last row sees
    all 131072 keys."""
    w = W.random_workload(11, "causal", [131072], num_heads=2, head_dim=128)
    o, lse = run_gpu(w)
    compare(w, o, lse, rows=sample_rows(w, n=24, seed=11), heads=[0, 1])
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_deterministic_repeats_bit_identical():
    w = full_workload(3)
    o1, l1 = run_gpu(w)
    o2, l2 = run_gpu(w)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_packing_invariance_bit_exact():
    """The same sequence packed at different batch positions gives bit-identical
    rows (xorl issue, "Batch / packing invariance")."""
    rng = np.random.default_rng(5)
    H, D = 2, 128
    A = 517
    others = [[], [300], [1, 129], [1000, 64]]
    qa, ka, va = (torch.randn(A, H, D, generator=torch.Generator().manual_seed(i)).bfloat16()
                  for i in range(3))
    ref = None
    for pre in others:
        lens = pre + [A] + [77]
        T = sum(lens)
        q, k, v = (torch.randn(T, H, D).bfloat16() for _ in range(3))
        s = sum(pre)
        q[s:s + A], k[s:s + A], v[s:s + A] = qa, ka, va
        w = W.Workload("pack", "causal", W._cu(lens), H, D, torch.bfloat16, q=q, k=k, v=v)
        o, lse = run_gpu(w)
        got = (o[s:s + A].cpu(), lse[:, s:s + A].cpu())
        if ref is None:
            ref = got
        else:
            assert torch.equal(ref[0], got[0]) and torch.equal(ref[1], got[1])


def test_empty_tiles_are_never_used():
    """K and V of tokens that only EMPTY tiles would reach are NaN; every row
    that cannot see them stays finite and correct (Ch. 9, Section 9.2: a
    skipped tile's loads never run)."""
    rng = np.random.default_rng(9)
    # causal: the last k-tile is EMPTY for every earlier q-tile
    w = W.random_workload(41, "causal", [1000], num_heads=2, head_dim=128)
    kp, vp = w.k.clone(), w.v.clone()
    kp[896:] = float("nan")
    vp[896:] = float("nan")
    o, lse = run_gpu(w, k=kp, v=vp)
    compare(w, o[:896], lse[:, :896], rows=list(range(896)))
    # shared prefix with tile-aligned segments: suffix 4 (tiles 8-9) is EMPTY
    # for the prefix and every other suffix
    seg = np.concatenate([np.zeros(256, np.int32)] + [np.full(256, i, np.int32) for i in range(1, 5)])
    w = W.Workload("sp", "shared_prefix", W._cu([len(seg)]), 2, 128, torch.bfloat16, seg=seg)
    g = torch.Generator().manual_seed(3)
    w.q, w.k, w.v = (torch.randn(len(seg), 2, 128, generator=g).bfloat16() for _ in range(3))
    kp, vp = w.k.clone(), w.v.clone()
    kp[1024:] = float("nan")
    vp[1024:] = float("nan")
    o, lse = run_gpu(w, k=kp, v=vp)
    keep = list(range(1024))
    O, L = oracle.attention(w.q, w.k, w.v, w.kind, w.cu_seqlens, w.meta(), rows=keep)
    assert np.abs(o[:1024].float().cpu().numpy() - O[:1024]).max() <= 2e-2
    assert np.abs(lse[:, :1024].cpu().numpy() - L[:, :1024]).max() <= 1e-3


def test_neighbour_sequence_nan_does_not_leak():
    """A ragged last tile loads rows of the next packed sequence; non-finite
    values there must not reach this sequence's output."""
    lens = [200, 300]
    w = W.random_workload(8, "causal", lens, num_heads=2, head_dim=128)
    kp, vp = w.k.clone(), w.v.clone()
    kp[200:] = float("inf")
    vp[200:] = float("nan")
    o, lse = run_gpu(w, k=kp, v=vp)
    O, L = oracle.attention(w.q, w.k, w.v, w.kind, w.cu_seqlens, rows=list(range(200)))
    assert np.abs(o[:200].float().cpu().numpy() - O[:200]).max() <= 2e-2
    assert np.abs(lse[:, :200].cpu().numpy() - L[:, :200]).max() <= 1e-3


def test_wrong_task_negative():
    """Ch. 21, Worked Example 21.2.2: causal output differs from non-causal
    attention by far more than rounding on the same inputs."""
    torch.manual_seed(0)
    q, k, v = (torch.randn(20, 8) for _ in range(3))
    # pad to D=32 with zeros: scores and values are unchanged
    pad = lambda x: torch.nn.functional.pad(x, (0, 24)).reshape(20, 1, 32)
    w = W.Workload("wrong_task", "causal", W._cu([20]), 1, 32, torch.float32,
                   q=pad(q), k=pad(k), v=pad(v))
    # the padded head_dim would change the default scale: pass 1/sqrt(8)
    dm = w.device_meta()
    bm = api.attn_block_mask_build("causal", dm["cu_seqlens"], 20, 20)
    o, lse = api.attn_fwd(w.q.cuda(), w.k.cuda(), w.v.cuda(), bm, "causal", dm["cu_seqlens"], 20,
                          scale=1 / np.sqrt(8))
    o = o.cpu()[:, 0, :8].double().numpy()
    noncausal = torch.softmax(q.double() @ k.double().T / np.sqrt(8), -1) @ v.double()
    causal_ref, _ = oracle.masked_attention(q.double().numpy(), k.double().numpy(),
                                            v.double().numpy(), np.tril(np.ones((20, 20), bool)),
                                            1 / np.sqrt(8))
    assert np.abs(o - causal_ref).max() < 1e-4
    assert abs(np.abs(o - noncausal.numpy()).max() - 1.7221667766571045) < 1e-4


def test_mask_mismatch_and_metadata_errors():
    w = W.random_workload(1, "shared_prefix", [300], num_heads=1, head_dim=64)
    dm = w.device_meta()
    bm = api.attn_block_mask_build(w.kind, dm["cu_seqlens"], w.total_tokens, w.max_seqlen,
                                   seg_id=dm["seg_id"])
    q = w.q.cuda()
    with pytest.raises(api.AttnError) as e:
        api.attn_fwd(q, q, q, bm, "causal", dm["cu_seqlens"], w.max_seqlen)
    assert e.value.status == 4
    with pytest.raises(api.AttnError) as e:
        api.attn_fwd(q, q, q, bm, w.kind, dm["cu_seqlens"], w.max_seqlen)
    assert e.value.status == 1
    other_cu = dm["cu_seqlens"].clone()
    with pytest.raises(api.AttnError) as e:
        api.attn_fwd(q, q, q, bm, w.kind, other_cu, w.max_seqlen, seg_id=dm["seg_id"])
    assert e.value.status == 4


def test_binding_refuses_misread_tensors():
    """Views, wrong element types and wrong shapes are refused by the binding
    (ATTN_ERR_INVALID_ARG) instead of being read as dense [T, H, D] data."""
    w = W.random_workload(1, "shared_prefix", [300], num_heads=2, head_dim=64)
    dm = w.device_meta()
    bm = api.attn_block_mask_build(w.kind, dm["cu_seqlens"], w.total_tokens, w.max_seqlen,
                                   seg_id=dm["seg_id"])
    q = w.q.cuda()
    seg = dm["seg_id"]
    bad = [
        dict(q=q.transpose(0, 1).contiguous().transpose(0, 1)),   # a strided view
        dict(k=q.float()),                                         # k's type differs from q's
        dict(v=q[:, :1]),                                          # wrong shape
        dict(seg_id=seg.long()),                                   # int64 ids
        dict(lse=torch.empty((w.total_tokens, 2), device="cuda")),  # [T, H] instead of [H, T]
    ]
    for over in bad:
        kw = dict(q=q, k=q, v=q, seg_id=seg)
        kw.update(over)
        extra = {"lse": kw.pop("lse")} if "lse" in kw else {}
        with pytest.raises(api.AttnError) as e:
            api.attn_fwd(kw["q"], kw["k"], kw["v"], bm, w.kind, dm["cu_seqlens"], w.max_seqlen,
                         seg_id=kw["seg_id"], **extra)
        assert e.value.status == 1, over.keys()
    with pytest.raises(api.AttnError) as e:
        api.attn_block_mask_build(w.kind, dm["cu_seqlens"].long(), w.total_tokens, w.max_seqlen,
                                  seg_id=seg)
    assert e.value.status == 1


def test_repeated_forwards_on_one_mask():
    """The forward's work counters return to zero after every launch, so a
    mask serves any number of forwards with different inputs."""
    w = W.random_workload(12, "causal_document", [900, 1300], num_heads=3, head_dim=128)
    dm = w.device_meta()
    bm = api.attn_block_mask_build(w.kind, dm["cu_seqlens"], w.total_tokens, w.max_seqlen,
                                   seg_id=dm["seg_id"])
    for i in range(3):
        g = torch.Generator().manual_seed(100 + i)
        q, k, v = (torch.randn(w.total_tokens, 3, 128, generator=g).bfloat16() for _ in range(3))
        o, lse = api.attn_fwd(q.cuda(), k.cuda(), v.cuda(), bm, w.kind, dm["cu_seqlens"],
                              w.max_seqlen, seg_id=dm["seg_id"])
        assert api.attn_get_status(bm) == api.ATTN_OK
        rows = list(range(0, w.total_tokens, 7))
        O, L = oracle.attention(q, k, v, w.kind, w.cu_seqlens, w.meta(), rows=rows)
        assert np.abs(o.float().cpu().numpy()[rows] - O[rows]).max() <= 2e-2
        assert np.abs(lse.cpu().numpy()[:, rows] - L[:, rows]).max() <= 1e-3
        assert bm.header()[8:10].tolist() == [0, 0]
