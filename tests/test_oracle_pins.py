"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Nothing here calls the CUDA path.  Each test names the passage it checks.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import core as oa
from block_sparse_masked_mask_gb300 import workloads as W

from conftest import GOLDEN


def _read_blocks(name):
    blocks, cur = {}, None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            toks = line.split()
            if len(toks) == 1 and not toks[0].lstrip("-").replace(".", "").isdigit():
                cur = toks[0]
                blocks[cur] = []
            else:
                blocks[cur].append(toks)
    return blocks


def _causal_mask(L):
    return oracle.sequence_mask("causal", np.array([0, L]), 0, {})


# ----------------------------------------------------------------------------
# Causal predicate: Ch. 9, Section 9.1, Worked Examples 9.1.1 and 9.1.2.
# ----------------------------------------------------------------------------

def test_causal_4x4_matches_page_table():
    g = _read_blocks("causal_4x4.txt")
    x = np.array(g["input"], dtype=float)
    want = np.array(g["causal_masked"], dtype=float)
    got = np.where(_causal_mask(4), x, 0.0)
    assert np.array_equal(got, want)
    assert np.array_equal(got, np.tril(x))


def test_strict_lt_trap_is_not_the_oracle():
    g = _read_blocks("strict_lt_4x4.txt")
    strict = np.array(g["strict_masked"], dtype=float)
    x = np.arange(1, 17, dtype=float).reshape(4, 4)
    got = np.where(_causal_mask(4), x, 0.0)
    assert not np.array_equal(got, strict)
    # the page's trap table is exactly the oracle's table minus the diagonal
    assert np.array_equal(got - np.diag(np.diag(x)), strict)


# ----------------------------------------------------------------------------
# Whole-oracle pin against a printed value: Ch. 21, Worked Example 21.2.2.
# ----------------------------------------------------------------------------

def _wrong_task_inputs():
    torch.manual_seed(0)
    q = torch.randn(20, 8)
    k = torch.randn(20, 8)
    v = torch.randn(20, 8)
    return q.double().numpy(), k.double().numpy(), v.double().numpy()


def test_wrong_task_max_diff_matches_page():
    vals = {}
    with open(os.path.join(GOLDEN, "wrong_task.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            a, b = line.split()
            vals[a] = b
    want = float(vals["max_abs_diff_causal_vs_noncausal"])
    q, k, v = _wrong_task_inputs()
    scale = 1.0 / math.sqrt(8)
    oc, _ = oracle.masked_attention(q, k, v, _causal_mask(20), scale)
    on, _ = oracle.masked_attention(q, k, v, np.ones((20, 20), bool), scale)
    diff = np.abs(oc - on).max()
    # the page computed in fp32; fp64 differs from it by rounding only
    assert abs(diff - want) < 1e-6, diff


def test_none_kind_reproduces_the_pages_wrong_task_numbers():
    """The "none" kind through the full attention() path is the non-causal
    attention of Worked Example 21.2.2: against the causal kind on the same
    inputs its largest difference is the page's printed figure."""
    vals = {}
    with open(os.path.join(GOLDEN, "wrong_task.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            a, b = line.split()
            vals[a] = b
    q, k, v = (x[:, None, :] for x in _wrong_task_inputs())
    cu = np.array([0, 20])
    on, _ = oracle.attention(q, k, v, "none", cu, scale=1 / math.sqrt(8))
    oc, _ = oracle.attention(q, k, v, "causal", cu, scale=1 / math.sqrt(8))
    assert abs(np.abs(oc - on).max() - float(vals["max_abs_diff_causal_vs_noncausal"])) < 1e-6


def test_none_kind_is_plain_softmax_per_sequence():
    """Ch. 21, Worked Example 21.1.1: flash attention verified against
    softmax(Q K^T / sqrt(d)) V computed the naive way on shapes aligned to no
    block; here per packed sequence, through the oracle's none kind."""
    rng = np.random.default_rng(17)
    lens = [17, 23, 1]
    cu = W._cu(lens)
    T, H, D = sum(lens), 2, 8
    q, k, v = (rng.standard_normal((T, H, D)) for _ in range(3))
    O, LSE = oracle.attention(q, k, v, "none", cu)
    for b in range(len(lens)):
        s = slice(cu[b], cu[b + 1])
        for h in range(H):
            sc = q[s, h] @ k[s, h].T / np.sqrt(D)
            p = np.exp(sc - sc.max(axis=1, keepdims=True))
            assert np.abs(O[s, h] - (p / p.sum(axis=1, keepdims=True)) @ v[s, h]).max() < 1e-12


def _dense_from(kind, cu, meta):
    """The bits of another kind's mask, packed as the dense kind reads them."""
    rows = [W.pack_rows(oracle.sequence_mask(kind, cu, b, meta)).ravel() for b in range(len(cu) - 1)]
    return np.concatenate(rows).astype(np.uint32), W.dense_offsets(np.diff(cu))


@pytest.mark.parametrize("kind", ["causal", "causal_document", "strip_thinking_dup"])
def test_dense_kind_carrying_a_predicate_equals_that_kind(kind):
    """A dense mask holding another kind's pairs gives that kind's outputs
    exactly, and the same tile labels."""
    rng = np.random.default_rng(31)
    lens = [150, 1, 290]
    meta = W.random_meta(rng, kind, lens)
    cu = W._cu(lens)
    bits, offs = _dense_from(kind, cu, meta)
    dmeta = {"dense_bits": bits, "dense_offsets": offs}
    T, H, D = sum(lens), 2, 16
    q, k, v = (rng.standard_normal((T, H, D)) for _ in range(3))
    O1, L1 = oracle.attention(q, k, v, kind, cu, meta)
    O2, L2 = oracle.attention(q, k, v, "dense", cu, dmeta)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)
    for a, b in zip(oracle.tile_labels(kind, cu, meta), oracle.tile_labels("dense", cu, dmeta)):
        assert np.array_equal(a, b)


def test_dense_causal_document_padding_equals_the_tokens_without_padding():
    """The causal + document + padding composition (xorl issue, "Current state
    in this tree": make_causal_block_mask) as a dense mask: padding tokens
    neither attend nor are attended, so every other token's output is the
    causal+document output of the sequence with the padding taken out; a
    padding token's row sees nothing (O = 0, LSE = -inf)."""
    rng = np.random.default_rng(32)
    docs = [40, 1, 75]
    pad = 30
    L = sum(docs) + pad
    seg = np.concatenate([np.full(n, i, np.int32) for i, n in enumerate(docs)] + [np.full(pad, -1, np.int32)])
    keep = seg >= 0
    qi, ki = np.arange(L)[:, None], np.arange(L)[None, :]
    m = (ki <= qi) & (seg[ki] == seg[qi]) & keep[ki] & keep[qi]
    dmeta = {"dense_bits": W.pack_rows(m, rng).ravel(), "dense_offsets": W.dense_offsets([L])}
    H, D = 2, 8
    q, k, v = (rng.standard_normal((L, H, D)) for _ in range(3))
    O, LSE = oracle.attention(q, k, v, "dense", np.array([0, L]), dmeta)
    Ok, Lk = oracle.attention(q[keep], k[keep], v[keep], "causal_document", np.array([0, keep.sum()]),
                              {"seg": seg[keep]})
    assert np.abs(O[keep] - Ok).max() < 1e-12 and np.abs(LSE[:, keep] - Lk).max() < 1e-12
    assert (O[~keep] == 0).all() and (LSE[:, ~keep] == -np.inf).all()


# ----------------------------------------------------------------------------
# Closed forms and special cases.
# ----------------------------------------------------------------------------

def test_causal_row0_is_v0_and_lse_is_s00():
    rng = np.random.default_rng(3)
    q, k, v = (rng.standard_normal((37, 16)) for _ in range(3))
    scale = 0.25
    o, lse = oracle.masked_attention(q, k, v, _causal_mask(37), scale)
    assert np.array_equal(o[0], v[0])
    assert lse[0] == (q[0] @ k[0]) * scale


def test_fully_masked_row_gives_zero_and_minus_inf():
    rng = np.random.default_rng(4)
    q, k, v = (rng.standard_normal((5, 8)) for _ in range(3))
    mask = np.ones((5, 5), bool)
    mask[2] = False
    o, lse = oracle.masked_attention(q, k, v, mask, 0.3)
    assert np.all(o[2] == 0) and lse[2] == -np.inf
    assert np.all(np.isfinite(o[[0, 1, 3, 4]]))


def test_single_key_visible_everywhere_returns_that_value():
    # softmax over one element is 1 whatever the score
    rng = np.random.default_rng(5)
    q, k, v = (rng.standard_normal((6, 4)) for _ in range(3))
    mask = np.zeros((6, 6), bool)
    mask[:, 3] = True
    o, lse = oracle.masked_attention(q, k, v, mask, 1.7)
    assert np.array_equal(o, np.repeat(v[3:4], 6, axis=0))
    assert np.allclose(lse, (q @ k[3]) * 1.7, rtol=0, atol=1e-15)


@pytest.mark.parametrize("kind", oracle.KINDS)
def test_matches_torch_sdpa_fp64(kind):
    """The softmax step reduces to a library routine: torch's fp64 SDPA with a
    boolean mask, and logsumexp for LSE."""
    rng = np.random.default_rng(11)
    lens = [70, 1, 33, 150]
    meta = W.random_meta(rng, kind, lens)
    cu = W._cu(lens)
    T, H, D = sum(lens), 3, 24
    q, k, v = (torch.randn(T, H, D, dtype=torch.float64) for _ in range(3))
    O, LSE = oracle.attention(q, k, v, kind, cu, meta)
    scale = 1 / math.sqrt(D)
    for b in range(len(lens)):
        s0, s1 = cu[b], cu[b + 1]
        mask = torch.from_numpy(oracle.sequence_mask(kind, cu, b, meta))
        for h in range(H):
            qh, kh, vh = q[s0:s1, h], k[s0:s1, h], v[s0:s1, h]
            ref = torch.nn.functional.scaled_dot_product_attention(
                qh[None], kh[None], vh[None], attn_mask=mask[None], scale=scale)[0]
            sc = (qh @ kh.T * scale).masked_fill(~mask, -math.inf)
            lse = torch.logsumexp(sc, -1).numpy()
            # a row that sees no key: O = 0 and LSE = -inf (SDPA gives NaN there)
            seen = mask.any(-1).numpy()
            assert (O[s0:s1, h][~seen] == 0).all() and (LSE[h, s0:s1][~seen] == -np.inf).all()
            assert np.abs(O[s0:s1, h][seen] - ref.numpy()[seen]).max(initial=0) < 1e-12
            assert np.abs(LSE[h, s0:s1][seen] - lse[seen]).max(initial=0) < 1e-12


def test_online_softmax_equals_three_pass():
    """The tiled online update of Ch. 21, Section 21.1 (running max m, running
    sum l, accumulator rescaled by alpha = exp(m_old - m_new), final acc / l),
    restated here in fp64, equals the oracle's three-pass definition for every
    tile width: the tile size is a performance knob, never a correctness one."""
    rng = np.random.default_rng(7)
    M, N, D = 17, 23, 8
    q, k, v = rng.standard_normal((M, D)), rng.standard_normal((N, D)), rng.standard_normal((N, D))
    mask = rng.random((M, N)) < 0.6
    mask[:, 0] = True
    scale = 1 / math.sqrt(D)
    want_o, want_lse = oracle.masked_attention(q, k, v, mask, scale)
    for bn in (1, 3, 4, 64, 128):
        m = np.full(M, -np.inf)
        l = np.zeros(M)
        acc = np.zeros((M, D))
        for n0 in range(0, N, bn):
            s = (q @ k[n0:n0 + bn].T) * scale
            s = np.where(mask[:, n0:n0 + bn], s, -np.inf)
            m_new = np.maximum(m, s.max(axis=1))
            m_safe = np.where(np.isfinite(m_new), m_new, 0.0)
            alpha = np.exp(m - m_safe)
            p = np.exp(s - m_safe[:, None])
            l = alpha * l + p.sum(axis=1)
            acc = alpha[:, None] * acc + p @ v[n0:n0 + bn]
            m = m_new
        assert np.abs(acc / l[:, None] - want_o).max() < 1e-12
        assert np.abs(m + np.log(l) - want_lse).max() < 1e-12


# ----------------------------------------------------------------------------
# Structured masks equal the separate computations they replace.
# ----------------------------------------------------------------------------

def test_shared_prefix_equals_separate_runs():
    """xorl issue, "Shared prefix": each suffix attends prefix + own suffix, which
    must equal running causal attention on P || S_i alone, and the prefix rows
    must equal causal attention over P alone."""
    rng = np.random.default_rng(21)
    P, sufs = 37, [20, 33, 9]
    seg = np.concatenate([np.zeros(P, np.int32)] + [np.full(n, i + 1, np.int32) for i, n in enumerate(sufs)])
    T, H, D = len(seg), 2, 16
    q, k, v = (rng.standard_normal((T, H, D)) for _ in range(3))
    O, LSE = oracle.attention(q, k, v, "shared_prefix", np.array([0, T]), {"seg": seg})
    Op, Lp = oracle.attention(q[:P], k[:P], v[:P], "causal", np.array([0, P]))
    assert np.abs(O[:P] - Op).max() < 1e-12 and np.abs(LSE[:, :P] - Lp).max() < 1e-12
    pos = P
    for n in sufs:
        idx = np.r_[0:P, pos:pos + n]
        Oi, Li = oracle.attention(q[idx], k[idx], v[idx], "causal", np.array([0, P + n]))
        assert np.abs(O[pos:pos + n] - Oi[P:]).max() < 1e-12
        assert np.abs(LSE[:, pos:pos + n] - Li[:, P:]).max() < 1e-12
        pos += n


def test_strip_thinking_equals_per_turn_recomputation():
    """xorl issue, "Strip-thinking multi-turn": turn t sees earlier turns' user
    and answer tokens plus all of its own turn; the naive alternative is one
    causal pass per turn over exactly those tokens."""
    rng = np.random.default_rng(22)
    turns = [(5, 9, 4), (3, 11, 6), (7, 2, 5), (4, 6, 3)]
    role, turn = W.strip_thinking_layout(turns)
    T, H, D = len(role), 2, 8
    q, k, v = (rng.standard_normal((T, H, D)) for _ in range(3))
    O, LSE = oracle.attention(q, k, v, "strip_thinking", np.array([0, T]),
                              {"role": role, "turn": turn, "role_think": W.ROLE_THINK})
    for t in range(1, len(turns) + 1):
        keep = np.nonzero((turn < t) & (role != W.ROLE_THINK) | (turn == t))[0]
        Ot, Lt = oracle.attention(q[keep], k[keep], v[keep], "causal", np.array([0, len(keep)]))
        rows = np.nonzero(turn[keep] == t)[0]
        assert np.abs(O[keep[rows]] - Ot[rows]).max() < 1e-12
        assert np.abs(LSE[:, keep[rows]] - Lt[:, rows]).max() < 1e-12


def _dup_inference_context(role, turn, i):
    """Tokens an inference engine holds when it produces token i of the
    duplicated layout, built from spans, not from the predicate: for turn t,
    every earlier turn contributes its user tokens and its answer-history copy;
    the own turn contributes its user tokens, then its thinking (for THINK and
    ANSWER tokens), then the span of token i itself up to i."""
    t, r = turn[i], role[i]
    idx = np.arange(len(role))
    ctx = [idx[(turn == u) & ((role == W.ROLE_USER) | (role == W.ROLE_ANSWER_HISTORY))] for u in range(1, t)]
    ctx.append(idx[(turn == t) & (role == W.ROLE_USER) & (idx <= i)])
    if r in (W.ROLE_THINK, W.ROLE_ANSWER):
        ctx.append(idx[(turn == t) & (role == W.ROLE_THINK) & (idx <= i)])
    if r in (W.ROLE_ANSWER, W.ROLE_ANSWER_HISTORY):
        ctx.append(idx[(turn == t) & (role == r) & (idx <= i)])
    return np.concatenate(ctx)


def test_strip_thinking_dup_equals_inference_contexts():
    """xorl issue, "The exactness question", option (b): with every answer
    duplicated, each token's output is exactly what inference computes from the
    context it would hold then: earlier turns stripped of thinking (user and
    answer-history tokens), its own turn's user tokens, its own thinking for
    THINK and ANSWER tokens, and its own span causally.  One softmax per token
    over exactly those keys."""
    rng = np.random.default_rng(24)
    turns = [(5, 9, 4), (3, 11, 6), (7, 2, 5), (4, 6, 3)]
    role, turn = W.strip_thinking_dup_layout(turns)
    T, H, D = len(role), 2, 8
    q, k, v = (rng.standard_normal((T, H, D)) for _ in range(3))
    meta = {"role": role, "turn": turn, "role_think": W.ROLE_THINK}
    O, LSE = oracle.attention(q, k, v, "strip_thinking_dup", np.array([0, T]), meta)
    scale = 1 / np.sqrt(D)
    for i in range(T):
        ctx = _dup_inference_context(role, turn, i)
        for h in range(H):
            s = k[ctx, h] @ q[i, h] * scale
            p = np.exp(s - s.max())
            assert abs(LSE[h, i] - (s.max() + np.log(p.sum()))) < 1e-12
            assert np.abs(O[i, h] - p @ v[ctx, h] / p.sum()).max() < 1e-12
    # the answer copy and its history copy differ (the history copy does not
    # see the thinking), and later turns see the history copy, not the answer
    a_rows = np.nonzero(role == W.ROLE_ANSWER)[0]
    h_rows = np.nonzero(role == W.ROLE_ANSWER_HISTORY)[0]
    assert np.abs(O[a_rows] - O[h_rows]).max() > 1e-2
    m = oracle.sequence_mask("strip_thinking_dup", np.array([0, T]), 0, meta)
    later = turn[:, None] > turn[None, :]
    assert not (m & later & (role[None, :] == W.ROLE_ANSWER)).any()
    assert not (m & later & (role[None, :] == W.ROLE_THINK)).any()
    assert (m | ~(later & (role[None, :] == W.ROLE_ANSWER_HISTORY))).all()


def test_strip_thinking_dup_workload_counts_closed_form():
    """Workload 6: per turn, tiles of user 128 (1) / think 768 (6) / answer
    256 (2) / history 256 (2), all spans tile-aligned."""
    w = W.make_workload(6, tensors=False)
    assert w.total_tokens == 11264
    nturn, u, th, a = 8, 128, 768, 256
    lab = oracle.tile_labels(w.kind, w.cu_seqlens, w.meta())[0]
    # closed forms for the pairs: own turn (user, think, answer copy causal over
    # user+think+itself, history copy over user+itself) and earlier turns
    # (user + history copy of each earlier turn, for every token of the turn)
    own = (u * (u + 1) // 2 + th * u + th * (th + 1) // 2 + a * (u + th) + a * (a + 1) // 2
           + a * u + a * (a + 1) // 2)
    per_turn_tokens = u + th + 2 * a
    hist = per_turn_tokens * (u + a)
    nnz = nturn * own + hist * sum(range(nturn))
    assert oracle.unmasked_pairs(w.kind, w.cu_seqlens, w.meta()) == nnz
    # tile labels: within a turn (11 tiles: U, T x6, A x2, H x2) the visible
    # key tiles of each query tile are whole spans, so only diagonal tiles are
    # PARTIAL; earlier turns contribute their U and H tiles FULL
    per = 11
    own_full = sum(len(r) for r in [[], [0], [0, 1], [0, 1, 2], [0, 1, 2, 3], [0, 1, 2, 3, 4],
                                    [0, 1, 2, 3, 4, 5], [0, 1, 2, 3, 4, 5, 6], [0, 1, 2, 3, 4, 5, 6, 7],
                                    [0], [0, 9]])
    full = nturn * own_full + per * 3 * sum(range(nturn))
    partial = nturn * per
    assert oracle.label_totals([lab]) == (full, partial, (nturn * per) ** 2 - full - partial)


def test_varlen_equals_independent_sequences():
    """cu_seqlens packing (xorl issue, Summary): a causal square per sequence and
    nothing across, i.e. each sequence alone."""
    rng = np.random.default_rng(23)
    lens = [13, 1, 40, 7]
    cu = W._cu(lens)
    T, H, D = sum(lens), 2, 8
    q, k, v = (rng.standard_normal((T, H, D)) for _ in range(3))
    O, LSE = oracle.attention(q, k, v, "causal", cu)
    for b, n in enumerate(lens):
        s = slice(cu[b], cu[b + 1])
        Ob, Lb = oracle.attention(q[s], k[s], v[s], "causal", np.array([0, n]))
        assert np.array_equal(O[s], Ob) and np.array_equal(LSE[:, s], Lb)


def test_predicate_truth_tables():
    text = "\n".join(l for l in open(os.path.join(GOLDEN, "predicate_tables.txt"))
                     .read().splitlines() if not l.startswith("#"))
    blocks = text.split("table ")[1:]
    seen = set()
    for blk in blocks:
        lines = [l.split() for l in blk.strip().splitlines() if l.strip() and not l.startswith("#")]
        kind = lines[0][0]
        meta, rows = {"role_think": 1}, []
        for toks in lines[1:]:
            if toks[0] in ("seg", "turn"):
                meta[toks[0]] = np.array(toks[1:], np.int32)
            elif toks[0] == "role":
                meta["role"] = np.array(toks[1:], np.int8)
            elif toks[0] == "len":
                pass
            elif toks[0] == "words":
                meta["dense_bits"] = np.array([int(x, 16) for x in toks[1:]], np.uint32)
                meta["dense_offsets"] = np.array([0, len(toks) - 1], np.int64)
            else:
                rows.append([int(x) for x in toks])
        want = np.array(rows, bool)
        L = want.shape[0]
        got = oracle.sequence_mask(kind, np.array([0, L]), 0, meta)
        assert np.array_equal(got, want), kind
        seen.add(kind)
    assert seen == set(oracle.KINDS)


# ----------------------------------------------------------------------------
# Tile labels and counts: closed forms derived from the workload structure.
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("L", [1, 2, 127, 128, 129, 255, 256, 257, 300, 513])
def test_causal_tile_labels_closed_form(L):
    lab = oracle.tile_labels("causal", np.array([0, L]))[0]
    n = -(-L // 128)
    for a in range(n):
        for b in range(n):
            if b > a:
                want = oracle.EMPTY
            elif b < a:
                want = oracle.FULL
            else:
                rows = min(128, L - 128 * a)
                want = oracle.FULL if rows == 1 else oracle.PARTIAL
            assert lab[a, b] == want


def test_shared_prefix_workload_counts_closed_form():
    w = W.make_workload(3, tensors=False)
    P, n, s = 2048, 16, 512
    tp, ts = P // 128, s // 128
    full = tp * (tp - 1) // 2 + n * (tp * ts + ts * (ts - 1) // 2)
    partial = tp + n * ts
    ntiles = (P + n * s) // 128
    lab = oracle.tile_labels(w.kind, w.cu_seqlens, w.meta())
    assert oracle.label_totals(lab) == (full, partial, ntiles * ntiles - full - partial)
    assert (full, partial) == (1240, 80)
    nnz = P * (P + 1) // 2 + n * (s * P + s * (s + 1) // 2)
    assert oracle.unmasked_pairs(w.kind, w.cu_seqlens, w.meta()) == nnz == 20_976_640


def test_strip_thinking_workload_counts_closed_form():
    w = W.make_workload(4, tensors=False)
    nturn, u, th, a = 8, 128, 768, 256
    per = (u + th + a) // 128                       # 9 tiles per turn
    own_full = per * (per - 1) // 2                 # strictly-lower tiles of a turn
    hist_full = per * ((u + a) // 128)              # q-tiles x (user + answer) tiles of an earlier turn
    full = nturn * own_full + hist_full * sum(range(nturn))
    partial = nturn * per
    nt = nturn * per
    lab = oracle.tile_labels(w.kind, w.cu_seqlens, w.meta())
    assert oracle.label_totals(lab) == (full, partial, nt * nt - full - partial)
    assert (full, partial) == (1044, 72)
    L = u + th + a
    nnz = nturn * L * (L + 1) // 2 + L * (u + a) * sum(range(nturn))
    assert oracle.unmasked_pairs(w.kind, w.cu_seqlens, w.meta()) == nnz == 17_699_328


def test_generic_workload_counts_closed_form():
    """Workload 7 (no mask inside a sequence) sees L^2 pairs per sequence;
    workload 8 (causal + document + padding, dense) sees m (m + 1) / 2 per
    document of m non-padding tokens, and its padding rows see nothing."""
    w7 = W.make_workload(7, tensors=False)
    assert w7.seqlens == W.make_workload(2, tensors=False).seqlens
    assert oracle.unmasked_pairs(w7.kind, w7.cu_seqlens) == sum(L * L for L in w7.seqlens) == 16_334_146
    lab7 = oracle.tile_labels("none", w7.cu_seqlens)
    assert all((l == oracle.FULL).all() for l in lab7)
    w5 = W.make_workload(5, tensors=False)
    seg = w5.seg.copy()
    seg[-2048:] = -1
    m = np.bincount(seg[seg >= 0])
    want = int((m * (m + 1) // 2).sum())
    assert want == 53_960_250
    w8 = W.make_workload(8, tensors=False)
    rows = oracle.sequence_mask("dense", w8.cu_seqlens, 0, w8.meta(), rows=np.arange(30000, 32768, 7))
    assert not rows[np.arange(30000, 32768, 7) >= 32768 - 2048].any()


def test_varlen_and_document_workload_counts_closed_form():
    w2 = W.make_workload(2, tensors=False)
    assert w2.seqlens == [860, 289, 1664, 1816, 272, 1814, 1638, 1843]
    lab2 = oracle.tile_labels("causal", w2.cu_seqlens)
    nts = [-(-L // 128) for L in w2.seqlens]
    ones = sum(1 for L in w2.seqlens if L % 128 == 1)   # a 1x1 diagonal tile is FULL
    f = sum(n * (n - 1) // 2 for n in nts) + ones
    p = sum(nts) - ones
    assert oracle.label_totals(lab2) == (f, p, sum(n * n for n in nts) - f - p) == (498, 84, 498)
    assert oracle.unmasked_pairs("causal", w2.cu_seqlens) == sum(L * (L + 1) // 2 for L in w2.seqlens)

    w5 = W.make_workload(5, tensors=False, document_form="cu_seqlens")
    w5d = W.make_workload(5, tensors=False, document_form="mask")
    nnz = sum(L * (L + 1) // 2 for L in w5.seqlens)
    assert nnz == 67_979_834
    assert oracle.unmasked_pairs(w5.kind, w5.cu_seqlens) == nnz
    assert oracle.unmasked_pairs(w5d.kind, w5d.cu_seqlens, w5d.meta()) == nnz
    nts = [-(-L // 128) for L in w5.seqlens]
    f = sum(n * (n - 1) // 2 for n in nts)
    assert oracle.label_totals(oracle.tile_labels("causal", w5.cu_seqlens)) == (f, sum(nts), f)


def test_document_form_labels_match_interval_reasoning():
    """For documents that are contiguous runs, a global tile pair is EMPTY iff no
    (q, k) pair is both causal and inside one document; checked by interval
    arithmetic on the document spans instead of counting the mask."""
    w = W.make_workload(5, tensors=False)
    lab = oracle.tile_labels(w.kind, w.cu_seqlens, w.meta())[0]
    bounds = np.concatenate([[0], np.cumsum(W.make_workload(5, tensors=False,
                                                           document_form="cu_seqlens").seqlens)])
    nt = lab.shape[0]
    for a in range(nt):
        q0, q1 = 128 * a, 128 * a + 127
        for b in range(nt):
            k0, k1 = 128 * b, 128 * b + 127
            any_vis = False
            all_vis = True
            for d in range(len(bounds) - 1):
                s, e = bounds[d], bounds[d + 1] - 1
                qa, qb = max(q0, s), min(q1, e)
                ka, kb = max(k0, s), min(k1, e)
                if qa <= qb and ka <= kb and ka <= qb:
                    any_vis = True
            # FULL iff every q row and k column share one document and k1 <= q0
            docs_q = set(np.searchsorted(bounds, [q0, q1], side="right"))
            docs_k = set(np.searchsorted(bounds, [k0, k1], side="right"))
            all_vis = k1 <= q0 and len(docs_q | docs_k) == 1
            want = oracle.FULL if all_vis else (oracle.PARTIAL if any_vis else oracle.EMPTY)
            assert lab[a, b] == want, (a, b)


def test_block_lists_and_lpt_order():
    lab = oracle.tile_labels("causal", np.array([0, 300, 300, 301]))
    bl = oracle.block_lists(lab)
    assert bl["qt_seq"].tolist() == [0, 0, 0, 2]
    assert bl["kcount"].tolist() == [1, 2, 3, 1]
    assert bl["kidx"].tolist() == [0, 0, 1, 0, 1, 2, 0]
    assert bl["klabel"].tolist() == [1, 2, 1, 2, 2, 1, 2]
    assert oracle.lpt_order(bl["kcount"]).tolist() == [2, 1, 0, 3]


# ----------------------------------------------------------------------------
# Planted mistakes: each plausible slip in the oracle must fail a pin above.
# ----------------------------------------------------------------------------

def _pins_pass():
    try:
        test_causal_4x4_matches_page_table()
        test_causal_row0_is_v0_and_lse_is_s00()
        test_predicate_truth_tables()
        test_shared_prefix_equals_separate_runs()
        test_strip_thinking_equals_per_turn_recomputation()
        test_strip_thinking_dup_equals_inference_contexts()
        test_wrong_task_max_diff_matches_page()
        test_none_kind_reproduces_the_pages_wrong_task_numbers()
        test_dense_causal_document_padding_equals_the_tokens_without_padding()
    except AssertionError:
        return False
    return True


def test_pins_pass_on_the_real_oracle():
    assert _pins_pass()


@pytest.mark.parametrize("mutant", ["strict_diagonal", "prefix_drops_seg0", "think_le_turn",
                                    "no_scale", "transposed_scores", "dup_history_sees_think",
                                    "dup_later_sees_answer", "dense_msb_first", "none_is_causal"])
def test_pins_catch_planted_mistakes(monkeypatch, mutant):
    real_pred, real_attn = oa.predicate, oa.masked_attention

    def pred(kind, qi, ki, seg=None, role=None, turn=None, role_think=1):
        qi, ki = np.asarray(qi), np.asarray(ki)
        if mutant == "strict_diagonal":
            c = qi > ki
            return c if kind == "causal" else c & real_pred(kind, qi, ki, seg, role, turn, role_think)
        if mutant == "prefix_drops_seg0" and kind == "shared_prefix":
            return (qi >= ki) & (seg[ki] == seg[qi])
        if mutant == "think_le_turn" and kind == "strip_thinking":
            return (qi >= ki) & ~((role[ki] == role_think) & (turn[ki] <= turn[qi]))
        if kind == "strip_thinking_dup" and mutant.startswith("dup_"):
            base = real_pred(kind, qi, ki, seg, role, turn, role_think)
            same, causal = turn[ki] == turn[qi], qi >= ki
            if mutant == "dup_history_sees_think":
                return base | (causal & same & (role[ki] == role_think) & (role[qi] == W.ROLE_ANSWER_HISTORY))
            return base | (causal & (turn[ki] < turn[qi]) & (role[ki] == W.ROLE_ANSWER))
        return real_pred(kind, qi, ki, seg, role, turn, role_think)

    def attn(q, k, v, mask, scale):
        if mutant == "no_scale":
            return real_attn(q, k, v, mask, 1.0)
        if mutant == "transposed_scores":
            q2 = np.asarray(q, float)
            if q2.shape[0] == np.asarray(k).shape[0]:
                # scores k q^T instead of q k^T
                return real_attn(k, q, v, mask, scale)
        return real_attn(q, k, v, mask, scale)

    real_bits, real_visible = oa.dense_bits, oa.visible

    def bits(meta, cu_seqlens, b, rows, cols):
        if mutant == "dense_msb_first":
            cols = np.asarray(cols, np.int64)
            return real_bits(meta, cu_seqlens, b, rows, (cols // 32) * 32 + 31 - cols % 32)
        return real_bits(meta, cu_seqlens, b, rows, cols)

    def vis(kind, cu_seqlens, b, meta, rows, cols):
        if mutant == "none_is_causal" and kind == "none":
            return np.asarray(cols)[None, :] <= np.asarray(rows)[:, None]
        return real_visible(kind, cu_seqlens, b, meta, rows, cols)

    monkeypatch.setattr(oa, "dense_bits", bits)
    monkeypatch.setattr(oa, "visible", vis)
    monkeypatch.setattr(oa, "predicate", pred)
    monkeypatch.setattr(oa, "masked_attention", attn)
    monkeypatch.setattr(oracle, "masked_attention", attn)
    assert not _pins_pass()


# ----------------------------------------------------------------------------
# Backward (dQ, dK, dV).  The oracle is the chain rule through the forward;
# pinned against torch autograd in fp64, finite differences, and invariants.
# ----------------------------------------------------------------------------

def _bwd_case(kind, seed=21, lens=(70, 1, 33, 150), H=2, D=16):
    rng = np.random.default_rng(seed)
    lens = list(lens)
    meta = W.random_meta(rng, kind, lens)
    cu = W._cu(lens)
    T = sum(lens)
    g = torch.Generator().manual_seed(seed)
    q, k, v, do = (torch.randn(T, H, D, dtype=torch.float64, generator=g) for _ in range(4))
    return cu, meta, q, k, v, do


def _autograd_grads(kind, cu, meta, q, k, v, do, scale):
    T, H, D = q.shape
    dq, dk, dv = (np.zeros((T, H, D)) for _ in range(3))
    for b in range(len(cu) - 1):
        s0, s1 = int(cu[b]), int(cu[b + 1])
        if s1 == s0:
            continue
        mask = torch.from_numpy(oracle.sequence_mask(kind, cu, b, meta))
        for h in range(H):
            qh, kh, vh = (t[s0:s1, h].clone().requires_grad_(True) for t in (q, k, v))
            o = torch.nn.functional.scaled_dot_product_attention(
                qh[None], kh[None], vh[None], attn_mask=mask[None], scale=scale)[0]
            o.backward(do[s0:s1, h])
            dq[s0:s1, h], dk[s0:s1, h], dv[s0:s1, h] = qh.grad.numpy(), kh.grad.numpy(), vh.grad.numpy()
    return dq, dk, dv


@pytest.mark.parametrize("kind", oracle.KINDS)
def test_backward_matches_torch_autograd_fp64(kind):
    """The backward reduces to a library routine: torch autograd through fp64
    SDPA with a boolean mask."""
    cu, meta, q, k, v, do = _bwd_case(kind)
    scale = 1 / math.sqrt(q.shape[2])
    got = oracle.attention_backward(q, k, v, do, kind, cu, meta)
    want = _autograd_grads(kind, cu, meta, q, k, v, do, scale)
    for g_, w_ in zip(got, want):
        assert np.abs(g_ - w_).max() < 1e-11


@pytest.mark.parametrize("kind", oracle.KINDS)
def test_sampled_backward_matches_torch_autograd_fp64(kind):
    """The row/column-sampled backward (used on sequences too long for the whole
    L x L backward) equals torch autograd through fp64 SDPA on the sampled rows,
    including rows of empty and single-token sequences and tile edges."""
    cu, meta, q, k, v, do = _bwd_case(kind, seed=33, lens=(150, 0, 1, 300))
    scale = 1 / math.sqrt(q.shape[2])
    want = _autograd_grads(kind, cu, meta, q, k, v, do, scale)
    rows = [0, 5, 127, 128, 149, 150, 151, 280, 450]
    dq, dk, dv = oracle.attention_backward_sampled(q, k, v, do, kind, cu, meta, q_rows=rows,
                                                   k_rows=rows[::-1], row_block=64)
    for got, ref in ((dq, want[0]), (dk, want[1]), (dv, want[2])):
        assert np.abs(got[rows] - ref[rows]).max() < 1e-11
        others = np.setdiff1d(np.arange(q.shape[0]), rows)
        assert np.isnan(got[others]).all()


def test_backward_matches_finite_differences():
    """Central differences of sum(O * dO) on a tiny causal case."""
    rng = np.random.default_rng(3)
    L, D, scale = 5, 3, 0.7
    q, k, v, do = (rng.standard_normal((L, D)) for _ in range(4))
    mask = oracle.sequence_mask("causal", np.array([0, L]), 0, {})
    dq, dk, dv = oracle.masked_attention_backward(q, k, v, do, mask, scale)

    def loss(q_, k_, v_):
        return float((oracle.masked_attention(q_, k_, v_, mask, scale)[0] * do).sum())

    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            num[idx] = (loss(**{k2 + "_": a for k2, a in args_p.items()}) -
                        loss(**{k2 + "_": a for k2, a in args_m.items()})) / (2 * eps)
        assert np.abs(num - g).max() < 1e-7, name


@pytest.mark.parametrize("kind", oracle.KINDS)
def test_backward_invariants(kind):
    """Per sequence and head: the rows of dS sum to zero, so the keys' dK sum to
    zero; the keys' dV sum to the dO of rows that see any key."""
    cu, meta, q, k, v, do = _bwd_case(kind, seed=5)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, kind, cu, meta)
    for b in range(len(cu) - 1):
        s0, s1 = int(cu[b]), int(cu[b + 1])
        if s1 == s0:
            continue
        seen = oracle.sequence_mask(kind, cu, b, meta).any(axis=1)
        for h in range(q.shape[1]):
            assert np.abs(dk[s0:s1, h].sum(axis=0)).max() < 1e-10
            want = do[s0:s1, h].numpy()[seen].sum(axis=0)
            assert np.abs(dv[s0:s1, h].sum(axis=0) - want).max() < 1e-10


def test_transposed_lists_are_the_transpose():
    lens = np.array([0, 300, 300, 301, 700])
    for kind, meta in (("causal", {}),):
        lab = oracle.tile_labels(kind, lens, meta)
        fwd = oracle.block_lists(lab)
        bwd = oracle.block_lists_transposed(lab)
        pairs_f = set()
        for g in range(len(fwd["kcount"])):
            for e in range(fwd["koff"][g], fwd["koff"][g + 1]):
                pairs_f.add((int(fwd["qt_seq"][g]), int(fwd["qt_idx"][g]), int(fwd["kidx"][e]), int(fwd["klabel"][e])))
        pairs_b = set()
        col = 0
        for b, l_ in enumerate(lab):
            for kt in range(l_.shape[1]):
                for e in range(bwd["qoff"][col], bwd["qoff"][col + 1]):
                    pairs_b.add((b, int(bwd["qidx"][e]), kt, int(bwd["qlabel"][e])))
                col += 1
        assert pairs_f == pairs_b
    # a causal 300-token sequence: k-tile 0 is seen by q-tiles 0 (PARTIAL), 1, 2 (FULL)
    bwd = oracle.block_lists_transposed(oracle.tile_labels("causal", np.array([0, 300])))
    assert bwd["qcount"].tolist() == [3, 2, 1]
    assert bwd["qidx"].tolist() == [0, 1, 2, 1, 2, 2]
    assert bwd["qlabel"].tolist() == [1, 2, 2, 1, 2, 1]


def _bwd_pins_pass(bwd):
    try:
        for kind in ("causal", "shared_prefix"):
            cu, meta, q, k, v, do = _bwd_case(kind, lens=(40, 17))
            mask_fn = lambda b: oracle.sequence_mask(kind, cu, b, meta)
            scale = 1 / math.sqrt(q.shape[2])
            want = _autograd_grads(kind, cu, meta, q, k, v, do, scale)
            for b in range(len(cu) - 1):
                s0, s1 = int(cu[b]), int(cu[b + 1])
                for h in range(q.shape[1]):
                    got = bwd(q[s0:s1, h].numpy(), k[s0:s1, h].numpy(), v[s0:s1, h].numpy(),
                              do[s0:s1, h].numpy(), mask_fn(b), scale)
                    for g_, w_ in zip(got, want):
                        assert np.abs(g_ - w_[s0:s1, h]).max() < 1e-11
    except AssertionError:
        return False
    return True


@pytest.mark.parametrize("mutant", ["drop_delta", "dq_no_scale", "dk_untransposed", "dv_from_dp"])
def test_backward_pins_catch_planted_mistakes(mutant):
    real = oracle.masked_attention_backward
    assert _bwd_pins_pass(real)

    def bad(q, k, v, do, mask, scale):
        dq, dk, dv = real(q, k, v, do, mask, scale)
        s = np.where(mask, (q @ k.T) * scale, -np.inf)
        m = np.where(np.isfinite(s.max(1)), s.max(1), 0)
        p = np.where(mask, np.exp(s - m[:, None]), 0)
        p = p / np.maximum(p.sum(1, keepdims=True), 1e-300)
        dp = do @ v.T
        if mutant == "drop_delta":
            ds = p * dp
            return (ds @ k) * scale, (ds.T @ q) * scale, dv
        if mutant == "dq_no_scale":
            return dq / scale, dk, dv
        if mutant == "dk_untransposed":
            ds = p * (dp - (do * (p @ v)).sum(1)[:, None])
            return dq, (ds @ q) * scale if ds.shape[0] == ds.shape[1] else dk * 0, dv
        if mutant == "dv_from_dp":
            return dq, dk, dp.T @ do
        return dq, dk, dv

    assert not _bwd_pins_pass(bad)
