"""GPU block-mask builder vs the oracle's brute-force labels: bit-exact.

Labels, per-q-tile compacted lists, q-tile descriptors, pair totals, the
longest-first orders and the transposed (k-major) lists must equal what
counting the materialised mask gives.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_masked_mask_gb300 import api
from block_sparse_masked_mask_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def build_on_gpu(w):
    dm = w.device_meta()
    bm = api.attn_block_mask_build(w.kind, dm["cu_seqlens"], w.total_tokens, w.max_seqlen,
                                   **w.api_kwargs(dm))
    assert api.attn_get_status(bm) == api.ATTN_OK
    return bm


def assert_matches_oracle(w, bm):
    labels = oracle.tile_labels(w.kind, w.cu_seqlens, w.meta())
    want = oracle.block_lists(labels)
    got = bm.lists()
    n = len(want["kcount"])
    assert int(got["header"][0]) == n
    assert np.array_equal(got["qt_seq"].numpy(), want["qt_seq"])
    assert np.array_equal(got["qt_idx"].numpy(), want["qt_idx"])
    for g in range(n):
        lab = labels[want["qt_seq"][g]][want["qt_idx"][g]]
        assert np.array_equal(got["labels"][g, :len(lab)].numpy(), lab), f"q-tile {g}"
    assert np.array_equal(got["kcount"].numpy(), want["kcount"])
    assert np.array_equal(got["koff"].numpy(), want["koff"])
    assert np.array_equal(got["kidx"].numpy(), want["kidx"])
    assert np.array_equal(got["klabel"].numpy(), want["klabel"])
    assert np.array_equal(got["order"].numpy(), oracle.lpt_order(want["kcount"]))
    f, p, e = oracle.label_totals(labels)
    assert got["header"][4:7].tolist() == [e, p, f]
    assert int(got["header"][1]) == int(want["koff"][-1])
    # q-tile pairs: tiles (2j, 2j+1) of one sequence, ordered by summed work
    q0 = [g for g in range(n) if want["qt_idx"][g] % 2 == 0]
    assert int(got["header"][3]) == len(q0)
    assert got["pair_q0"].tolist() == q0
    work = [int(want["kcount"][g]) + (int(want["kcount"][g + 1])
            if g + 1 < n and want["qt_seq"][g + 1] == want["qt_seq"][g] else 0) for g in q0]
    assert got["pair_order"].tolist() == oracle.lpt_order(work).tolist()
    # transposed (k-major) lists for the backward, and the k-tiles' order
    wt = oracle.block_lists_transposed(labels)
    assert np.array_equal(got["qcount"].numpy(), wt["qcount"])
    assert np.array_equal(got["qoff"].numpy(), wt["qoff"])
    assert np.array_equal(got["qidx"].numpy(), wt["qidx"])
    assert np.array_equal(got["qlabel"].numpy(), wt["qlabel"])
    assert np.array_equal(got["korder"].numpy(), oracle.lpt_order(wt["qcount"]))


@pytest.mark.parametrize("c", [1, 2, 3, 4, 5, 6, 7, 8])
def test_workload_masks_bit_exact(c):
    w = W.make_workload(c, tensors=False)
    assert_matches_oracle(w, build_on_gpu(w))


def test_document_workload_cu_seqlens_form_bit_exact():
    w = W.make_workload(5, tensors=False, document_form="cu_seqlens")
    assert_matches_oracle(w, build_on_gpu(w))


LENGTH_SETS = [
    [1], [127], [128], [129], [300, 1, 129, 517, 0, 128], [700, 255, 256, 257],
    [0, 0, 5], [1000, 3, 999],
]


@pytest.mark.parametrize("kind", oracle.KINDS)
@pytest.mark.parametrize("li", range(len(LENGTH_SETS)))
def test_random_metadata_bit_exact(kind, li):
    for seed in range(3):
        rng = np.random.default_rng(1000 * li + seed)
        lens = LENGTH_SETS[li]
        m = W.random_meta(rng, kind, lens)
        w = W.Workload(f"rand_{kind}", kind, W._cu(lens), 1, 128, torch.bfloat16,
                       seg=m["seg"], role=m["role"], turn=m["turn"], dense_bits=m["dense_bits"],
                       dense_offsets=m["dense_offsets"])
        assert_matches_oracle(w, build_on_gpu(w))


def test_large_random_documents_bit_exact():
    rng = np.random.default_rng(77)
    lens = [4096 + 333, 2000]
    seg, _, _ = W.random_metadata(rng, "causal_document", lens)
    w = W.Workload("rand_doc_big", "causal_document", W._cu(lens), 1, 128, torch.bfloat16, seg=seg)
    assert_matches_oracle(w, build_on_gpu(w))


def test_role_think_code_is_a_parameter():
    role, turn = W.strip_thinking_layout([(40, 200, 60)] * 3)
    role = np.where(role == W.ROLE_THINK, 7, role).astype(np.int8)
    w = W.Workload("think7", "strip_thinking", W._cu([len(role)]), 1, 128, torch.bfloat16,
                   role=role, turn=turn, role_think=7)
    assert_matches_oracle(w, build_on_gpu(w))


@pytest.mark.parametrize("cu,maxlen", [
    ([1, 10, 20], 64),      # does not start at 0
    ([0, 30, 20], 64),      # decreasing
    ([0, 10, 200], 64),     # a sequence longer than max_seqlen
])
def test_malformed_cu_seqlens_reported_by_device(cu, maxlen):
    cu_t = torch.tensor(cu, dtype=torch.int32, device="cuda")
    T = 20 if cu[1] > cu[2] else cu[-1]
    bm = api.attn_block_mask_build("causal", cu_t, T, maxlen)
    assert api.attn_get_status(bm) == 7
    assert bm.n_qtiles == 0


def test_last_entry_must_equal_total_tokens():
    cu_t = torch.tensor([0, 10, 20], dtype=torch.int32, device="cuda")
    bm = api.attn_block_mask_build("causal", cu_t, 25, 64)
    assert api.attn_get_status(bm) == 7


@pytest.mark.parametrize("kind", ["causal_document", "shared_prefix", "strip_thinking",
                                  "strip_thinking_dup"])
@pytest.mark.parametrize("li", [4, 5, 7])
def test_random_metadata_repeating_ids_bit_exact(kind, li):
    """Ids drawn from a small alphabet (they repeat, fall and skip), so the
    classifier's interval reasoning meets tiles whose id ranges overlap
    without sharing ids."""
    for seed in range(3):
        rng = np.random.default_rng(7000 + 100 * li + seed)
        lens = LENGTH_SETS[li]
        seg, role, turn = W.random_metadata(rng, kind, lens, id_alphabet=4)
        w = W.Workload(f"rand_ids_{kind}", kind, W._cu(lens), 1, 128, torch.bfloat16,
                       seg=seg, role=role, turn=turn)
        assert_matches_oracle(w, build_on_gpu(w))
