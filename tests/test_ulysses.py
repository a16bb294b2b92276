"""Head-sharded (Ulysses) attention: the token/head layout exchanges and the
metadata all-gather, on two gloo ranks on the CPU, and the whole wrapper on
one GPU against the library's own single-rank calls.

xorl issue, Open constraints, CP/SP bullet: a block mask has to shard
consistently with sequence parallelism; Ulysses shards heads, and the mask
(head-independent) is built whole on every rank.  The CPU test checks every
exchange bit for bit against slices of the whole tensors, and runs the
exchange around the fp64 oracle (standing in, in this test only, for each
rank's attention on its head group) to show that the sharded pipeline gives
exactly the whole-batch result.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from block_sparse_masked_mask_gb300 import ulysses as U
from block_sparse_masked_mask_gb300 import workloads as W


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_token_splits_are_contiguous_and_near_equal():
    for T, g in [(10, 2), (11, 2), (7, 4), (3, 4), (32768, 8)]:
        s = U.token_splits(T, g)
        assert sum(s) == T and len(s) == g
        assert max(s) - min(s) <= 1 and s == sorted(s, reverse=True)


CASES = [("strip_thinking", [300, 129, 517], None),      # near-equal split
         ("shared_prefix", [700, 255], [880, 75])]        # a skewed split


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        out = []
        for ci, (kind, lens, split) in enumerate(CASES):
            w = W.random_workload(90 + ci, kind, lens, num_heads=4, head_dim=16)
            T, H, D = w.q.shape
            splits = U.token_splits(T, ws) if split is None else split
            a = sum(splits[:rank])
            b = a + splits[rank]
            Hg = H // ws
            hs = slice(rank * Hg, (rank + 1) * Hg)
            res = {}
            # Q/K/V: token shard -> head group and back, bit for bit
            qh = U.seq_to_heads(w.q[a:b], splits)
            res["seq_to_heads"] = torch.equal(qh, w.q[:, hs])
            res["round_trip"] = torch.equal(U.heads_to_seq(qh, splits), w.q[a:b])
            # LSE: [H/g, T] of the head group <-> [H, T_r] of the token shard
            lse = torch.randn(H, T, generator=torch.Generator().manual_seed(ci))
            res["lse_to_seq"] = torch.equal(U.lse_heads_to_seq(lse[hs].contiguous(), splits), lse[:, a:b])
            res["lse_to_heads"] = torch.equal(U.lse_seq_to_heads(lse[:, a:b].contiguous(), splits), lse[hs])
            # per-token metadata: every rank ends with the whole arrays
            meta = {"seg": w.seg, "role": w.role, "turn": w.turn}
            for name, arr in meta.items():
                if arr is None:
                    continue
                full = torch.from_numpy(np.ascontiguousarray(arr))
                res[f"gather_{name}"] = torch.equal(U.gather_tokens(full[a:b].contiguous(), splits), full)
            # the default split is each rank's own shard length
            res["rows"] = U._all_rows(b - a, None) == list(splits)
            # the exchange around a per-head-group attention gives the whole-batch
            # result: the oracle stands in for each rank's attention
            kh, vh = U.seq_to_heads(w.k[a:b], splits), U.seq_to_heads(w.v[a:b], splits)
            gmeta = dict(w.meta())
            for name in ("seg", "role", "turn"):
                if gmeta[name] is not None:
                    t = torch.from_numpy(np.ascontiguousarray(gmeta[name]))
                    gmeta[name] = U.gather_tokens(t[a:b].contiguous(), splits).numpy()
            Oh, Lh = oracle.attention(qh, kh, vh, kind, w.cu_seqlens, gmeta)
            O = U.heads_to_seq(torch.from_numpy(Oh), splits)
            L = U.lse_heads_to_seq(torch.from_numpy(Lh), splits)
            Ofull, Lfull = oracle.attention(w.q, w.k, w.v, kind, w.cu_seqlens, w.meta())
            res["oracle_O"] = np.array_equal(O.numpy(), Ofull[a:b])
            res["oracle_LSE"] = np.array_equal(L.numpy(), Lfull[:, a:b])
            out.append(res)
        q.put((rank, out))
    finally:
        dist.destroy_process_group()


def test_exchanges_on_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=300) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, out in results:
        for ci, res in enumerate(out):
            bad = [k for k, ok in res.items() if not ok]
            assert not bad, f"rank {rank}, case {CASES[ci][0]}: {bad}"


@pytest.mark.gpu
def test_wrapper_on_one_rank_equals_the_library_calls():
    """On a group of one the exchanges are copies: the wrapper's O, LSE and
    gradients equal attn_fwd / attn_bwd on the same inputs bit for bit."""
    from block_sparse_masked_mask_gb300 import api
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0,
                            world_size=1)
    try:
        w = W.random_workload(95, "strip_thinking", [700, 255, 1000], num_heads=4, head_dim=128)
        dm = w.device_meta()
        kw = w.api_kwargs(dm)
        q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
        do = W.grad_output(w, seed=95).cuda()
        bm = api.attn_block_mask_build(w.kind, dm["cu_seqlens"], w.total_tokens, w.max_seqlen, **kw)
        o_ref, l_ref = api.attn_fwd(q, k, v, bm, w.kind, dm["cu_seqlens"], w.max_seqlen, **kw)
        g_ref = api.attn_bwd(q, k, v, o_ref, l_ref, do, bm, w.kind, dm["cu_seqlens"], w.max_seqlen, **kw)
        o, lse, ctx = U.ulysses_attn_fwd(q, k, v, w.kind, dm["cu_seqlens"], w.max_seqlen, **kw)
        grads = U.ulysses_attn_bwd(do, ctx)
        assert api.attn_get_status(ctx.mask) == api.ATTN_OK
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
        for x, y in zip(grads, g_ref):
            assert torch.equal(x, y)
    finally:
        dist.destroy_process_group()
