"""Head-sharded (Ulysses) structured-mask attention over the ranks of a group.

The xorl issue ("Block-mask attention: shared-prefix and strip-thinking
multi-turn training that cu_seqlens cannot express", Open constraints, CP/SP
bullet) asks that a block mask shard consistently with sequence parallelism,
and notes that Ulysses, which shards heads, is the tractable case: the mask
depends only on token metadata, never on the head, so every rank can hold the
whole mask while attending over a slice of the heads.

Layout.  The packed batch (total_tokens T, H heads) is cut into g contiguous
token shards, one per rank of the group (``token_splits``); rank r holds
Q, K, V (and dO) rows [start_r, end_r) of every head, plus the matching
slice of the per-token metadata (seg_id, role, turn).  cu_seqlens, and for
the DENSE kind the bit rows and offsets, are global and given on every rank.
H must be a multiple of g; rank r attends over heads [r H/g, (r+1) H/g).

Forward (``ulysses_attn_fwd``):
  1. all-gather the per-token metadata, so every rank builds the same block
     mask of the whole batch (``attn_block_mask_build``, on the device);
  2. all-to-all Q, K, V from token shards [T_r, H, D] to head groups
     [T, H/g, D] (``seq_to_heads``);
  3. ``attn_fwd`` over the H/g heads with the whole mask;
  4. all-to-all O back to [T_r, H, D] and LSE back to [H, T_r]
     (``heads_to_seq``).
Backward (``ulysses_attn_bwd``): dO goes through step 2, ``attn_bwd`` runs on
the head group with the forward's head-sharded O and LSE, and dQ, dK, dV go
through step 4.

The exchanges are torch.distributed collectives (NCCL on GPUs, gloo on the
CPU), moved as raw bytes so any element type passes; no kernel reads another
rank's memory, and every attention step is the library's own CUDA call.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional

import torch
import torch.distributed as dist

from . import api


def token_splits(total_tokens: int, world: int) -> List[int]:
    """Contiguous shard sizes: the first ``total_tokens % world`` ranks hold one
    token more than the others."""
    base, extra = divmod(int(total_tokens), int(world))
    return [base + (1 if r < extra else 0) for r in range(world)]


def _group_info(group):
    return dist.get_world_size(group), dist.get_rank(group)


def _as_bytes(x: torch.Tensor, rows: int) -> torch.Tensor:
    """A contiguous tensor seen as ``rows`` rows of raw bytes."""
    return x.contiguous().view(torch.uint8).view(rows, -1)


def seq_to_heads(x: torch.Tensor, splits: List[int], group=None) -> torch.Tensor:
    """[T_r, H, D] (this rank's tokens, every head) -> [T, H/g, D] (every token,
    this rank's head group), by one all-to-all."""
    g, r = _group_info(group)
    T_r, H, D = x.shape
    if T_r != splits[r] or H % g:
        raise ValueError(f"seq_to_heads: shard {tuple(x.shape)} does not match splits {splits} "
                         f"and {g} ranks")
    Hg = H // g
    # head group j of this rank's tokens goes to rank j
    send = x.reshape(T_r, g, Hg, D).permute(1, 0, 2, 3).contiguous()
    send = _as_bytes(send, g * T_r)
    recv = torch.empty((sum(splits), send.shape[1]), dtype=torch.uint8, device=x.device)
    dist.all_to_all_single(recv, send, output_split_sizes=list(splits),
                           input_split_sizes=[T_r] * g, group=group)
    return recv.view(x.dtype).view(sum(splits), Hg, D)


def heads_to_seq(y: torch.Tensor, splits: List[int], group=None) -> torch.Tensor:
    """[T, H/g, D] (every token, this rank's head group) -> [T_r, H, D], the
    inverse of ``seq_to_heads``."""
    g, r = _group_info(group)
    T, Hg, D = y.shape
    if T != sum(splits):
        raise ValueError(f"heads_to_seq: {T} tokens, splits {splits}")
    T_r = splits[r]
    send = _as_bytes(y, T)
    recv = torch.empty((g * T_r, send.shape[1]), dtype=torch.uint8, device=y.device)
    dist.all_to_all_single(recv, send, output_split_sizes=[T_r] * g,
                           input_split_sizes=list(splits), group=group)
    # block j holds head group j of this rank's tokens
    x = recv.view(y.dtype).view(g, T_r, Hg, D).permute(1, 0, 2, 3)
    return x.reshape(T_r, g * Hg, D)


def lse_heads_to_seq(lse: torch.Tensor, splits: List[int], group=None) -> torch.Tensor:
    """LSE [H/g, T] of this rank's head group -> [H, T_r] of this rank's tokens."""
    Hg, T = lse.shape
    x = heads_to_seq(lse.t().contiguous().view(T, Hg, 1), splits, group)
    return x.view(x.shape[0], -1).t().contiguous()


def lse_seq_to_heads(lse: torch.Tensor, splits: List[int], group=None) -> torch.Tensor:
    """LSE [H, T_r] of this rank's tokens -> [H/g, T] of its head group."""
    H, T_r = lse.shape
    y = seq_to_heads(lse.t().contiguous().view(T_r, H, 1), splits, group)
    return y.view(y.shape[0], -1).t().contiguous()


def gather_tokens(x: Optional[torch.Tensor], splits: List[int], group=None) -> Optional[torch.Tensor]:
    """All-gather of a per-token array: this rank's [T_r, ...] -> [T, ...] in
    rank order (shards padded to the longest for the collective)."""
    if x is None:
        return None
    g, r = _group_info(group)
    if x.shape[0] != splits[r]:
        raise ValueError(f"gather_tokens: {x.shape[0]} rows, splits {splits}")
    tail = tuple(x.shape[1:])
    width = x.element_size()
    for n in tail:
        width *= int(n)
    m = max(splits)
    buf = torch.zeros((m, width), dtype=torch.uint8, device=x.device)
    if x.shape[0]:
        buf[: x.shape[0]] = _as_bytes(x, x.shape[0])
    parts = [torch.empty_like(buf) for _ in range(g)]
    dist.all_gather(parts, buf, group=group)
    full = torch.cat([p[:n] for p, n in zip(parts, splits)], dim=0).contiguous()
    return full.view(x.dtype).view((sum(splits),) + tail)


@dataclass
class UlyssesContext:
    """What the backward needs from the forward: the group, the split, the
    whole-batch block mask and metadata, and this rank's head-group tensors."""
    group: object
    splits: List[int]
    mask: api.BlockMask
    kind: object
    cu_seqlens: torch.Tensor
    max_seqlen: int
    meta: dict
    scale: float
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    o: torch.Tensor
    lse: torch.Tensor


def ulysses_attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, kind,
                     cu_seqlens: torch.Tensor, max_seqlen: int, seg_id=None, role=None, turn=None,
                     role_think: int = 1, scale: float = 0.0, dense_bits=None, dense_offsets=None,
                     group=None, splits: Optional[List[int]] = None, mask_workspace=None):
    """Masked attention forward over head-sharded ranks.

    q, k, v: this rank's token shard [T_r, H, D]; seg_id / role / turn: this
    rank's shard of the per-token metadata (or None when the kind needs none);
    cu_seqlens (device int32 [batch + 1]) and the DENSE kind's bits / offsets:
    global.  Returns (O [T_r, H, D], LSE [H, T_r] fp32, context for
    ``ulysses_attn_bwd``).  Every rank of ``group`` must call it with the same
    global arguments; ``splits`` (every rank's shard length, in rank order)
    saves one small all-gather when the caller knows it.
    """
    # the shards are contiguous in rank order; by default each rank's length is
    # whatever it holds (token_splits gives the usual near-equal cut)
    splits = _all_rows(q.shape[0], group) if splits is None else list(splits)
    meta = {"seg_id": gather_tokens(seg_id, splits, group), "role": gather_tokens(role, splits, group),
            "turn": gather_tokens(turn, splits, group)}
    T = sum(splits)
    bm = api.attn_block_mask_build(kind, cu_seqlens, T, max_seqlen, role_think=role_think,
                                   workspace=mask_workspace, dense_bits=dense_bits,
                                   dense_offsets=dense_offsets, **meta)
    qh, kh, vh = (seq_to_heads(x, splits, group) for x in (q, k, v))
    kw = dict(meta, role_think=role_think, dense_bits=dense_bits, dense_offsets=dense_offsets)
    oh, lh = api.attn_fwd(qh, kh, vh, bm, kind, cu_seqlens, max_seqlen, scale=scale, **kw)
    o = heads_to_seq(oh, splits, group)
    lse = lse_heads_to_seq(lh, splits, group)
    ctx = UlyssesContext(group, splits, bm, kind, cu_seqlens, max_seqlen, kw, scale, qh, kh, vh, oh, lh)
    return o, lse, ctx


def ulysses_attn_bwd(do: torch.Tensor, ctx: UlyssesContext, workspace=None):
    """Backward of ``ulysses_attn_fwd`` for this rank's upstream gradient shard
    dO [T_r, H, D]; returns this rank's (dQ, dK, dV) shards [T_r, H, D]."""
    doh = seq_to_heads(do, ctx.splits, ctx.group)
    dqh, dkh, dvh = api.attn_bwd(ctx.q, ctx.k, ctx.v, ctx.o, ctx.lse, doh, ctx.mask, ctx.kind,
                                 ctx.cu_seqlens, ctx.max_seqlen, scale=ctx.scale, workspace=workspace,
                                 **ctx.meta)
    return tuple(heads_to_seq(x, ctx.splits, ctx.group) for x in (dqh, dkh, dvh))


def _all_rows(n: int, group) -> List[int]:
    """Every rank's shard length (one small all-gather)."""
    g, _ = _group_info(group)
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    mine = torch.tensor([int(n)], dtype=torch.int64, device=dev)
    parts = [torch.empty_like(mine) for _ in range(g)]
    dist.all_gather(parts, mine, group=group)
    return [int(p.item()) for p in parts]
