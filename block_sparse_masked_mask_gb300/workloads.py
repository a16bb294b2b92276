"""Seeded synthetic inputs for the structured-mask attention forward.

This module generates data: sequence lengths, per-token segment / role / turn
metadata and random Q, K, V.  It holds none of the method's arithmetic (no
softmax, no tiling, no tile classification), so both the CUDA path and the
fp64 oracle can be fed from it without sharing any code that computes a
result.  One generator composes a mask itself: the DENSE kind's input bits of
workload 8 (``causal_document_padding_bits``), which a caller of that kind
supplies by definition.  The library only reads those bits; the oracle pins
the composition independently (its causal + document + padding equals the
sequence with the padding removed).

The six workloads follow the shapes the block-mask pages describe:

* ``causal_s64_d32_fp32`` - one causal sequence, S=64, H=1, D=32, fp32
  ("Triton from first principles" Ch. 21, Section 21.2, which checks causal
  flash attention at toy sizes).
* ``varlen_causal_8seq`` - eight packed sequences of seeded lengths in
  [128, 2048], causal inside each, nothing across (the cu_seqlens packing of
  the xorl issue "Block-mask attention: shared-prefix and strip-thinking",
  Summary).
* ``shared_prefix_2048_16x512`` - a 2048-token prefix (segment 0) and sixteen
  512-token suffixes (segments 1..16) (same issue, Mask specifications,
  "Shared prefix").
* ``strip_thinking_8turns`` - eight turns of user 128 / think 768 / answer
  256 tokens, roles USER=0, THINK=1, ANSWER=2, turns numbered from 1 (same
  issue, "Strip-thinking multi-turn").
* ``causal_document_32k`` - 32768 tokens cut into twelve documents of seeded
  lengths (each at least 512), causal inside a document and block-diagonal
  across (the issue's "Move document boundaries into the mask" decision).
* ``strip_thinking_dup_8turns`` - the strip-thinking conversation with each
  answer span followed by its history copy (ANSWER_HISTORY=3): user 128 /
  think 768 / answer 256 / history 256 per turn, 11264 tokens (same issue,
  "The exactness question", option (b), token duplication).

Generation recipe (per workload number ``c`` = 1..6): a CPU
``torch.Generator`` seeded with ``c``; metadata lengths are drawn first, then
Q, K and V, each ``torch.randn((T, H, D)) * sigma`` in fp32, then cast to the
workload dtype.  The inputs are synthetic stand-ins: the pages measure on
private training data that is not reproduced here.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

ROLE_USER = 0
ROLE_THINK = 1
ROLE_ANSWER = 2
ROLE_ANSWER_HISTORY = 3  # the duplicated answer copy later turns attend


@dataclasses.dataclass
class Workload:
    name: str
    kind: str                      # "causal" | "causal_document" | "shared_prefix" | "strip_thinking"
    cu_seqlens: np.ndarray         # int32 [B+1]
    num_heads: int
    head_dim: int
    dtype: torch.dtype
    sigma: float = 1.0
    seg: Optional[np.ndarray] = None    # int32 [T]
    role: Optional[np.ndarray] = None   # int8  [T]
    turn: Optional[np.ndarray] = None   # int32 [T]
    dense_bits: Optional[np.ndarray] = None     # uint32, the "dense" kind's bit rows
    dense_offsets: Optional[np.ndarray] = None  # int64 [B+1], first word of each sequence
    role_think: int = ROLE_THINK
    seed: int = 0
    q: Optional[torch.Tensor] = None    # [T, H, D] on CPU, workload dtype
    k: Optional[torch.Tensor] = None
    v: Optional[torch.Tensor] = None

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def batch(self) -> int:
        return len(self.cu_seqlens) - 1

    @property
    def max_seqlen(self) -> int:
        lens = np.diff(self.cu_seqlens)
        return int(lens.max()) if len(lens) else 0

    @property
    def seqlens(self) -> list:
        return [int(x) for x in np.diff(self.cu_seqlens)]

    def meta(self) -> dict:
        return {"seg": self.seg, "role": self.role, "turn": self.turn,
                "role_think": self.role_think, "dense_bits": self.dense_bits,
                "dense_offsets": self.dense_offsets}

    def device_meta(self, device="cuda") -> dict:
        """cu_seqlens and the per-token metadata as device tensors (the dense
        mask's uint32 words as int32, the same bytes)."""
        def dev(a):
            return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(device)
        bits = None if self.dense_bits is None else self.dense_bits.view(np.int32)
        return {"cu_seqlens": dev(self.cu_seqlens), "seg_id": dev(self.seg),
                "role": dev(self.role), "turn": dev(self.turn), "dense_bits": dev(bits),
                "dense_offsets": dev(self.dense_offsets)}

    def api_kwargs(self, dm: dict) -> dict:
        """The mask keyword arguments of the library calls, from device_meta()."""
        return {"seg_id": dm["seg_id"], "role": dm["role"], "turn": dm["turn"],
                "role_think": self.role_think, "dense_bits": dm["dense_bits"],
                "dense_offsets": dm["dense_offsets"]}


WORKLOAD_NAMES = {
    1: "causal_s64_d32_fp32",
    2: "varlen_causal_8seq",
    3: "shared_prefix_2048_16x512",
    4: "strip_thinking_8turns",
    5: "causal_document_32k",
    6: "strip_thinking_dup_8turns",
    7: "varlen_noncausal_8seq",
    8: "dense_causal_document_padding_32k",
}


def _cu(lengths) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(lengths, dtype=np.int64))]).astype(np.int32)


def _randn(g: torch.Generator, T: int, H: int, D: int, sigma: float, dtype: torch.dtype) -> torch.Tensor:
    x = torch.randn((T, H, D), generator=g, dtype=torch.float32)
    if sigma != 1.0:
        x = x * sigma
    return x.to(dtype)


def _fill_tensors(w: Workload, g: torch.Generator) -> None:
    T, H, D = w.total_tokens, w.num_heads, w.head_dim
    w.q = _randn(g, T, H, D, w.sigma, w.dtype)
    w.k = _randn(g, T, H, D, w.sigma, w.dtype)
    w.v = _randn(g, T, H, D, w.sigma, w.dtype)


def grad_output(w: Workload, seed: int = 1000) -> torch.Tensor:
    """A seeded upstream gradient dO [T, H, D] for the backward: N(0, 1) in fp32
    from ``torch.Generator`` seeded with ``seed``, cast to the workload dtype."""
    g = torch.Generator().manual_seed(seed)
    return _randn(g, w.total_tokens, w.num_heads, w.head_dim, 1.0, w.dtype)


def make_workload(c: int, tensors: bool = True, document_form: str = "mask") -> Workload:
    """Workload number ``c`` (1..8).  Workload 6 is workload 4's conversation
    with every answer span duplicated (user 128 / think 768 / answer 256 /
    answer history copy 256 per turn, 11264 tokens): the exact variant of
    strip-thinking.  Workload 7 is workload 2's sequences without a mask
    inside a sequence (the "none" kind).  Workload 8 is workload 5's 32768
    tokens as a caller-supplied dense mask: causal, inside a document, and
    with the last 2048 tokens padding (they neither attend nor are attended).

    ``document_form`` only matters for workload 5: ``"mask"`` is one packed
    sequence with the document index in ``seg`` and kind causal_document;
    ``"cu_seqlens"`` is the same tokens as twelve sequences under plain causal.
    Both describe the same set of visible (query, key) pairs.
    """
    g = torch.Generator().manual_seed(c)
    if c == 1:
        w = Workload(WORKLOAD_NAMES[1], "causal", _cu([64]), 1, 32, torch.float32, seed=c)
    elif c == 2:
        lens = torch.randint(128, 2049, (8,), generator=g).tolist()
        w = Workload(WORKLOAD_NAMES[2], "causal", _cu(lens), 16, 128, torch.bfloat16, seed=c)
    elif c == 3:
        seg = np.concatenate([np.zeros(2048, np.int32)] +
                             [np.full(512, i, np.int32) for i in range(1, 17)])
        w = Workload(WORKLOAD_NAMES[3], "shared_prefix", _cu([len(seg)]), 32, 128,
                     torch.bfloat16, seg=seg, seed=c)
    elif c == 4:
        role, turn = strip_thinking_layout([(128, 768, 256)] * 8)
        w = Workload(WORKLOAD_NAMES[4], "strip_thinking", _cu([len(role)]), 32, 128,
                     torch.bfloat16, sigma=0.5, role=role, turn=turn, seed=c)
    elif c == 7:
        lens = torch.randint(128, 2049, (8,), generator=torch.Generator().manual_seed(2)).tolist()
        w = Workload(WORKLOAD_NAMES[7], "none", _cu(lens), 16, 128, torch.bfloat16, seed=c)
    elif c == 8:
        g5 = torch.Generator().manual_seed(5)
        cuts = torch.randint(0, 26625, (11,), generator=g5).sort().values.tolist()
        bounds = [0] + cuts + [26624]
        lens = [bounds[i + 1] - bounds[i] + 512 for i in range(12)]
        seg = np.concatenate([np.full(n, i, np.int32) for i, n in enumerate(lens)])
        seg[-2048:] = -1  # padding
        bits, offs = causal_document_padding_bits(seg)
        w = Workload(WORKLOAD_NAMES[8], "dense", _cu([len(seg)]), 32, 128, torch.bfloat16,
                     seg=None, dense_bits=bits, dense_offsets=offs, seed=c)
    elif c == 6:
        role, turn = strip_thinking_dup_layout([(128, 768, 256)] * 8)
        w = Workload(WORKLOAD_NAMES[6], "strip_thinking_dup", _cu([len(role)]), 32, 128,
                     torch.bfloat16, sigma=0.5, role=role, turn=turn, seed=c)
    elif c == 5:
        cuts = torch.randint(0, 26625, (11,), generator=g).sort().values.tolist()
        bounds = [0] + cuts + [26624]
        lens = [bounds[i + 1] - bounds[i] + 512 for i in range(12)]
        if document_form == "mask":
            seg = np.concatenate([np.full(n, i, np.int32) for i, n in enumerate(lens)])
            w = Workload(WORKLOAD_NAMES[5], "causal_document", _cu([sum(lens)]), 32, 128,
                         torch.bfloat16, seg=seg, seed=c)
        elif document_form == "cu_seqlens":
            w = Workload(WORKLOAD_NAMES[5] + "_cu_seqlens", "causal", _cu(lens), 32, 128,
                         torch.bfloat16, seed=c)
        else:
            raise ValueError(document_form)
    else:
        raise ValueError(f"workload number must be 1..8, got {c}")
    if tensors:
        _fill_tensors(w, g)
    return w


def strip_thinking_layout(turns):
    """Role and turn arrays for turns given as (user, think, answer) lengths."""
    role, turn = [], []
    for t, (nu, nt, na) in enumerate(turns, start=1):
        role += [ROLE_USER] * nu + [ROLE_THINK] * nt + [ROLE_ANSWER] * na
        turn += [t] * (nu + nt + na)
    return np.asarray(role, np.int8), np.asarray(turn, np.int32)


def strip_thinking_dup_layout(turns):
    """Role and turn arrays for turns given as (user, think, answer) lengths,
    each answer span followed by its history copy of the same length."""
    role, turn = [], []
    for t, (nu, nt, na) in enumerate(turns, start=1):
        role += [ROLE_USER] * nu + [ROLE_THINK] * nt + [ROLE_ANSWER] * na + [ROLE_ANSWER_HISTORY] * na
        turn += [t] * (nu + nt + 2 * na)
    return np.asarray(role, np.int8), np.asarray(turn, np.int32)


def random_metadata(rng: np.random.Generator, kind: str, lengths, role_think: int = ROLE_THINK,
                    id_alphabet: int = 0):
    """Random per-token metadata for ``kind`` over packed sequences ``lengths``.

    Segment ids are runs (documents / prefix-suffix segments) of random length;
    roles and turns are random runs too, so tile boundaries cut through runs.
    By default ids count up run by run (0, 1, 2, ...) and turns count up from 1.
    With ``id_alphabet`` = n > 0 every run draws its segment id from 0..n-1 and
    every turn its number from 1..n instead, so ids repeat, fall and skip.
    """
    T = int(sum(lengths))
    seg = role = turn = None
    if kind in ("causal_document", "shared_prefix"):
        seg = np.empty(T, np.int32)
        pos = 0
        for L in lengths:
            s, cur = 0, 0
            while s < L:
                n = int(rng.integers(1, max(2, L // 2 + 2)))
                seg[pos + s: pos + min(L, s + n)] = cur if id_alphabet <= 0 else int(rng.integers(0, id_alphabet))
                s += n
                cur += 1
            pos += L
    if kind in ("strip_thinking", "strip_thinking_dup"):
        role = np.empty(T, np.int8)
        turn = np.empty(T, np.int32)
        spans = (ROLE_USER, role_think, ROLE_ANSWER) if kind == "strip_thinking" else \
            (ROLE_USER, role_think, ROLE_ANSWER, ROLE_ANSWER_HISTORY)
        pos = 0
        for L in lengths:
            s, t = 0, 1
            while s < L:
                tt = t if id_alphabet <= 0 else int(rng.integers(1, id_alphabet + 1))
                for r in spans:
                    n = int(rng.integers(1, 200))
                    role[pos + s: pos + min(L, s + n)] = r
                    turn[pos + s: pos + min(L, s + n)] = tt
                    s += n
                    if s >= L:
                        break
                t += 1
            pos += L
    return seg, role, turn


def dense_offsets(lengths) -> np.ndarray:
    """First uint32 word of each sequence's bit rows (L rows of ceil(L / 32)
    words each), and the total, as int64 [B+1]."""
    words = [L * ((L + 31) // 32) for L in lengths]
    return np.concatenate([[0], np.cumsum(words)]).astype(np.int64)


def pack_rows(rows: np.ndarray, pad_rng: Optional[np.random.Generator] = None) -> np.ndarray:
    """Bool rows [R, L] packed as uint32 words, bit j % 32 of word j // 32.  The
    bits past L in the last word are random when ``pad_rng`` is given (they
    must be ignored), else zero."""
    R, L = rows.shape
    W = (L + 31) // 32
    full = np.zeros((R, W * 32), bool)
    full[:, :L] = rows
    if pad_rng is not None and W * 32 > L:
        full[:, L:] = pad_rng.random((R, W * 32 - L)) < 0.5
    return np.packbits(full, axis=1, bitorder="little").view(np.uint32).reshape(R, W)


def causal_document_padding_bits(seg: np.ndarray, block: int = 128):
    """The caller's input of the DENSE kind for workload 8: one sequence's bit
    rows composed as the pages' causal + document + padding (key at or before
    the query, same document id, neither token padding, id < 0).  This is input
    data, like seg_id for the other kinds: the library reads the bits and the
    oracle checks the composition on its own.  Returns (bits uint32, offsets
    int64 [2])."""
    L = len(seg)
    rows = []
    for r0 in range(0, L, block):
        qi = np.arange(r0, min(L, r0 + block))[:, None]
        ki = np.arange(L)[None, :]
        m = (ki <= qi) & (seg[ki] == seg[qi]) & (seg[ki] >= 0) & (seg[qi] >= 0)
        rows.append(pack_rows(m).ravel())
    return np.concatenate(rows).astype(np.uint32), dense_offsets([L])


def random_dense_mask(rng: np.random.Generator, lengths, tile: int = 128):
    """A random caller-supplied mask per sequence for the "dense" kind: every
    tile x tile block is drawn as all hidden, all visible, random bits, or a
    random lower-left staircase; a few rows see nothing at all; the bits past
    a row's end are random.  Returns (bits uint32, offsets int64 [B+1])."""
    out = []
    for L in lengths:
        nt = -(-L // tile)
        m = np.zeros((L, L), bool)
        for a in range(nt):
            for c in range(nt):
                r0, r1, c0, c1 = a * tile, min(L, (a + 1) * tile), c * tile, min(L, (c + 1) * tile)
                mode = rng.choice(4, p=[0.3, 0.3, 0.25, 0.15])
                if mode == 1:
                    m[r0:r1, c0:c1] = True
                elif mode == 2:
                    m[r0:r1, c0:c1] = rng.random((r1 - r0, c1 - c0)) < rng.uniform(0.05, 0.95)
                elif mode == 3:
                    shift = int(rng.integers(-tile, tile))
                    ii = np.arange(r0, r1)[:, None]
                    jj = np.arange(c0, c1)[None, :]
                    m[r0:r1, c0:c1] = jj - c0 <= ii - r0 + shift
        empty = rng.random(L) < 0.02
        m[empty] = False
        out.append(pack_rows(m, rng).ravel())
    bits = np.concatenate(out) if out else np.zeros(0, np.uint32)
    return bits.astype(np.uint32), dense_offsets(lengths)


def random_meta(rng: np.random.Generator, kind: str, lengths, role_think: int = ROLE_THINK,
                id_alphabet: int = 0) -> dict:
    """random_metadata as the dict the oracle takes, with a random dense mask
    for the "dense" kind."""
    seg, role, turn = random_metadata(rng, kind, lengths, role_think, id_alphabet)
    bits = offs = None
    if kind == "dense":
        bits, offs = random_dense_mask(rng, lengths)
    return {"seg": seg, "role": role, "turn": turn, "role_think": role_think,
            "dense_bits": bits, "dense_offsets": offs}


def random_workload(seed: int, kind: str, lengths, num_heads: int, head_dim: int,
                    dtype: torch.dtype = torch.bfloat16, sigma: float = 1.0,
                    id_alphabet: int = 0) -> Workload:
    """A small seeded case for parity tests (ragged lengths, any kind); see
    random_metadata for ``id_alphabet``."""
    rng = np.random.default_rng(seed)
    m = random_meta(rng, kind, lengths, id_alphabet=id_alphabet)
    w = Workload(f"random_{kind}_{seed}", kind, _cu(lengths), num_heads, head_dim, dtype,
                 sigma=sigma, seg=m["seg"], role=m["role"], turn=m["turn"],
                 dense_bits=m["dense_bits"], dense_offsets=m["dense_offsets"], seed=seed)
    _fill_tensors(w, torch.Generator().manual_seed(10_000 + seed))
    return w
