"""Plain fp64 CPU oracle for the structured-mask attention forward.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this module:
only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
It shares no code with the CUDA library (no kernels, headers, helpers or
constant tables); the two only meet on the seeded inputs.

What it computes, step by step and in the pages' terms:

1. For each packed sequence (cu_seqlens, the xorl issue "Block-mask attention:
   shared-prefix and strip-thinking", Summary) it materialises the boolean mask
   M[i, j] by evaluating the mask predicate literally on every (query, key)
   pair of that sequence.  Pairs from different sequences are never visible.
2. For each head it forms the scaled scores s = (q . k) / sqrt(d) in fp64,
   drops masked entries (they get zero weight, the same as exp(-inf)), and
   takes the three-pass softmax: m = max s, l = sum exp(s - m), LSE = m + ln l,
   O = sum exp(s - m) v / l  ("Triton from first principles" Ch. 21,
   Section 21.1, the naive softmax(QK^T/sqrt(d))V the kernel is checked
   against).  A row with no visible key gets O = 0 and LSE = -inf.
3. Tile labels by brute force: count the visible in-bounds pairs of every
   128x128 (q-tile, k-tile) block of M; EMPTY if none, FULL if all, PARTIAL
   otherwise ("Triton from first principles" Ch. 21, Section 21.2 diagram:
   all-valid / diagonal / skipped tiles).  Lists are in ascending k order.

Readings of points the pages leave open (each is listed in the design notes):
* the diagonal is visible under every kind (``j <= i``, Ch. 9, Section 9.1);
* LSE is the natural log of the sum of exp of the *scaled* scores;
* roles are USER=0, THINK=1, ANSWER=2 with the THINK code a parameter;
* a ragged tail tile is labelled from its in-bounds pairs only;
* tile grids restart at every sequence's first token.

Every input array is widened to fp64 before use; bf16 and fp32 widen exactly.
"""
from __future__ import annotations

import numpy as np

KINDS = ("causal", "causal_document", "shared_prefix", "strip_thinking", "strip_thinking_dup",
         "none", "dense")

# Roles of the duplicated-answer layout: the answer copy that attends its own
# turn's thinking (and carries the loss), and the history copy later turns see.
ROLE_ANSWER, ROLE_ANSWER_HISTORY = 2, 3

EMPTY, PARTIAL, FULL = 0, 1, 2


# ----------------------------------------------------------------------------
# Mask predicates.  qi / ki are global packed token indices of one sequence,
# so ``qi >= ki`` is the same test as comparing positions inside the sequence.
# ----------------------------------------------------------------------------

def predicate(kind: str, qi, ki, seg=None, role=None, turn=None, role_think: int = 1):
    """Visibility of key ``ki`` to query ``qi`` (broadcasting integer arrays).

    * causal          : key at or before the query, diagonal included
                        ("Triton from first principles" Ch. 9, Section 9.1,
                        Worked Example 9.1.1: ``cols <= rows``).
    * causal_document : causal and the same document id (the xorl issue,
                        "Decisions this settles", item 4: document boundaries
                        move into the mask).
    * shared_prefix   : ``(qi >= ki) & ((seg[ki] == 0) | (seg[ki] == seg[qi]))``
                        (the xorl issue, Mask specifications, "Shared prefix").
    * strip_thinking  : ``(qi >= ki) & ~((role[ki] == THINK) & (turn[ki] < turn[qi]))``
                        (the xorl issue, Mask specifications, "Strip-thinking").
    * strip_thinking_dup : the same conversation with every answer span
                        duplicated (the xorl issue, "The exactness question",
                        option (b)): the ANSWER copy attends its own turn's
                        thinking, the ANSWER_HISTORY copy attends the stripped
                        context and is what later turns see.  With the key at
                        or before the query, a key is visible when it is
                        - neither THINK nor an answer copy (user / context);
                        - THINK of the query's own turn, and the query is THINK
                          or ANSWER of that turn;
                        - ANSWER of the query's own turn, and the query is
                          ANSWER (the copy itself, causally);
                        - ANSWER_HISTORY of an earlier turn, or of the query's
                          own turn with the query ANSWER_HISTORY too.
    """
    qi = np.asarray(qi)
    ki = np.asarray(ki)
    causal = qi >= ki
    if kind == "causal":
        return causal
    if kind == "causal_document":
        return causal & (seg[ki] == seg[qi])
    if kind == "shared_prefix":
        return causal & ((seg[ki] == 0) | (seg[ki] == seg[qi]))
    if kind == "strip_thinking":
        return causal & ~((role[ki] == role_think) & (turn[ki] < turn[qi]))
    if kind == "strip_thinking_dup":
        rk, rq, tk, tq = role[ki], role[qi], turn[ki], turn[qi]
        same = tk == tq
        think_k, ans_k, hist_k = rk == role_think, rk == ROLE_ANSWER, rk == ROLE_ANSWER_HISTORY
        context_k = ~(think_k | ans_k | hist_k)
        think_seen = think_k & same & ((rq == role_think) | (rq == ROLE_ANSWER))
        ans_seen = ans_k & same & (rq == ROLE_ANSWER)
        hist_seen = hist_k & ((tk < tq) | (same & (rq == ROLE_ANSWER_HISTORY)))
        return causal & (context_k | think_seen | ans_seen | hist_seen)
    raise ValueError(f"unknown mask kind {kind!r}")


def dense_bits(meta: dict, cu_seqlens, b: int, rows, cols):
    """The caller-supplied mask of sequence ``b`` at local rows x cols, for the
    ``dense`` kind: bit (i, j) of the sequence, row-major with rows of
    ceil(L / 32) uint32 words from word ``dense_offsets[b]``, bit j % 32 of
    word j // 32, 1 = visible."""
    L = int(cu_seqlens[b + 1] - cu_seqlens[b])
    W = (L + 31) // 32
    rows = np.asarray(rows, np.int64)[:, None]
    cols = np.asarray(cols, np.int64)[None, :]
    words = np.asarray(meta["dense_bits"], np.uint32)[int(meta["dense_offsets"][b]) + rows * W + cols // 32]
    return ((words >> (cols % 32).astype(np.uint32)) & 1).astype(bool)


def visible(kind: str, cu_seqlens, b: int, meta: dict, rows, cols):
    """Mask of sequence ``b`` at local query rows x key columns, [rows, cols]:
    the predicate for the metadata kinds, all True for ``none`` (attention
    without a mask inside each sequence: "Triton from first principles"
    Ch. 21, Section 21.1, the plain flash_attn_kernel), and the caller's bits
    for ``dense``."""
    meta = meta or {}
    rows = np.asarray(rows, np.int64)
    cols = np.asarray(cols, np.int64)
    if kind == "none":
        return np.ones((len(rows), len(cols)), bool)
    if kind == "dense":
        return dense_bits(meta, cu_seqlens, b, rows, cols)
    start = int(cu_seqlens[b])
    return predicate(kind, start + rows[:, None], start + cols[None, :], meta.get("seg"),
                     meta.get("role"), meta.get("turn"), meta.get("role_think", 1))


def sequence_mask(kind: str, cu_seqlens, b: int, meta: dict, row_lo: int = 0, row_hi=None,
                  rows=None):
    """Rows of sequence ``b``'s full boolean mask, shape [rows, L].

    With the default arguments this is the whole L x L mask.  ``row_lo`` /
    ``row_hi`` (a range) or ``rows`` (explicit local row indices) only bound
    memory for long sequences; every entry is the same literal predicate.
    """
    start, end = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
    L = end - start
    if rows is None:
        if row_hi is None:
            row_hi = L
        rows = np.arange(row_lo, row_hi)
    return visible(kind, cu_seqlens, b, meta, rows, np.arange(L))


# ----------------------------------------------------------------------------
# Attention by the definition.
# ----------------------------------------------------------------------------

def masked_attention(q, k, v, mask, scale):
    """softmax(q k^T * scale, masked) v for one sequence and one head, in fp64.

    q: [M, D], k: [N, D], v: [N, D], mask: bool [M, N].  Returns O [M, D] and
    LSE [M] (natural log).  Three passes: row max, sum of exponentials, then
    the normalised weighted sum ("Triton from first principles" Ch. 21,
    Section 21.1, the naive reference).  Masked entries carry zero weight.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    mask = np.asarray(mask, bool)
    s = (q @ k.T) * float(scale)
    s = np.where(mask, s, -np.inf)
    m = s.max(axis=1) if s.shape[1] else np.full(s.shape[0], -np.inf)
    has_key = np.isfinite(m)
    m_safe = np.where(has_key, m, 0.0)
    e = np.where(mask, np.exp(s - m_safe[:, None]), 0.0)
    l = e.sum(axis=1)
    o = np.zeros((q.shape[0], v.shape[1]), np.float64)
    o[has_key] = (e[has_key] @ v) / l[has_key, None]
    lse = np.full(q.shape[0], -np.inf)
    lse[has_key] = m[has_key] + np.log(l[has_key])
    return o, lse


def _as_f64(x):
    """Widen a torch tensor or array to a float64 numpy array (exact for bf16/fp32)."""
    if hasattr(x, "detach"):
        x = x.detach().cpu()
        if str(x.dtype) == "torch.bfloat16":
            x = x.float()
        x = x.double().numpy()
    return np.asarray(x, np.float64)


def attention(q, k, v, kind: str, cu_seqlens, meta=None, scale=None, heads=None,
              rows=None, row_block: int = 512):
    """O [T, H, D] and LSE [H, T] of the masked attention forward, fp64.

    q, k, v: [T, H, D] (numpy or torch, any float dtype).  ``heads`` selects
    heads (default all); ``rows`` optionally restricts the computed query rows
    to a list of global token indices (the others stay NaN), which is how the
    full-size parity tests sample outputs one by one.
    """
    T, H, D = q.shape
    cu = np.asarray(cu_seqlens, np.int64)
    if scale is None or scale == 0:
        scale = 1.0 / np.sqrt(D)
    heads = range(H) if heads is None else heads
    O = np.full((T, H, D), np.nan)
    LSE = np.full((H, T), np.nan)
    row_set = None if rows is None else np.unique(np.asarray(rows, np.int64))
    for b in range(len(cu) - 1):
        start, end = int(cu[b]), int(cu[b + 1])
        L = end - start
        if L == 0:
            continue
        if row_set is None:
            local_rows = np.arange(L)
        else:
            sel = row_set[(row_set >= start) & (row_set < end)]
            if len(sel) == 0:
                continue
            local_rows = sel - start
        for c0 in range(0, len(local_rows), row_block):
            lr = local_rows[c0:c0 + row_block]
            mask = sequence_mask(kind, cu, b, meta, rows=lr)
            for h in heads:
                o, lse = masked_attention(_as_f64(q[start + lr, h]), _as_f64(k[start:end, h]),
                                          _as_f64(v[start:end, h]), mask, scale)
                O[start + lr, h] = o
                LSE[h, start + lr] = lse
    return O, LSE


def masked_attention_backward(q, k, v, do, mask, scale):
    """dQ, dK, dV of O = softmax(q k^T * scale, masked) v for one sequence and
    one head, in fp64, given the upstream gradient dO.

    The plain definition: the chain rule through the three-pass forward above
    (the forward of "Triton from first principles" Ch. 21, Section 21.1), with
    masked entries carrying zero weight and no gradient:
      P = softmax(S), S = q k^T * scale (masked), O = P v
      dV = P^T dO,  dP = dO v^T,  D_i = sum_j P_ij dP_ij = sum_d dO_id O_id,
      dS = P * (dP - D),  dQ = dS k * scale,  dK = dS^T q * scale.
    Rows with no visible key have P = 0 and contribute nothing.  The xorl
    issue (Verified FA4 gaps, items 1 and 3) asks for this backward over the
    same block-sparse masks.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    do = np.asarray(do, np.float64)
    mask = np.asarray(mask, bool)
    s = (q @ k.T) * float(scale)
    s = np.where(mask, s, -np.inf)
    m = s.max(axis=1) if s.shape[1] else np.full(s.shape[0], -np.inf)
    has_key = np.isfinite(m)
    m_safe = np.where(has_key, m, 0.0)
    e = np.where(mask, np.exp(s - m_safe[:, None]), 0.0)
    l = e.sum(axis=1)
    p = np.zeros_like(e)
    p[has_key] = e[has_key] / l[has_key, None]
    o = p @ v
    dv = p.T @ do
    dp = do @ v.T
    dlt = (do * o).sum(axis=1)
    ds = p * (dp - dlt[:, None])
    dq = (ds @ k) * float(scale)
    dk = (ds.T @ q) * float(scale)
    return dq, dk, dv


def attention_backward(q, k, v, do, kind: str, cu_seqlens, meta=None, scale=None, heads=None):
    """dQ, dK, dV [T, H, D] of the masked attention (fp64), for upstream
    gradient dO [T, H, D]; sequences of cu_seqlens are independent.  Heads not
    selected by ``heads`` stay NaN."""
    T, H, D = q.shape
    cu = np.asarray(cu_seqlens, np.int64)
    if scale is None or scale == 0:
        scale = 1.0 / np.sqrt(D)
    heads = range(H) if heads is None else heads
    dQ = np.full((T, H, D), np.nan)
    dK = np.full((T, H, D), np.nan)
    dV = np.full((T, H, D), np.nan)
    for b in range(len(cu) - 1):
        start, end = int(cu[b]), int(cu[b + 1])
        if end == start:
            continue
        mask = sequence_mask(kind, cu, b, meta)
        for h in heads:
            dq, dk, dv = masked_attention_backward(_as_f64(q[start:end, h]), _as_f64(k[start:end, h]),
                                                   _as_f64(v[start:end, h]), _as_f64(do[start:end, h]),
                                                   mask, scale)
            dQ[start:end, h] = dq
            dK[start:end, h] = dk
            dV[start:end, h] = dv
    return dQ, dK, dV


def attention_backward_sampled(q, k, v, do, kind: str, cu_seqlens, meta=None, scale=None,
                               heads=None, q_rows=(), k_rows=(), row_block: int = 512):
    """dQ at sampled query rows and dK, dV at sampled key rows (global token
    indices), fp64, for sequences too long for the whole L x L backward.

    The same definition as masked_attention_backward, evaluated row by row for
    dQ and column by column for dK and dV, with P written as
    P_ij = exp(s_ij - LSE_i) over the visible pairs (the softmax normalised by
    its log-sum-exp; LSE and O of every query row come from ``attention``, the
    three-pass forward, and give D_i = sum_d dO_id O_id):
      dQ_i = scale * sum_j P_ij (dP_ij - D_i) k_j,  dP_ij = dO_i . v_j
      dV_j = sum_i P_ij dO_i,  dK_j = scale * sum_i P_ij (dP_ij - D_i) q_i
    Returns dQ, dK, dV [T, H, D] with NaN outside the sampled rows and heads.
    """
    T, H, D = q.shape
    cu = np.asarray(cu_seqlens, np.int64)
    if scale is None or scale == 0:
        scale = 1.0 / np.sqrt(D)
    scale = float(scale)
    heads = list(range(H)) if heads is None else list(heads)
    qr = np.unique(np.asarray(q_rows, np.int64))
    kr = np.unique(np.asarray(k_rows, np.int64))
    meta = meta or {}
    dQ = np.full((T, H, D), np.nan)
    dK = np.full((T, H, D), np.nan)
    dV = np.full((T, H, D), np.nan)
    for b in range(len(cu) - 1):
        start, end = int(cu[b]), int(cu[b + 1])
        sq = qr[(qr >= start) & (qr < end)]
        sk = kr[(kr >= start) & (kr < end)]
        if len(sq) == 0 and len(sk) == 0:
            continue
        tok = np.arange(start, end)
        # The query rows that see at least one sampled key: every other row has
        # P = 0 on all of them and adds exactly nothing to their dK and dV.
        vis_k = visible(kind, cu, b, meta, tok - start, sk - start) if len(sk) else None
        rows_k = tok[vis_k.any(axis=1)] if len(sk) else tok[:0]
        # LSE and O of the query rows used below (the forward oracle)
        need = np.union1d(sq, rows_k)
        O, LSE = attention(q, k, v, kind, cu, meta, scale, heads=heads, rows=need,
                           row_block=row_block)
        for h in heads:
            qh, kh, vh, doh = (_as_f64(x[start:end, h]) for x in (q, k, v, do))
            lse_h = LSE[h, start:end]
            lse_safe = np.where(np.isfinite(lse_h), lse_h, 0.0)  # rows with no key have P = 0
            if len(sq):
                li = sq - start
                vis = visible(kind, cu, b, meta, sq - start, tok - start)
                s = (qh[li] @ kh.T) * scale
                p = np.where(vis, np.exp(np.where(vis, s, 0.0) - lse_safe[li, None]), 0.0)
                d_i = (doh[li] * O[sq, h]).sum(axis=1)
                ds = p * ((doh[li] @ vh.T) - d_i[:, None])
                dQ[sq, h] = (ds @ kh) * scale
            if len(sk):
                lj, li = sk - start, rows_k - start
                vis = vis_k[li]
                dlt = (doh[li] * O[rows_k, h]).sum(axis=1)
                s = (qh[li] @ kh[lj].T) * scale
                p = np.where(vis, np.exp(np.where(vis, s, 0.0) - lse_safe[li, None]), 0.0)
                ds = p * ((doh[li] @ vh[lj].T) - dlt[:, None])
                dV[sk, h] = p.T @ doh[li]
                dK[sk, h] = (ds.T @ qh[li]) * scale
    return dQ, dK, dV


def block_lists_transposed(labels):
    """Per-k-tile compacted lists (the backward's orientation) from per-sequence
    label matrices: the transpose of block_lists.  For every k-tile (sequences
    in order, k-tiles ascending) the ascending q-tiles whose label is not EMPTY,
    with their labels.  Returns qcount, qoff (CSR), qidx (q-tile index within
    the sequence), qlabel.  The xorl issue (Verified FA4 gaps, item 1) names
    this transposed view as the backward's missing metadata.
    """
    qcount, qidx, qlabel = [], [], []
    for lab in labels:
        for kt in range(lab.shape[1]):
            col = lab[:, kt]
            nz = np.nonzero(col)[0]
            qcount.append(len(nz))
            qidx.extend(nz.tolist())
            qlabel.extend(col[nz].tolist())
    qcount = np.asarray(qcount, np.int32)
    qoff = np.zeros(len(qcount) + 1, np.int32)
    qoff[1:] = np.cumsum(qcount)
    return {"qcount": qcount, "qoff": qoff, "qidx": np.asarray(qidx, np.int32),
            "qlabel": np.asarray(qlabel, np.uint8)}


def unmasked_pairs(kind: str, cu_seqlens, meta=None, row_block: int = 1024) -> int:
    """Number of visible (query, key) pairs per head: the nnz that the
    effective-FLOP count 4*D*H*nnz is built on."""
    cu = np.asarray(cu_seqlens, np.int64)
    total = 0
    for b in range(len(cu) - 1):
        L = int(cu[b + 1] - cu[b])
        for r0 in range(0, L, row_block):
            total += int(sequence_mask(kind, cu, b, meta, r0, min(L, r0 + row_block)).sum())
    return total


# ----------------------------------------------------------------------------
# Tile labels and per-q-tile lists by brute-force counting.
# ----------------------------------------------------------------------------

def tile_labels(kind: str, cu_seqlens, meta=None, block_m: int = 128, block_n: int = 128):
    """Per sequence, a uint8 matrix [n_q_tiles, n_k_tiles] of EMPTY/PARTIAL/FULL.

    Each label comes from counting the visible pairs of the tile's in-bounds
    part of the materialised mask: 0 -> EMPTY, all -> FULL, else PARTIAL.
    """
    cu = np.asarray(cu_seqlens, np.int64)
    out = []
    for b in range(len(cu) - 1):
        L = int(cu[b + 1] - cu[b])
        nq = -(-L // block_m)
        nk = -(-L // block_n)
        lab = np.zeros((nq, nk), np.uint8)
        for a in range(nq):
            r0, r1 = a * block_m, min(L, (a + 1) * block_m)
            rows = sequence_mask(kind, cu, b, meta, r0, r1)
            padded = np.zeros((r1 - r0, nk * block_n), bool)
            padded[:, :L] = rows
            counts = padded.reshape(r1 - r0, nk, block_n).sum(axis=(0, 2))
            kn = np.minimum(block_n, L - np.arange(nk) * block_n)
            inb = (r1 - r0) * kn
            lab[a] = np.where(counts == 0, EMPTY, np.where(counts == inb, FULL, PARTIAL))
        out.append(lab)
    return out


def block_lists(labels):
    """Per-q-tile compacted lists from per-sequence label matrices.

    q-tiles are numbered sequence-major (sequence 0's tiles first, each in
    ascending order).  Returns a dict with numpy arrays: ``qt_seq``,
    ``qt_idx`` (q-tile index inside its sequence), ``kcount``, ``koff``
    (CSR offsets, length n+1), ``kidx`` (ascending k-tile indices) and
    ``klabel`` (PARTIAL or FULL per list entry).
    """
    qt_seq, qt_idx, kcount, kidx, klabel = [], [], [], [], []
    for b, lab in enumerate(labels):
        for a in range(lab.shape[0]):
            nz = np.nonzero(lab[a] != EMPTY)[0]
            qt_seq.append(b)
            qt_idx.append(a)
            kcount.append(len(nz))
            kidx.extend(nz.tolist())
            klabel.extend(lab[a, nz].tolist())
    kcount = np.asarray(kcount, np.int64)
    return {
        "qt_seq": np.asarray(qt_seq, np.int64),
        "qt_idx": np.asarray(qt_idx, np.int64),
        "kcount": kcount,
        "koff": np.concatenate([[0], np.cumsum(kcount)]).astype(np.int64),
        "kidx": np.asarray(kidx, np.int64),
        "klabel": np.asarray(klabel, np.uint8),
    }


def lpt_order(kcount):
    """q-tiles by descending work (list length), ties by ascending tile number:
    the longest-processing-time-first order a one-launch varlen scheduler uses
    ("Triton from first principles" Ch. 9, Section 9.3: one launch covers the
    whole ragged batch)."""
    kcount = np.asarray(kcount, np.int64)
    return np.lexsort((np.arange(len(kcount)), -kcount)).astype(np.int64)


def label_totals(labels):
    """(FULL, PARTIAL, EMPTY) counts over all sequences."""
    f = sum(int((l == FULL).sum()) for l in labels)
    p = sum(int((l == PARTIAL).sum()) for l in labels)
    e = sum(int((l == EMPTY).sum()) for l in labels)
    return f, p, e
