// Block-mask builder: tile summaries, exact FULL/PARTIAL/EMPTY classification
// of every (q-tile, k-tile) pair of each sequence, compacted per-q-tile k-tile
// lists (forward, q-major orientation) and a longest-first q-tile order.
//
// "Triton from first principles" Ch. 9, Section 9.2 skips whole tiles on a
// per-tile scalar flag, and Ch. 21, Section 21.2 names the three tile classes
// (all-valid, diagonal/partial, skipped).  The xorl issue "Block-mask
// attention: shared-prefix and strip-thinking" builds such a mask once from
// per-token segment / role / turn tensors and reuses it (Proposed work,
// item 3); its forward metadata is per-q-block lists of k-blocks.
//
// Exactness: a label is decided from per-tile metadata summaries only when the
// summaries prove it (interval reasoning below); every other pair is counted
// pair by pair with the predicate, so labels always equal brute-force counts.
#include "common.cuh"

namespace attnmask {
namespace {

constexpr int kUnknown = -1;

__device__ __forceinline__ int warp_sum(int x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
__device__ __forceinline__ int warp_min(int x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = min(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ int warp_max(int x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = max(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// Block-wide exclusive prefix sum of one value per thread (blockDim.x a
// multiple of 32, at most 1024); returns the prefix and sets *total.
__device__ __forceinline__ int block_exclusive_scan(int x, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nw) s_warp[lane] = w;
  }
  __syncthreads();
  const int before = (warp ? s_warp[warp - 1] : 0) + incl - x;
  *total = s_warp[nw - 1];
  __syncthreads();
  return before;
}

// 1 CTA: validate cu_seqlens; per-sequence q-tile and q-tile-pair offsets;
// q-tile -> (seq, idx); pair -> first q-tile.  A pair is q-tiles (2j, 2j+1)
// of one sequence (the second is absent when the sequence has an odd count).
__global__ void __launch_bounds__(1024) bm_prepare_kernel(BmView v) {
  __shared__ int s_err;
  __shared__ int s_warp[32];
  __shared__ int s_carry;
  __shared__ int s_pcarry;
  const int tid = threadIdx.x;
  if (tid == 0) { s_err = 0; s_carry = 0; s_pcarry = 0; }
  __syncthreads();
  const int B = v.batch;
  int err = 0;
  for (int b = tid; b < B; b += blockDim.x) {
    const int c0 = v.cu[b], c1 = v.cu[b + 1];
    if (c1 < c0) err |= kErrCuOrder;
    else if (c1 - c0 > v.max_seqlen) err |= kErrSeqTooLong;
  }
  if (tid == 0) {
    if (v.cu[0] != 0) err |= kErrCuFirst;
    if (v.cu[B] != v.total_tokens) err |= kErrCuLast;
  }
  if (err) atomicOr(&s_err, err);
  __syncthreads();
  const int bad = s_err;

  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + tid;
    int nt = 0;
    if (!bad && b < B) nt = (v.cu[b + 1] - v.cu[b] + kTile - 1) / kTile;
    int tot_t, tot_p;
    const int bt = block_exclusive_scan(nt, s_warp, &tot_t);
    const int bp = block_exclusive_scan((nt + 1) / 2, s_warp, &tot_p);
    if (b < B) {
      v.qt_off[b] = s_carry + bt;
      v.pair_off[b] = s_pcarry + bp;
    }
    __syncthreads();
    if (tid == 0) { s_carry += tot_t; s_pcarry += tot_p; }
    __syncthreads();
  }
  const int n_qt = s_carry, n_pairs = s_pcarry;
  if (tid == 0) {
    v.qt_off[B] = n_qt;
    v.pair_off[B] = n_pairs;
    v.header[kHdrQtiles] = n_qt;
    v.header[kHdrEntries] = 0;
    v.header[kHdrError] = bad;
    v.header[kHdrPairs] = n_pairs;
    v.header[kHdrEmpty] = 0;
    v.header[kHdrPartial] = 0;
    v.header[kHdrFull] = 0;
    for (int i = 7; i < kHdrInts; ++i) v.header[i] = 0;
  }
  __syncthreads();
  for (int g = tid; g < n_qt; g += blockDim.x) {
    // sequence b with qt_off[b] <= g < qt_off[b+1] (empty sequences own no tile)
    int lo = 0, hi = B;  // answer in [lo, hi)
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (v.qt_off[mid] <= g) lo = mid; else hi = mid;
    }
    v.qt_seq[g] = lo;
    v.qt_idx[g] = g - v.qt_off[lo];
    v.qcount[g] = 0;  // counted by the classifier
  }
  for (int p = tid; p < n_pairs; p += blockDim.x) {
    int lo = 0, hi = B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (v.pair_off[mid] <= p) lo = mid; else hi = mid;
    }
    v.pair_q0[p] = v.qt_off[lo] + 2 * (p - v.pair_off[lo]);
  }
}

// Per 128-token tile: the metadata summary the classifier reasons with.
//   causal_document / shared_prefix: [0] min seg, [1] max seg, [2] any seg == 0
//   strip_thinking: [0] min turn, [1] max turn, [2] #THINK tokens,
//                   [3] min THINK turn, [4] max THINK turn, [5] #tokens
//   strip_thinking_dup: as strip_thinking with [2]-[4] over the private
//                   tokens (THINK and ANSWER copies), [6] the max turn of
//                   ANSWER_HISTORY tokens and [7] the set of classes present
//                   (bit c for class c of dup_class)
__global__ void __launch_bounds__(128) bm_summary_kernel(BmView v, MaskArgs m) {
  const int g = blockIdx.x;
  if (g >= v.header[kHdrQtiles] || !kind_codes(m.kind)) return;
  __shared__ int s_red[4][8];
  const int b = v.qt_seq[g], a = v.qt_idx[g];
  const int s0 = v.cu[b], L = v.cu[b + 1] - s0;
  const int n = min(kTile, L - a * kTile);
  const int r = threadIdx.x, lane = r & 31, warp = r >> 5;
  const bool in = r < n;
  const int tok = s0 + a * kTile + r;
  int x[8];
  if (m.kind == ATTN_MASK_STRIP_THINKING || m.kind == ATTN_MASK_STRIP_THINKING_DUP) {
    const int t = in ? m.turn[tok] : 0;
    const int cls = in ? (m.kind == ATTN_MASK_STRIP_THINKING ? ((int)m.role[tok] == m.role_think ? 1 : 0)
                                                             : dup_class(m.role[tok], m.role_think))
                       : 0;
    const bool priv = cls == 1 || cls == 2;  // THINK (and, duplicated, the ANSWER copy)
    x[0] = warp_min(in ? t : INT_MAX);
    x[1] = warp_max(in ? t : INT_MIN);
    x[2] = warp_sum(priv ? 1 : 0);
    x[3] = warp_min(priv ? t : INT_MAX);
    x[4] = warp_max(priv ? t : INT_MIN);
    x[5] = warp_sum(in ? 1 : 0);
    x[6] = warp_max(cls == 3 ? t : INT_MIN);
    x[7] = int(__reduce_or_sync(0xffffffffu, in ? (1u << cls) : 0u));
  } else {
    const int sg = in ? m.seg[tok] : 0;
    x[0] = warp_min(in ? sg : INT_MAX);
    x[1] = warp_max(in ? sg : INT_MIN);
    x[2] = warp_sum(in && sg == 0 ? 1 : 0);
    x[3] = x[4] = x[5] = x[7] = 0;
    x[6] = INT_MIN;
  }
  if (lane == 0)
    for (int i = 0; i < 8; ++i) s_red[warp][i] = x[i];
  __syncthreads();
  if (r == 0) {
    int* out = v.summary + size_t(g) * kSumInts;
    int mn0 = INT_MAX, mx1 = INT_MIN, c2 = 0, mn3 = INT_MAX, mx4 = INT_MIN, c5 = 0, mx6 = INT_MIN, or7 = 0;
    for (int w = 0; w < 4; ++w) {
      mn0 = min(mn0, s_red[w][0]);
      mx1 = max(mx1, s_red[w][1]);
      c2 += s_red[w][2];
      mn3 = min(mn3, s_red[w][3]);
      mx4 = max(mx4, s_red[w][4]);
      c5 += s_red[w][5];
      mx6 = max(mx6, s_red[w][6]);
      or7 |= s_red[w][7];
    }
    out[0] = mn0; out[1] = mx1; out[2] = c2; out[3] = mn3; out[4] = mx4; out[5] = c5;
    out[6] = mx6; out[7] = or7;
  }
}

// Label of the pair (q rows i0..i1, k columns j0..j1, local positions) when the
// summaries prove it, else kUnknown.  Every rule is a sufficient condition.
__device__ __forceinline__ int decide(int kind, int i0, int i1, int j0, int j1,
                                      const int* sq, const int* sk) {
  if (kind == ATTN_MASK_NONE) return ATTN_TILE_FULL;
  if (j0 > i1) return ATTN_TILE_EMPTY;           // every key after every query
  const bool all_causal = j1 <= i0;              // every key at or before every query
  switch (kind) {
    case ATTN_MASK_CAUSAL:
      // j0 <= i1 gives a visible pair (i1, j0); j1 > i0 a hidden one (i0, j1)
      return all_causal ? ATTN_TILE_FULL : ATTN_TILE_PARTIAL;
    case ATTN_MASK_CAUSAL_DOCUMENT:
      if (sq[1] < sk[0] || sk[1] < sq[0]) return ATTN_TILE_EMPTY;  // no shared document id
      if (sq[0] == sq[1] && sk[0] == sk[1] && sq[0] == sk[0])       // one document throughout
        return all_causal ? ATTN_TILE_FULL : ATTN_TILE_PARTIAL;      // else (i1, j0) seen, (i0, j1) not
      // Every key precedes every query and all keys share one id, held by the
      // first or last query id (so some query row has it): that row sees every
      // key, a row with another id (the ids differ) sees none.
      if (all_causal && sk[0] == sk[1] && sq[0] != sq[1] && (sk[0] == sq[0] || sk[0] == sq[1]))
        return ATTN_TILE_PARTIAL;
      return kUnknown;
    case ATTN_MASK_SHARED_PREFIX:
      if (sk[2] == 0 && (sq[1] < sk[0] || sk[1] < sq[0])) return ATTN_TILE_EMPTY;
      if (all_causal && sk[0] == 0 && sk[1] == 0) return ATTN_TILE_FULL;       // all prefix keys
      if (sq[0] == sq[1] && sk[0] == sk[1] && sq[0] == sk[0])                  // one segment throughout
        return all_causal ? ATTN_TILE_FULL : ATTN_TILE_PARTIAL;
      // As for documents, with suffix keys (id != 0) only: the query row holding
      // their id sees them all, a row with another id sees none.
      if (all_causal && sk[0] == sk[1] && sk[0] != 0 && sq[0] != sq[1] && (sk[0] == sq[0] || sk[0] == sq[1]))
        return ATTN_TILE_PARTIAL;
      return kUnknown;
    case ATTN_MASK_STRIP_THINKING:
      // hidden iff key is THINK with an earlier turn than the query
      if (all_causal && (sk[2] == 0 || sk[3] >= sq[1])) return ATTN_TILE_FULL;
      if (sk[2] == sk[5] && sk[4] < sq[0]) return ATTN_TILE_EMPTY;
      return kUnknown;
    case ATTN_MASK_STRIP_THINKING_DUP:
      // only context keys and history copies of turns before every query's
      if (all_causal && sk[2] == 0 && sk[6] < sq[0]) return ATTN_TILE_FULL;
      // only THINK / ANSWER-copy keys of turns before every query's
      if (sk[2] == sk[5] && sk[4] < sq[0]) return ATTN_TILE_EMPTY;
      // Both tiles inside one turn each, every key before every query: a pair
      // is visible by its two classes alone, and every combination of a key
      // class and a query class present in the tiles occurs as a pair.
      if (all_causal && sq[0] == sq[1] && sk[0] == sk[1]) {
        bool seen = false, hidden = false;
        for (int kc = 0; kc < 4; ++kc)
          for (int qc = 0; qc < 4; ++qc)
            if (((sk[7] >> kc) & 1) && ((sq[7] >> qc) & 1)) {
              if (dup_visible(4 * sq[0] + qc, 4 * sk[0] + kc)) seen = true;
              else hidden = true;
            }
        return seen ? (hidden ? ATTN_TILE_PARTIAL : ATTN_TILE_FULL) : ATTN_TILE_EMPTY;
      }
      return kUnknown;
  }
  return kUnknown;
}

// ATTN_MASK_DENSE: the label of q-tile rows i0 .. i0+qn-1 against k-tile bt,
// by counting the caller's bits (one thread per k-tile, so a warp's loads of
// one row are contiguous); bits past the sequence end do not count.
__device__ __forceinline__ int dense_label(const MaskArgs& m, int b, int L, int i0, int qn, int bt) {
  const int j0 = bt * kTile, kn = min(kTile, L - j0);
  uint32_t keep[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const int n = kn - 32 * w;
    keep[w] = n <= 0 ? 0u : (n >= 32 ? 0xffffffffu : ((1u << n) - 1u));
  }
  const int nw = (kn + 31) >> 5;
  int cnt = 0;
  for (int i = i0; i < i0 + qn; ++i)
#pragma unroll
    for (int w = 0; w < 4; ++w)
      if (w < nw) cnt += __popc(dense_word(m, b, L, i, (j0 >> 5) + w) & keep[w]);
  return cnt == 0 ? ATTN_TILE_EMPTY : (cnt == qn * kn ? ATTN_TILE_FULL : ATTN_TILE_PARTIAL);
}

// One CTA per q-tile: labels of its whole row, and its non-EMPTY count.
// Each thread decides one k-tile from the summaries; only the pairs the
// summaries leave undecided are counted pair by pair, one at a time.
__global__ void __launch_bounds__(128) bm_classify_kernel(BmView v, MaskArgs m) {
  const int g = blockIdx.x;
  if (g >= v.header[kHdrQtiles]) return;
  __shared__ int s_kcode[kTile];
  __shared__ int s_red[4];
  __shared__ int s_unknown[kTile];
  __shared__ int s_nunk;
  __shared__ uint8_t s_lab[kTile];
  const int b = v.qt_seq[g], a = v.qt_idx[g];
  const int s0 = v.cu[b], L = v.cu[b + 1] - s0;
  const int nt = (L + kTile - 1) / kTile;
  const int i0 = a * kTile, i1 = min(L, i0 + kTile) - 1, qn = i1 - i0 + 1;
  const int r = threadIdx.x, lane = r & 31, warp = r >> 5;
  const bool row_in = r < qn;
  const int qcode = row_in ? query_code(m, s0 + i0 + r) : 0;
  int sq[kSumInts];
  const int* qsum = v.summary + size_t(g) * kSumInts;
  for (int i = 0; i < kSumInts; ++i) sq[i] = kind_codes(m.kind) ? qsum[i] : 0;
  const int gbase = v.qt_off[b];
  uint8_t* row = v.labels + size_t(g) * v.max_nt;
  int n_empty = 0, n_partial = 0, n_full = 0;  // meaningful in thread 0
  for (int c0 = 0; c0 < nt; c0 += kTile) {
    const int bt = c0 + r;
    int lab = ATTN_TILE_EMPTY;
    if (r == 0) s_nunk = 0;
    __syncthreads();
    if (bt < nt && m.kind == ATTN_MASK_DENSE) {
      lab = dense_label(m, b, L, i0, qn, bt);
    } else if (bt < nt) {
      int sk[kSumInts];
      const int* ks = v.summary + size_t(gbase + bt) * kSumInts;
      for (int i = 0; i < kSumInts; ++i) sk[i] = kind_codes(m.kind) ? ks[i] : 0;
      const int j0 = bt * kTile, j1 = min(L, j0 + kTile) - 1;
      lab = decide(m.kind, i0, i1, j0, j1, sq, sk);
      if (lab == kUnknown) s_unknown[atomicAdd(&s_nunk, 1)] = r;
    }
    s_lab[r] = uint8_t(lab < 0 ? 0 : lab);
    __syncthreads();
    const int nunk = s_nunk;
    for (int u = 0; u < nunk; ++u) {
      const int bu = c0 + s_unknown[u];
      const int j0 = bu * kTile, kn = min(L, j0 + kTile) - j0;
      if (r < kn) s_kcode[r] = key_code(m, s0 + j0 + r);
      __syncthreads();
      int cnt = 0;
      if (row_in) {
        const int lim = min(kn, i0 + r - j0 + 1);  // keys with j <= i
        for (int c = 0; c < lim; ++c) cnt += code_visible(m.kind, qcode, s_kcode[c]) ? 1 : 0;
      }
      cnt = warp_sum(cnt);
      if (lane == 0) s_red[warp] = cnt;
      __syncthreads();
      if (r == 0) {
        const int total = s_red[0] + s_red[1] + s_red[2] + s_red[3];
        s_lab[s_unknown[u]] = uint8_t(total == 0 ? ATTN_TILE_EMPTY
                                                 : (total == qn * kn ? ATTN_TILE_FULL : ATTN_TILE_PARTIAL));
      }
      __syncthreads();
    }
    if (bt < nt) {
      row[bt] = s_lab[r];
      if (s_lab[r] != ATTN_TILE_EMPTY) atomicAdd(v.qcount + gbase + bt, 1);  // k-tile bt's column
    }
    const int fl = bt < nt ? s_lab[r] : -1;
    const int e = warp_sum(fl == ATTN_TILE_EMPTY), pa = warp_sum(fl == ATTN_TILE_PARTIAL),
              fu = warp_sum(fl == ATTN_TILE_FULL);
    __syncthreads();
    if (lane == 0) { s_red[warp] = e | (pa << 10) | (fu << 20); }
    __syncthreads();
    if (r == 0) {
      for (int w = 0; w < 4; ++w) {
        n_empty += s_red[w] & 1023;
        n_partial += (s_red[w] >> 10) & 1023;
        n_full += (s_red[w] >> 20) & 1023;
      }
    }
    __syncthreads();
  }
  if (r == 0) {
    v.kcount[g] = n_partial + n_full;
    atomicAdd(v.header + kHdrEmpty, n_empty);
    atomicAdd(v.header + kHdrPartial, n_partial);
    atomicAdd(v.header + kHdrFull, n_full);
  }
}

// Exclusive prefix sum of n counts into off[0..n] (1 CTA of 1024 threads).
__device__ void csr_offsets(const int32_t* count, int32_t* off, int n, int* s_warp, int* s_carry) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  if (tid == 0) *s_carry = 0;
  __syncthreads();
  for (int base = 0; base < n; base += blockDim.x) {
    const int g = base + tid;
    const int x = g < n ? count[g] : 0;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = lane < nw ? s_warp[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      if (lane < nw) s_warp[lane] = w;
    }
    __syncthreads();
    if (g < n) off[g] = *s_carry + (warp ? s_warp[warp - 1] : 0) + incl - x;
    __syncthreads();
    if (tid == 0) *s_carry += s_warp[nw - 1];
    __syncthreads();
  }
  if (tid == 0) off[n] = *s_carry;
  __syncthreads();
}

// 1 CTA: CSR offsets koff (q-major lists) and qoff (k-major lists).
__global__ void __launch_bounds__(1024) bm_scan_kernel(BmView v) {
  __shared__ int s_warp[32];
  __shared__ int s_carry;
  const int n = v.header[kHdrQtiles];
  csr_offsets(v.kcount, v.koff, n, s_warp, &s_carry);
  if (threadIdx.x == 0) v.header[kHdrEntries] = v.koff[n];
  csr_offsets(v.qcount, v.qoff, n, s_warp, &s_carry);
}

// One CTA per q-tile: compact its row into ascending (kidx, klabel) entries,
// and place it in the longest-first order (descending kcount, ties by number).
__global__ void __launch_bounds__(128) bm_fill_kernel(BmView v) {
  const int g = blockIdx.x;
  const int n_qt = v.header[kHdrQtiles];
  if (g >= n_qt) return;
  __shared__ int s_warp[4];
  const int r = threadIdx.x, lane = r & 31, warp = r >> 5;
  const int b = v.qt_seq[g];
  const int L = v.cu[b + 1] - v.cu[b];
  const int nt = (L + kTile - 1) / kTile;
  const uint8_t* row = v.labels + size_t(g) * v.max_nt;
  int pos = v.koff[g];
  for (int c0 = 0; c0 < nt; c0 += kTile) {
    const int bt = c0 + r;
    const int lab = bt < nt ? row[bt] : ATTN_TILE_EMPTY;
    const bool keep = lab != ATTN_TILE_EMPTY;
    const unsigned bal = __ballot_sync(0xffffffffu, keep);
    if (lane == 0) s_warp[warp] = __popc(bal);
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += s_warp[w];
    before += __popc(bal & ((1u << lane) - 1u));
    if (keep) {
      v.kidx[pos + before] = bt;
      v.klabel[pos + before] = uint8_t(lab);
    }
    pos += s_warp[0] + s_warp[1] + s_warp[2] + s_warp[3];
    __syncthreads();
  }
  const int mine = v.kcount[g];
  int ahead = 0;
  for (int g2 = r; g2 < n_qt; g2 += blockDim.x) {
    const int k2 = v.kcount[g2];
    ahead += (k2 > mine) || (k2 == mine && g2 < g);
  }
  ahead = warp_sum(ahead);
  if (lane == 0) s_warp[warp] = ahead;
  __syncthreads();
  if (r == 0) v.order[s_warp[0] + s_warp[1] + s_warp[2] + s_warp[3]] = g;
  __syncthreads();
  // The same CTA compacts k-tile g's column (the backward's lists) and places
  // it in the k-tiles' longest-first order.
  {
    const int gbase = v.qt_off[b], bt = v.qt_idx[g];
    int qpos = v.qoff[g];
    for (int a0 = 0; a0 < nt; a0 += kTile) {
      const int a = a0 + r;
      const int lab = a < nt ? v.labels[size_t(gbase + a) * v.max_nt + bt] : ATTN_TILE_EMPTY;
      const bool keep = lab != ATTN_TILE_EMPTY;
      const unsigned bal = __ballot_sync(0xffffffffu, keep);
      if (lane == 0) s_warp[warp] = __popc(bal);
      __syncthreads();
      int before = 0;
      for (int w = 0; w < warp; ++w) before += s_warp[w];
      before += __popc(bal & ((1u << lane) - 1u));
      if (keep) {
        v.qidx[qpos + before] = a;
        v.qlabel[qpos + before] = uint8_t(lab);
      }
      qpos += s_warp[0] + s_warp[1] + s_warp[2] + s_warp[3];
      __syncthreads();
    }
    const int qmine = v.qcount[g];
    int qahead = 0;
    for (int g2 = r; g2 < n_qt; g2 += blockDim.x) {
      const int c2 = v.qcount[g2];
      qahead += (c2 > qmine) || (c2 == qmine && g2 < g);
    }
    qahead = warp_sum(qahead);
    if (lane == 0) s_warp[warp] = qahead;
    __syncthreads();
    if (r == 0) v.korder[s_warp[0] + s_warp[1] + s_warp[2] + s_warp[3]] = g;
    __syncthreads();
  }
  // The CTA of a pair's first q-tile places the pair in the longest-first
  // pair order (work = kcount of both q-tiles, ties by pair number).
  const int qa = v.qt_idx[g];
  if (qa & 1) return;
  auto pair_work = [&](int g0) {
    const bool two = g0 + 1 < n_qt && v.qt_seq[g0 + 1] == v.qt_seq[g0];
    return v.kcount[g0] + (two ? v.kcount[g0 + 1] : 0);
  };
  const int n_pairs = v.header[kHdrPairs];
  const int p = v.pair_off[b] + qa / 2;
  const int wp = pair_work(g);
  int pahead = 0;
  for (int p2 = r; p2 < n_pairs; p2 += blockDim.x) {
    const int w2 = pair_work(v.pair_q0[p2]);
    pahead += (w2 > wp) || (w2 == wp && p2 < p);
  }
  pahead = warp_sum(pahead);
  __syncthreads();
  if (lane == 0) s_warp[warp] = pahead;
  __syncthreads();
  if (r == 0) v.pair_order[s_warp[0] + s_warp[1] + s_warp[2] + s_warp[3]] = p;
}

}  // namespace

cudaError_t launch_block_mask_build(const BmView& v, const MaskArgs& m, cudaStream_t s) {
  const int grid = v.max_qt > 0 ? v.max_qt : 1;
  bm_prepare_kernel<<<1, 1024, 0, s>>>(v);
  bm_summary_kernel<<<grid, 128, 0, s>>>(v, m);
  bm_classify_kernel<<<grid, 128, 0, s>>>(v, m);
  bm_scan_kernel<<<1, 1024, 0, s>>>(v);
  bm_fill_kernel<<<grid, 128, 0, s>>>(v);
  return cudaGetLastError();
}

}  // namespace attnmask
