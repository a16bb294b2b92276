// Internal declarations shared by the translation units of libattnmask.
// Not installed; the public interface is include/attn_block_mask.h.
#pragma once

#include <cstddef>
#include <cstdint>
#include <climits>

#include <cuda_runtime.h>

#include "attn_block_mask.h"

namespace attnmask {

constexpr uint32_t kMaskMagic = 0x4B53414Du;  // "MASK"
constexpr int kTile = 128;                    // q-tile rows = k-tile columns

// Device error bits, kept in header[kHdrError] of the block-mask workspace.
enum : int32_t {
  kErrCuFirst = 1 << 0,      // cu_seqlens[0] != 0
  kErrCuOrder = 1 << 1,      // cu_seqlens decreases somewhere
  kErrCuLast = 1 << 2,       // cu_seqlens[batch] != total_tokens
  kErrSeqTooLong = 1 << 3,   // a sequence is longer than max_seqlen
  kErrTimeout = 1 << 8,      // a pipeline wait gave up (bits 9.. hold the wait site)
  kErrInputMask = kErrCuFirst | kErrCuOrder | kErrCuLast | kErrSeqTooLong,
};

// Header words of the block-mask workspace (the kernels' work counters are
// per launch, not here: words 7 and up are reserved and zeroed by the build).
enum : int { kHdrQtiles = 0, kHdrEntries = 1, kHdrError = 2, kHdrPairs = 3, kHdrEmpty = 4,
             kHdrPartial = 5, kHdrFull = 6, kHdrInts = 16 };

enum : int { kSumInts = 8 };  // ints per tile summary

// Byte layout of the block-mask workspace.
struct BmLayout {
  int max_qt = 0, max_nt = 0;
  uint64_t header = 0, qt_seq = 0, qt_idx = 0, labels = 0, kcount = 0, koff = 0, kidx = 0,
           klabel = 0, order = 0, qt_off = 0, summary = 0, pair_off = 0, pair_q0 = 0,
           pair_order = 0, qcount = 0, qoff = 0, qidx = 0, qlabel = 0, korder = 0, total = 0;
};

// False when a STRIP_THINKING_DUP mask names role 2 or 3 as THINK.
bool role_think_valid(int kind, const attn_mask_params* params);
// False when a DENSE mask lacks its bits or offsets (or they are misaligned).
bool dense_valid(int kind, const attn_mask_params* params);

// Returns false on overflow / invalid sizes.
bool bm_layout(int batch, int total_tokens, int max_seqlen, BmLayout* out);

// Device-side view of a built block mask.
struct BmView {
  int32_t* header;
  int32_t* qt_seq;
  int32_t* qt_idx;
  uint8_t* labels;
  int32_t* kcount;
  int32_t* koff;
  int32_t* kidx;
  uint8_t* klabel;
  int32_t* order;
  int32_t* qt_off;
  int32_t* summary;
  int32_t* pair_off;
  int32_t* pair_q0;
  int32_t* pair_order;
  int32_t* qcount;   // transposed (k-major) lists
  int32_t* qoff;
  int32_t* qidx;
  uint8_t* qlabel;
  int32_t* korder;
  const int32_t* cu;
  int max_qt, max_nt, batch, total_tokens, max_seqlen;
};

// Per-token mask metadata as the kernels see it.
struct MaskArgs {
  int kind;
  int role_think;
  const int32_t* seg;
  const int8_t* role;
  const int32_t* turn;
  const uint32_t* bits;    // ATTN_MASK_DENSE: the caller's bit rows
  const int64_t* bit_off;  // ATTN_MASK_DENSE: first word of each sequence
};

// Kinds that only keep keys at or before the query.
__host__ __device__ constexpr bool kind_causal(int kind) { return kind <= ATTN_MASK_STRIP_THINKING_DUP; }
// Kinds whose PARTIAL tiles are decided by per-token codes (below).
__host__ __device__ constexpr bool kind_codes(int kind) {
  return kind >= ATTN_MASK_CAUSAL_DOCUMENT && kind <= ATTN_MASK_STRIP_THINKING_DUP;
}

// ATTN_MASK_DENSE: word jw (keys 32 jw .. 32 jw + 31) of local row i of
// sequence b, whose length is L.
__device__ __forceinline__ uint32_t dense_word(const MaskArgs& m, int b, int L, int i, int jw) {
  return __ldg(m.bits + m.bit_off[b] + int64_t(i) * ((L + 31) >> 5) + jw);
}

// The four predicates factor as  (ki <= qi) && code_visible(qcode(qi), kcode(ki)):
//   causal          : always true
//   causal_document : seg[k] == seg[q]
//   shared_prefix   : seg[k] == 0 || seg[k] == seg[q]
//   strip_thinking  : !(role[k] == THINK && turn[k] < turn[q]); the key code is
//                     turn[k] for THINK keys and INT_MAX otherwise, so the test
//                     becomes kcode >= turn[q].
//   strip_thinking_dup: both codes are 4 turn + class, class 1 THINK, 2 ANSWER
//                     (the copy that sees its own thinking), 3 ANSWER_HISTORY,
//                     0 anything else; see dup_visible.
__device__ __forceinline__ int dup_class(int role, int role_think) {
  return role == role_think ? 1 : (role == 2 ? 2 : (role == 3 ? 3 : 0));
}

// Duplicated answers: context keys are seen by every later query; THINK keys
// by their own turn's THINK and ANSWER queries; ANSWER keys only by their own
// turn's ANSWER queries; ANSWER_HISTORY keys by every later turn and by their
// own turn's ANSWER_HISTORY queries.
__device__ __forceinline__ bool dup_visible(int qcode, int kcode) {
  const int kc = kcode & 3, qc = qcode & 3, kt = kcode >> 2, qt = qcode >> 2;
  if (kc == 0) return true;
  if (kc == 1) return kt == qt && (qc == 1 || qc == 2);
  if (kc == 2) return kt == qt && qc == 2;
  return kt < qt || (kt == qt && qc == 3);
}

__device__ __forceinline__ int query_code(const MaskArgs& m, int qi) {
  switch (m.kind) {
    case ATTN_MASK_CAUSAL_DOCUMENT:
    case ATTN_MASK_SHARED_PREFIX: return m.seg[qi];
    case ATTN_MASK_STRIP_THINKING: return m.turn[qi];
    case ATTN_MASK_STRIP_THINKING_DUP: return 4 * m.turn[qi] + dup_class(m.role[qi], m.role_think);
    default: return 0;
  }
}

__device__ __forceinline__ int key_code(const MaskArgs& m, int ki) {
  switch (m.kind) {
    case ATTN_MASK_CAUSAL_DOCUMENT:
    case ATTN_MASK_SHARED_PREFIX: return m.seg[ki];
    case ATTN_MASK_STRIP_THINKING:
      return (int)m.role[ki] == m.role_think ? m.turn[ki] : INT_MAX;
    case ATTN_MASK_STRIP_THINKING_DUP: return 4 * m.turn[ki] + dup_class(m.role[ki], m.role_think);
    default: return 0;
  }
}

__device__ __forceinline__ bool code_visible(int kind, int qcode, int kcode) {
  switch (kind) {
    case ATTN_MASK_CAUSAL_DOCUMENT: return kcode == qcode;
    case ATTN_MASK_SHARED_PREFIX: return kcode == 0 || kcode == qcode;
    case ATTN_MASK_STRIP_THINKING: return kcode >= qcode;
    case ATTN_MASK_STRIP_THINKING_DUP: return dup_visible(qcode, kcode);
    default: return true;
  }
}

// Remember a CUDA failure for attn_last_error_message(); returns ATTN_ERR_CUDA.
attn_status record_cuda_error(cudaError_t e, const char* where);

// Launchers (return a cudaError_t of the launch).
cudaError_t launch_block_mask_build(const BmView& v, const MaskArgs& m, cudaStream_t s);

struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int total_tokens, num_heads, head_dim;
  float scale;
  BmView bm;
  MaskArgs mask;
};

// Returns ATTN_OK or an error status (tensor-map encoding or launch failure).
attn_status launch_attn_fwd_bf16(const FwdArgs& a, cudaStream_t s);
attn_status launch_attn_fwd_f32(const FwdArgs& a, cudaStream_t s);

// Byte layout of the backward's workspace: per q-tile and head the side values
// of its 128 rows, fp32 [H][max_qtiles][kBwdSideFloats] (LSE * log2 e, +inf
// for rows that see no key or lie past the sequence end; D = rowsum(dO * O);
// the fixed-point multiplier m_i), ||dO_i|| fp32 [H, T], the bound words of
// every (sequence, head) (fp32 [batch][H][4]), and the dQ accumulator, int32
// fixed point [T, H, D].
constexpr int kBwdSideFloats = 3 * kTile;
struct BwdLayout {
  uint64_t side = 0, dnorm = 0, bounds = 0, dqacc = 0, total = 0;
};
bool bwd_layout(int batch, int total_tokens, int num_heads, int head_dim, int max_qt, BwdLayout* out);

struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dout;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  void* workspace;
  BwdLayout ws;
  int total_tokens, num_heads, head_dim;
  float scale;
  BmView bm;
  MaskArgs mask;
};

attn_status launch_attn_bwd_bf16(const BwdArgs& a, cudaStream_t s);

}  // namespace attnmask
