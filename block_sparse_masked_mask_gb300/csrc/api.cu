// C ABI of libattnmask: argument checks, workspace layout and dispatch.
#include <cmath>
#include <cstdio>
#include <cstdint>
#include <cstring>

#include "common.cuh"

namespace attnmask {

static thread_local char g_last_error[256] = "";

attn_status record_cuda_error(cudaError_t e, const char* where) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", where, cudaGetErrorName(e),
                cudaGetErrorString(e));
  return ATTN_ERR_CUDA;
}

static uint64_t align256(uint64_t x) { return (x + 255u) & ~uint64_t(255u); }

bool bm_layout(int batch, int total_tokens, int max_seqlen, BmLayout* out) {
  if (batch < 0 || total_tokens < 0 || max_seqlen < 0) return false;
  const uint64_t nq = (uint64_t(total_tokens) + kTile - 1) / kTile + uint64_t(batch);
  const uint64_t nk = (uint64_t(max_seqlen) + kTile - 1) / kTile;
  if (nq > uint64_t(INT_MAX) || nq * (nk ? nk : 1) > uint64_t(INT_MAX)) return false;
  BmLayout l;
  l.max_qt = int(nq);
  l.max_nt = int(nk);
  uint64_t p = 0;
  auto take = [&](uint64_t bytes) { uint64_t at = p; p = align256(p + (bytes ? bytes : 1)); return at; };
  l.header = take(sizeof(int32_t) * kHdrInts);
  l.qt_seq = take(4 * nq);
  l.qt_idx = take(4 * nq);
  l.labels = take(nq * nk);
  l.kcount = take(4 * nq);
  l.koff = take(4 * (nq + 1));
  l.kidx = take(4 * nq * nk);
  l.klabel = take(nq * nk);
  l.order = take(4 * nq);
  l.qt_off = take(4 * (uint64_t(batch) + 1));
  l.summary = take(4 * kSumInts * nq);
  l.pair_off = take(4 * (uint64_t(batch) + 1));
  l.pair_q0 = take(4 * nq);
  l.pair_order = take(4 * nq);
  l.qcount = take(4 * nq);
  l.qoff = take(4 * (nq + 1));
  l.qidx = take(4 * nq * nk);
  l.qlabel = take(nq * nk);
  l.korder = take(4 * nq);
  l.total = p;
  *out = l;
  return true;
}

bool bwd_layout(int batch, int total_tokens, int num_heads, int head_dim, int max_qt, BwdLayout* out) {
  if (batch < 1 || total_tokens < 0 || num_heads < 1 || head_dim < 1 || max_qt < 0) return false;
  const uint64_t H = uint64_t(num_heads), T = uint64_t(total_tokens);
  BwdLayout l;
  uint64_t p = 0;
  auto take = [&](uint64_t bytes) { uint64_t at = p; p = align256(p + (bytes ? bytes : 1)); return at; };
  l.side = take(4 * H * uint64_t(max_qt) * kBwdSideFloats);
  l.dnorm = take(4 * H * T);
  l.bounds = take(4 * uint64_t(batch) * H * 4);
  l.dqacc = take(4 * T * H * uint64_t(head_dim));
  l.total = p;
  *out = l;
  return true;
}

static BmView make_view(const attn_block_mask* bm) {
  char* base = static_cast<char*>(bm->workspace);
  BmView v;
  v.header = reinterpret_cast<int32_t*>(base + bm->off_header);
  v.qt_seq = reinterpret_cast<int32_t*>(base + bm->off_qt_seq);
  v.qt_idx = reinterpret_cast<int32_t*>(base + bm->off_qt_idx);
  v.labels = reinterpret_cast<uint8_t*>(base + bm->off_labels);
  v.kcount = reinterpret_cast<int32_t*>(base + bm->off_kcount);
  v.koff = reinterpret_cast<int32_t*>(base + bm->off_koff);
  v.kidx = reinterpret_cast<int32_t*>(base + bm->off_kidx);
  v.klabel = reinterpret_cast<uint8_t*>(base + bm->off_klabel);
  v.order = reinterpret_cast<int32_t*>(base + bm->off_order);
  v.qt_off = reinterpret_cast<int32_t*>(base + bm->off_qt_off);
  v.summary = reinterpret_cast<int32_t*>(base + bm->off_summary);
  v.pair_off = reinterpret_cast<int32_t*>(base + bm->off_pair_off);
  v.pair_q0 = reinterpret_cast<int32_t*>(base + bm->off_pair_q0);
  v.pair_order = reinterpret_cast<int32_t*>(base + bm->off_pair_order);
  v.qcount = reinterpret_cast<int32_t*>(base + bm->off_qcount);
  v.qoff = reinterpret_cast<int32_t*>(base + bm->off_qoff);
  v.qidx = reinterpret_cast<int32_t*>(base + bm->off_qidx);
  v.qlabel = reinterpret_cast<uint8_t*>(base + bm->off_qlabel);
  v.korder = reinterpret_cast<int32_t*>(base + bm->off_korder);
  v.cu = bm->cu_seqlens;
  v.max_qt = bm->max_qtiles;
  v.max_nt = bm->max_ktiles;
  v.batch = bm->batch;
  v.total_tokens = bm->total_tokens;
  v.max_seqlen = bm->max_seqlen;
  return v;
}

// The duplicated-answer kind reserves role codes 2 (ANSWER) and 3
// (ANSWER_HISTORY); THINK must be another code.
bool role_think_valid(int kind, const attn_mask_params* params) {
  const int rt = params ? params->role_think : 1;
  return kind != ATTN_MASK_STRIP_THINKING_DUP || (rt != 2 && rt != 3);
}

// ATTN_MASK_DENSE needs its bit rows and offsets (8-byte aligned offsets).
bool dense_valid(int kind, const attn_mask_params* params) {
  if (kind != ATTN_MASK_DENSE) return true;
  return params && params->dense_bits && params->dense_offsets &&
         (reinterpret_cast<uintptr_t>(params->dense_bits) & 3u) == 0 &&
         (reinterpret_cast<uintptr_t>(params->dense_offsets) & 7u) == 0;
}

// A DENSE mask is used with the bits it was built from.
static bool dense_matches(int kind, const attn_mask_params* params, const attn_block_mask* bm) {
  if (kind != ATTN_MASK_DENSE) return true;
  return params && params->dense_bits == bm->dense_bits && params->dense_offsets == bm->dense_offsets;
}

static bool valid_kind(int kind) { return kind >= ATTN_MASK_CAUSAL && kind <= ATTN_MASK_DENSE; }

static bool metadata_present(int kind, const int32_t* seg, const int8_t* role, const int32_t* turn) {
  switch (kind) {
    case ATTN_MASK_CAUSAL_DOCUMENT:
    case ATTN_MASK_SHARED_PREFIX: return seg != nullptr;
    case ATTN_MASK_STRIP_THINKING:
    case ATTN_MASK_STRIP_THINKING_DUP: return role != nullptr && turn != nullptr;
    default: return true;
  }
}

}  // namespace attnmask

using namespace attnmask;

extern "C" {

int32_t attn_version(void) { return 100; }

const char* attn_last_error_message(void) { return g_last_error; }

const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case ATTN_ERR_MASK_MISMATCH: return "block mask does not match the call";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_DEVICE_TIMEOUT: return "a kernel pipeline wait timed out";
    case ATTN_ERR_DEVICE_INVALID_INPUT: return "device found malformed cu_seqlens";
  }
  return "unknown status";
}

attn_status attn_block_mask_workspace_size(int32_t batch, int32_t total_tokens,
                                           int32_t max_seqlen, int32_t block_m,
                                           int32_t block_n, size_t* bytes) {
  if (bytes == nullptr) return ATTN_ERR_INVALID_ARG;
  if (block_m != kTile || block_n != kTile) return ATTN_ERR_UNSUPPORTED;
  BmLayout l;
  if (batch < 1 || !bm_layout(batch, total_tokens, max_seqlen, &l)) return ATTN_ERR_INVALID_ARG;
  *bytes = size_t(l.total);
  return ATTN_OK;
}

attn_status attn_block_mask_build(attn_mask_kind kind, const attn_mask_params* params,
                                  const int32_t* cu_seqlens, int32_t batch,
                                  int32_t total_tokens, int32_t max_seqlen,
                                  const int32_t* seg_id, const int8_t* role,
                                  const int32_t* turn, int32_t block_m, int32_t block_n,
                                  void* workspace, size_t workspace_bytes,
                                  attn_block_mask* out, attn_stream_t stream) {
  if (out == nullptr || cu_seqlens == nullptr || workspace == nullptr) return ATTN_ERR_INVALID_ARG;
  if (!valid_kind(kind) || batch < 1 || total_tokens < 0 || max_seqlen < 0) return ATTN_ERR_INVALID_ARG;
  if (block_m != kTile || block_n != kTile) return ATTN_ERR_UNSUPPORTED;
  if (!metadata_present(kind, seg_id, role, turn)) return ATTN_ERR_INVALID_ARG;
  if (!role_think_valid(kind, params) || !dense_valid(kind, params)) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ATTN_ERR_INVALID_ARG;
  BmLayout l;
  if (!bm_layout(batch, total_tokens, max_seqlen, &l)) return ATTN_ERR_INVALID_ARG;
  if (workspace_bytes < l.total) return ATTN_ERR_WORKSPACE_TOO_SMALL;

  attn_block_mask bm;
  std::memset(&bm, 0, sizeof(bm));
  bm.magic = kMaskMagic;
  bm.kind = kind;
  bm.role_think = params ? params->role_think : 1;
  if (kind == ATTN_MASK_DENSE) {
    bm.dense_bits = params->dense_bits;
    bm.dense_offsets = params->dense_offsets;
  }
  bm.batch = batch;
  bm.total_tokens = total_tokens;
  bm.max_seqlen = max_seqlen;
  bm.block_m = block_m;
  bm.block_n = block_n;
  bm.max_qtiles = l.max_qt;
  bm.max_ktiles = l.max_nt;
  bm.cu_seqlens = cu_seqlens;
  bm.workspace = workspace;
  bm.workspace_bytes = workspace_bytes;
  bm.off_header = l.header;
  bm.off_qt_seq = l.qt_seq;
  bm.off_qt_idx = l.qt_idx;
  bm.off_labels = l.labels;
  bm.off_kcount = l.kcount;
  bm.off_koff = l.koff;
  bm.off_kidx = l.kidx;
  bm.off_klabel = l.klabel;
  bm.off_order = l.order;
  bm.off_qt_off = l.qt_off;
  bm.off_summary = l.summary;
  bm.off_pair_off = l.pair_off;
  bm.off_pair_q0 = l.pair_q0;
  bm.off_pair_order = l.pair_order;
  bm.off_qcount = l.qcount;
  bm.off_qoff = l.qoff;
  bm.off_qidx = l.qidx;
  bm.off_qlabel = l.qlabel;
  bm.off_korder = l.korder;

  MaskArgs m{kind, bm.role_think, seg_id, role, turn, bm.dense_bits, bm.dense_offsets};
  cudaError_t e = launch_block_mask_build(make_view(&bm), m, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return record_cuda_error(e, "attn_block_mask_build launch");
  *out = bm;
  return ATTN_OK;
}

attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                     attn_dtype dtype, int32_t total_tokens, int32_t num_heads,
                     int32_t head_dim, float scale, const int32_t* cu_seqlens,
                     int32_t batch, int32_t max_seqlen, attn_mask_kind kind,
                     const attn_mask_params* params, const int32_t* seg_id,
                     const int8_t* role, const int32_t* turn, const attn_block_mask* bm,
                     attn_stream_t stream) {
  if (!q || !k || !v || !o || !lse || !cu_seqlens || !bm) return ATTN_ERR_INVALID_ARG;
  if (!valid_kind(kind) || total_tokens < 0 || num_heads < 1 || batch < 1) return ATTN_ERR_INVALID_ARG;
  if (!(std::isfinite(scale)) || scale < 0.f) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_DTYPE_BF16 && dtype != ATTN_DTYPE_FP32) return ATTN_ERR_INVALID_ARG;
  if (head_dim != 32 && head_dim != 64 && head_dim != 128) return ATTN_ERR_UNSUPPORTED;
  if (!metadata_present(kind, seg_id, role, turn)) return ATTN_ERR_INVALID_ARG;
  for (const void* p : {q, k, v, static_cast<const void*>(o)})
    if ((reinterpret_cast<uintptr_t>(p) & 15u) != 0) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return ATTN_ERR_INVALID_ARG;
  const int role_think = params ? params->role_think : 1;
  if (bm->magic != kMaskMagic || bm->kind != kind || bm->cu_seqlens != cu_seqlens ||
      bm->batch != batch || bm->total_tokens != total_tokens || bm->max_seqlen != max_seqlen ||
      bm->role_think != role_think || bm->block_m != kTile || bm->block_n != kTile ||
      !dense_matches(kind, params, bm))
    return ATTN_ERR_MASK_MISMATCH;
  if (uint64_t(total_tokens) * uint64_t(num_heads) * uint64_t(head_dim) > (uint64_t(1) << 40))
    return ATTN_ERR_UNSUPPORTED;
  if (total_tokens == 0) return ATTN_OK;

  FwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.total_tokens = total_tokens;
  a.num_heads = num_heads;
  a.head_dim = head_dim;
  a.scale = scale > 0.f ? scale : 1.0f / std::sqrt(float(head_dim));
  a.bm = make_view(bm);
  a.mask = MaskArgs{kind, role_think, seg_id, role, turn, bm->dense_bits, bm->dense_offsets};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return dtype == ATTN_DTYPE_BF16 ? launch_attn_fwd_bf16(a, s) : launch_attn_fwd_f32(a, s);
}

attn_status attn_bwd_workspace_size(const attn_block_mask* bm, int32_t num_heads, int32_t head_dim,
                                    size_t* bytes) {
  if (bm == nullptr || bytes == nullptr || num_heads < 1) return ATTN_ERR_INVALID_ARG;
  if (head_dim != 32 && head_dim != 64 && head_dim != 128) return ATTN_ERR_UNSUPPORTED;
  BwdLayout l;
  if (!bwd_layout(bm->batch, bm->total_tokens, num_heads, head_dim, bm->max_qtiles, &l))
    return ATTN_ERR_INVALID_ARG;
  if (l.total > uint64_t(SIZE_MAX)) return ATTN_ERR_INVALID_ARG;
  *bytes = size_t(l.total);
  return ATTN_OK;
}

attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, attn_dtype dtype,
                     int32_t total_tokens, int32_t num_heads, int32_t head_dim, float scale,
                     const int32_t* cu_seqlens, int32_t batch, int32_t max_seqlen,
                     attn_mask_kind kind, const attn_mask_params* params, const int32_t* seg_id,
                     const int8_t* role, const int32_t* turn, const attn_block_mask* bm,
                     void* workspace, size_t workspace_bytes, attn_stream_t stream) {
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !cu_seqlens || !bm || !workspace)
    return ATTN_ERR_INVALID_ARG;
  if (!valid_kind(kind) || total_tokens < 0 || num_heads < 1 || batch < 1) return ATTN_ERR_INVALID_ARG;
  if (!(std::isfinite(scale)) || scale < 0.f) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_DTYPE_BF16 && dtype != ATTN_DTYPE_FP32) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_DTYPE_BF16) return ATTN_ERR_UNSUPPORTED;
  if (head_dim != 32 && head_dim != 64 && head_dim != 128) return ATTN_ERR_UNSUPPORTED;
  if (!metadata_present(kind, seg_id, role, turn)) return ATTN_ERR_INVALID_ARG;
  for (const void* p : {q, k, v, o, dout, static_cast<const void*>(dq), static_cast<const void*>(dk),
                        static_cast<const void*>(dv)})
    if ((reinterpret_cast<uintptr_t>(p) & 15u) != 0) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0 || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return ATTN_ERR_INVALID_ARG;
  const int role_think = params ? params->role_think : 1;
  if (bm->magic != kMaskMagic || bm->kind != kind || bm->cu_seqlens != cu_seqlens ||
      bm->batch != batch || bm->total_tokens != total_tokens || bm->max_seqlen != max_seqlen ||
      bm->role_think != role_think || bm->block_m != kTile || bm->block_n != kTile ||
      !dense_matches(kind, params, bm))
    return ATTN_ERR_MASK_MISMATCH;
  if (uint64_t(total_tokens) * uint64_t(num_heads) * uint64_t(head_dim) > (uint64_t(1) << 40))
    return ATTN_ERR_UNSUPPORTED;
  BwdLayout l;
  if (!bwd_layout(batch, total_tokens, num_heads, head_dim, bm->max_qtiles, &l)) return ATTN_ERR_INVALID_ARG;
  if (uint64_t(workspace_bytes) < l.total) return ATTN_ERR_WORKSPACE_TOO_SMALL;
  if (total_tokens == 0) return ATTN_OK;

  BwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.workspace = workspace;
  a.ws = l;
  a.total_tokens = total_tokens;
  a.num_heads = num_heads;
  a.head_dim = head_dim;
  a.scale = scale > 0.f ? scale : 1.0f / std::sqrt(float(head_dim));
  a.bm = make_view(bm);
  a.mask = MaskArgs{kind, role_think, seg_id, role, turn, bm->dense_bits, bm->dense_offsets};
  return launch_attn_bwd_bf16(a, reinterpret_cast<cudaStream_t>(stream));
}

attn_status attn_get_status(const attn_block_mask* bm, attn_stream_t stream) {
  if (bm == nullptr || bm->magic != kMaskMagic) return ATTN_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return record_cuda_error(e, "attn_get_status synchronize");
  int32_t err = 0;
  const char* base = static_cast<const char*>(bm->workspace);
  e = cudaMemcpy(&err, base + bm->off_header + sizeof(int32_t) * kHdrError, sizeof(err),
                 cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return record_cuda_error(e, "attn_get_status read");
  e = cudaGetLastError();
  if (e != cudaSuccess) return record_cuda_error(e, "attn_get_status");
  if (err & kErrTimeout) return ATTN_ERR_DEVICE_TIMEOUT;
  if (err & kErrInputMask) return ATTN_ERR_DEVICE_INVALID_INPUT;
  return ATTN_OK;
}

}  // extern "C"
