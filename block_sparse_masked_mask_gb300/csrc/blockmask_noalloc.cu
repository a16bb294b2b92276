// attn_block_mask_build_noalloc: the block-mask builder for callers that
// cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: hosts whose memory manager owns every
// device byte and forbids allocations behind its back (embedded runtimes,
// fixed-footprint inference servers), and latency-critical loops where an
// allocation, with the device-wide synchronisation it may bring, is not
// allowed.  Such a caller still has the buffers it already must provide: the
// metadata inputs and the block-mask output buffer.  This entry point asks for
// nothing else.  The builder's temporary
// arrays (per-tile metadata summaries, the dense tile-label matrix and the
// per-sequence tile offsets) live instead in one file-scope device array of
// fixed size, present on every GPU that loads this library until the process
// exits.
//
// Rules of use:
//  * The scratch holds kNoallocScratchBytes (4 MiB).  A problem whose scratch
//    would not fit (max_qtiles * max_ktiles + 32 * max_qtiles + 8 * (batch + 1)
//    bytes, each part rounded up to 256 bytes) is rejected with
//    ATTN_ERR_UNSUPPORTED before anything is launched.  For one sequence that
//    is up to 259,968 tokens (2031 tiles).
//  * The first call on a device looks up the array's device address with that
//    device current (a one-time set-up).  Make that first call before any
//    stream capture.  The address is kept for the life of the process: after
//    cudaDeviceReset (or anything else that destroys and recreates the
//    device's primary context) it names memory of the old context, so a
//    process that resets a device must not call this entry point on it again.
//  * Every call on a device shares the one array and leaves its contents in
//    place.  Calls whose kernels overlap on the GPU (other streams, other host
//    threads) race on it; serialise them.  Nothing in the scratch has to start
//    at zero: every entry is written before it is read within one call.
//  * No cudaMalloc, cudaFree or other allocating call is made.
#include <mutex>
#include <cstdio>
#include <cstring>

#include "common.cuh"

namespace attnmask {
namespace {

constexpr size_t kNoallocScratchBytes = size_t(4) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_bm_scratch[kNoallocScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

uint64_t round256(uint64_t x) { return (x + 255u) & ~uint64_t(255u); }

// Device address of this device's scratch array (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_bm_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace attnmask

using namespace attnmask;

extern "C" attn_status attn_block_mask_build_noalloc(
    attn_mask_kind kind, const attn_mask_params* params, const int32_t* cu_seqlens, int32_t batch,
    int32_t total_tokens, int32_t max_seqlen, const int32_t* seg_id, const int8_t* role,
    const int32_t* turn, int32_t block_m, int32_t block_n, void* workspace, size_t workspace_bytes,
    attn_block_mask* out, attn_stream_t stream) {
  if (out == nullptr || cu_seqlens == nullptr || workspace == nullptr) return ATTN_ERR_INVALID_ARG;
  if (kind < ATTN_MASK_CAUSAL || kind > ATTN_MASK_DENSE || batch < 1 || total_tokens < 0 ||
      max_seqlen < 0)
    return ATTN_ERR_INVALID_ARG;
  if (block_m != kTile || block_n != kTile) return ATTN_ERR_UNSUPPORTED;
  if ((kind == ATTN_MASK_CAUSAL_DOCUMENT || kind == ATTN_MASK_SHARED_PREFIX) && seg_id == nullptr)
    return ATTN_ERR_INVALID_ARG;
  if ((kind == ATTN_MASK_STRIP_THINKING || kind == ATTN_MASK_STRIP_THINKING_DUP) &&
      (role == nullptr || turn == nullptr))
    return ATTN_ERR_INVALID_ARG;
  if (!role_think_valid(kind, params) || !dense_valid(kind, params)) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ATTN_ERR_INVALID_ARG;
  BmLayout l;
  if (!bm_layout(batch, total_tokens, max_seqlen, &l)) return ATTN_ERR_INVALID_ARG;
  if (workspace_bytes < l.total) return ATTN_ERR_WORKSPACE_TOO_SMALL;

  // Scratch layout inside the static array.
  const uint64_t nq = uint64_t(l.max_qt), nk = uint64_t(l.max_nt);
  const uint64_t s_labels = 0;
  const uint64_t s_summary = s_labels + round256(nq * (nk ? nk : 1));
  const uint64_t s_qt_off = s_summary + round256(4 * kSumInts * nq);
  const uint64_t s_pair_off = s_qt_off + round256(4 * (uint64_t(batch) + 1));
  const uint64_t s_total = s_pair_off + round256(4 * (uint64_t(batch) + 1));
  if (s_total > kNoallocScratchBytes) return ATTN_ERR_UNSUPPORTED;

  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) return record_cuda_error(e, "attn_block_mask_build_noalloc scratch lookup");

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
  // Output arrays at their usual workspace offsets.  The scratch arrays are not
  // kept: their offsets name workspace regions this call leaves unwritten.
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

  char* base = static_cast<char*>(workspace);
  char* sbase = static_cast<char*>(scratch);
  BmView v;
  v.header = reinterpret_cast<int32_t*>(base + l.header);
  v.qt_seq = reinterpret_cast<int32_t*>(base + l.qt_seq);
  v.qt_idx = reinterpret_cast<int32_t*>(base + l.qt_idx);
  v.labels = reinterpret_cast<uint8_t*>(sbase + s_labels);
  v.kcount = reinterpret_cast<int32_t*>(base + l.kcount);
  v.koff = reinterpret_cast<int32_t*>(base + l.koff);
  v.kidx = reinterpret_cast<int32_t*>(base + l.kidx);
  v.klabel = reinterpret_cast<uint8_t*>(base + l.klabel);
  v.order = reinterpret_cast<int32_t*>(base + l.order);
  v.qt_off = reinterpret_cast<int32_t*>(sbase + s_qt_off);
  v.summary = reinterpret_cast<int32_t*>(sbase + s_summary);
  v.pair_off = reinterpret_cast<int32_t*>(sbase + s_pair_off);
  v.pair_q0 = reinterpret_cast<int32_t*>(base + l.pair_q0);
  v.pair_order = reinterpret_cast<int32_t*>(base + l.pair_order);
  v.qcount = reinterpret_cast<int32_t*>(base + l.qcount);
  v.qoff = reinterpret_cast<int32_t*>(base + l.qoff);
  v.qidx = reinterpret_cast<int32_t*>(base + l.qidx);
  v.qlabel = reinterpret_cast<uint8_t*>(base + l.qlabel);
  v.korder = reinterpret_cast<int32_t*>(base + l.korder);
  v.cu = cu_seqlens;
  v.max_qt = l.max_qt;
  v.max_nt = l.max_nt;
  v.batch = batch;
  v.total_tokens = total_tokens;
  v.max_seqlen = max_seqlen;

  MaskArgs m{kind, bm.role_think, seg_id, role, turn, bm.dense_bits, bm.dense_offsets};
  e = launch_block_mask_build(v, m, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return record_cuda_error(e, "attn_block_mask_build_noalloc launch");
  *out = bm;
  return ATTN_OK;
}
