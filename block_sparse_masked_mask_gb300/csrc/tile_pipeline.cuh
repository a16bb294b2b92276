// Pieces shared by the tcgen05 attention kernels: bounded mbarrier waits, the
// 128-row bf16 tile layout in shared memory (TMA-swizzled row chunks) with its
// MMA operand descriptors, the two MMA shapes (scores and P.V-like
// products), tensor-map encoding, and the mask-code helpers.
#pragma once

#include <atomic>

#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "ptx.cuh"

// Bound on one pipeline wait.  A build may lower it (-DATTN_WAIT_TIMEOUT_NS=...)
// to make ordinary waits run out and exercise the abort path; the library
// itself uses 1 s, far above any legitimate wait.
#ifndef ATTN_WAIT_TIMEOUT_NS
#define ATTN_WAIT_TIMEOUT_NS 1000000000ull
#endif

namespace attnmask {
namespace {

constexpr uint64_t kWaitTimeoutNs = ATTN_WAIT_TIMEOUT_NS;
constexpr uint64_t kDrainTimeoutNs = 200000000ull;  // bound on waiting for in-flight work

// Work counters of the persistent kernels.  Each launch takes one slot of a
// small per-device pool (file scope, so every translation unit that includes
// this header has its own): [0] the next work ticket, [1] the CTAs that have
// finished.  The last CTA of a launch returns its slot to zero.  Because the
// counters belong to the launch, not to the block mask, launches that share a
// mask may overlap on the GPU; two launches collide only if more than
// kSchedSlots launches of one translation unit's kernels are in flight on a
// device at once.
constexpr int kSchedSlots = 256;
__device__ int32_t g_sched[kSchedSlots][2] = {};

// Host: the slot of the next launch (round robin).
inline int next_sched_slot() {
  static std::atomic<uint32_t> next{0};
  return int(next.fetch_add(1u, std::memory_order_relaxed) % uint32_t(kSchedSlots));
}

__device__ __forceinline__ int take_ticket(int slot) { return atomicAdd(&g_sched[slot][0], 1); }

// Called once per CTA (one thread) after its last ticket: every CTA has taken
// its last ticket before it counts itself finished, so the last one can
// return both counters to zero for the next launch using the slot.
__device__ __forceinline__ void finish_sched(int slot) {
  __threadfence();
  if (atomicAdd(&g_sched[slot][1], 1) == int(gridDim.x) - 1) {
    atomicExch(&g_sched[slot][0], 0);
    atomicExch(&g_sched[slot][1], 0);
  }
}

// Launch settings, queried on every launch for the current device (cheap
// runtime calls): they then follow the caller across devices and threads.
inline cudaError_t current_sm_count(int* n) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev);
  return e;
}

// A 128-row x D bf16 tile as TMA writes it: D split into row chunks of 128 B
// (64 B for D = 32), each chunk 128 rows with the matching swizzle.
template <int D>
struct TileLayout {
  static constexpr int CE = D >= 64 ? 64 : 32;        // bf16 elements per swizzled row chunk
  static constexpr int ROWB = CE * 2;                 // bytes per row chunk (128 or 64)
  static constexpr int NCH = D / CE;                  // row chunks per tile
  static constexpr int CHUNK = kTile * ROWB;          // bytes of one chunk of a 128-row tile
  static constexpr int TILE = NCH * CHUNK;            // 128 x D bf16
  static constexpr uint32_t SW = D >= 64 ? ptx::kSwizzle128B : ptx::kSwizzle64B;
  static constexpr int SBO = 8 * ROWB;                // 8-row core-matrix group stride
  // M = 128 x N = 128 scores (both operands K-major) and M = 128 x N = D
  // products whose B operand is MN-major (P.V and its kin)
  static constexpr uint32_t IDESC_S = ptx::idesc_bf16_f32(128, 128, false, false);
  static constexpr uint32_t IDESC_PV = ptx::idesc_bf16_f32(128, D, false, true);
};

// Bounded wait on an mbarrier phase.  Returns false when this CTA is aborting.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                         int32_t* err, int site) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((i & 15u) == 0) {
      if (*abort_flag) return false;
      if (ptx::globaltimer() - t0 > kWaitTimeoutNs) {
        *abort_flag = 1u;
        atomicOr(err, kErrTimeout | (site << 9));
        return false;
      }
    }
  }
}

// The same, agreed by the whole warp: every lane waits, and the warp goes on only
// if all lanes saw the phase (keeps later .sync.aligned instructions convergent).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                          int32_t* err, int site) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, err, site));
}

// One arrival for the whole warp: every lane's earlier memory and tensor-memory
// operations are ordered before it by the warp barrier (each lane issues its
// own fences first), and one shared-memory atomic replaces 32 on a word that
// other warps arrive on too.
__device__ __forceinline__ void warp_arrive(uint32_t bar, int lane) {
  __syncwarp();
  if (lane == 0) ptx::mbar_arrive(bar);
}

// Bounded wait that ignores the abort flag: used to let copies and MMAs this
// CTA issued finish before it frees shared and tensor memory.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity, int32_t* err) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > kDrainTimeoutNs) {
      atomicOr(err, kErrTimeout);
      return;
    }
  }
}

__device__ __forceinline__ uint32_t prefix_bits(int n) {
  return n <= 0 ? 0u : (n >= 32 ? 0xffffffffu : ((1u << n) - 1u));
}

// Visibility bits of keys [32q, 32q+32) of a k-tile for one query code, from
// the keys' codes the producer staged in shared memory.
template <int KIND>
__device__ __forceinline__ uint32_t code_word(const int* codes, int q, int qcode) {
  uint32_t w = 0;
  const int4* c4 = reinterpret_cast<const int4*>(codes + 32 * q);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const int4 k = c4[c];
    w |= (uint32_t(code_visible(KIND, qcode, k.x)) << (4 * c)) |
         (uint32_t(code_visible(KIND, qcode, k.y)) << (4 * c + 1)) |
         (uint32_t(code_visible(KIND, qcode, k.z)) << (4 * c + 2)) |
         (uint32_t(code_visible(KIND, qcode, k.w)) << (4 * c + 3));
  }
  return w;
}

// The same for a kind known only at run time, as a compact loop, for kinds
// whose rows rarely hold different codes: it keeps the hot loop around it
// small enough for the instruction cache.
__device__ __forceinline__ uint32_t code_word_rt(int kind, const int* codes, int q, int qcode) {
  uint32_t w = 0;
  const int4* c4 = reinterpret_cast<const int4*>(codes + 32 * q);
#pragma unroll 1
  for (int c = 0; c < 8; ++c) {
    const int4 k = c4[c];
    w |= (uint32_t(code_visible(kind, qcode, k.x)) << (4 * c)) |
         (uint32_t(code_visible(kind, qcode, k.y)) << (4 * c + 1)) |
         (uint32_t(code_visible(kind, qcode, k.z)) << (4 * c + 2)) |
         (uint32_t(code_visible(kind, qcode, k.w)) << (4 * c + 3));
  }
  return w;
}

// Shared-memory descriptors: one base per tile; each k-step adds a constant to
// the start-address field (addresses stay below 2^18, so no carry leaves it).
// K-major operand (Q or K): k-step kk covers elements [16kk, 16kk+16) of D.
template <int D>
__device__ __forceinline__ uint64_t kmajor_base(uint32_t tile_addr) {
  using C = TileLayout<D>;
  return ptx::smem_desc(tile_addr, 16u, C::SBO, C::SW);
}
template <int D>
__host__ __device__ constexpr uint64_t kmajor_step(int kk) {
  using C = TileLayout<D>;
  return uint64_t(((16 * kk) / C::CE) * C::CHUNK + ((16 * kk) % C::CE) * 2) >> 4;
}
// MN-major operand V (N = D across chunks, K = keys): k-step kk covers keys [16kk, 16kk+16).
template <int D>
__device__ __forceinline__ uint64_t v_base(uint32_t tile_addr) {
  using C = TileLayout<D>;
  return ptx::smem_desc(tile_addr, C::CHUNK, C::SBO, C::SW);
}
template <int D>
__host__ __device__ constexpr uint64_t v_step(int kk) {
  using C = TileLayout<D>;
  return uint64_t(kk * 16 * C::ROWB) >> 4;
}


template <int D>
__device__ __forceinline__ void issue_s(uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc) {
  using C = TileLayout<D>;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk)
    ptx::mma_ss(d_tmem, q_desc + kmajor_step<D>(kk), k_desc + kmajor_step<D>(kk), C::IDESC_S, kk > 0);
}

// O += P V over the 128 keys of a k-tile: P (bf16) of keys 0-63 sits over the
// first 32 columns of the S buffer, P of keys 64-127 over columns 64-95 (each
// half writes P over its own score columns); eight k-steps of 16 keys.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t s_tmem, uint64_t v_desc, bool acc) {
  using C = TileLayout<D>;
#pragma unroll
  for (int kk = 0; kk < kTile / 16; ++kk)
    ptx::mma_ts(d_tmem, s_tmem + uint32_t(kk >> 2) * 64u + uint32_t(kk & 3) * 8u, v_desc + v_step<D>(kk),
                C::IDESC_PV, (acc || kk > 0) ? 1u : 0u);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// [T, H, D] bf16 viewed as a 3-D tensor (d, h, t); box = one swizzled row chunk x 128 tokens.
template <int D>
bool make_map(CUtensorMap* m, const void* ptr, int T, int H) {
  using C = TileLayout<D>;
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(H), cuuint64_t(T)};
  cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(H) * D * 2};
  cuuint32_t box[3] = {cuuint32_t(C::CE), 1, cuuint32_t(kTile)};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle sw = D >= 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


}  // namespace
}  // namespace attnmask
