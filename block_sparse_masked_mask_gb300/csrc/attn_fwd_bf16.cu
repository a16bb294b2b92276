// bf16 attention forward on the sm_103a tensor cores (tcgen05 + TMA + TMEM).
//
// The loop is the online-softmax flash attention of "Triton from first
// principles" Ch. 21, Section 21.1 (running max m, running sum l, accumulator
// rescaled by alpha = exp(m_old - m_new), one division at the end), with the
// causal / structured mask applied inside the loop as in Section 21.2, and
// only the k-tiles the block mask lists for a q-tile are visited (Ch. 9,
// Section 9.2: a skipped tile is never loaded).
//
// One CTA handles one (q-tile of 128 rows, head) work item.  Warp roles:
//   warp 0     TMA producer: Q once, then K and V tiles of the listed k-tiles
//              into a 2-stage shared-memory ring; key mask codes for PARTIAL
//              tiles.
//   warp 1     tcgen05 issuer (one thread): S = Q K^T into one of two TMEM
//              score buffers, then O += P V with P read from TMEM.
//   warps 2-5  softmax: one thread per query row.  Each thread reads its row
//              of S from TMEM, applies the mask (PARTIAL tiles: predicate and
//              bounds; FULL tiles: bounds only on a ragged last tile), updates
//              m and l, rescales its row of O in TMEM when m grew, writes P as
//              bf16 over the first half of its S row, and finally writes
//              O / l and LSE.
// TMEM columns: S0 [0,128), S1 [128,256), O [256, 256+D).
// Every mbarrier wait is bounded: on timeout the CTA records kErrTimeout in
// the block-mask error word, drains what it issued, frees TMEM and exits.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "ptx.cuh"

namespace attnmask {
namespace {

constexpr uint64_t kWaitTimeoutNs = 1000000000ull;  // 1 s: far above any legitimate wait
constexpr uint64_t kDrainTimeoutNs = 200000000ull;  // bound on waiting for in-flight copies

template <int D>
struct Cfg {
  static constexpr int NST = 2;                       // K/V ring stages
  static constexpr int CE = D >= 64 ? 64 : 32;        // bf16 elements per swizzled row chunk
  static constexpr int ROWB = CE * 2;                 // bytes per row chunk (128 or 64)
  static constexpr int NCH = D / CE;                  // row chunks per tile
  static constexpr int CHUNK = kTile * ROWB;          // bytes of one chunk of a 128-row tile
  static constexpr int TILE = NCH * CHUNK;            // 128 x D bf16
  static constexpr uint32_t SW = D >= 64 ? ptx::kSwizzle128B : ptx::kSwizzle64B;
  static constexpr int SBO = 8 * ROWB;                // 8-row core-matrix group stride
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + TILE;
  static constexpr int OFF_V = OFF_K + NST * TILE;
  static constexpr int OFF_KCODE = OFF_V + NST * TILE;
  // barriers: q, kfull[NST], vfull[NST], empty[NST], sfull[2], pfull[2], odone, drain
  static constexpr int B_Q = 0, B_KFULL = 1, B_VFULL = 1 + NST, B_EMPTY = 1 + 2 * NST,
                       B_SFULL = 1 + 3 * NST, B_PFULL = B_SFULL + 2, B_ODONE = B_PFULL + 2,
                       B_DRAIN = B_ODONE + 1, NBAR = B_DRAIN + 1;
  static constexpr int OFF_BAR = OFF_KCODE + NST * kTile * 4;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_USED = OFF_MISC + 16;
  // + slack to align the base to 1024 B; at least 116 KB so that one CTA holds an SM
  // (and its 512 TMEM columns) alone.
  static constexpr int SMEM_ALLOC = SMEM_USED + 1024 > 116 * 1024 ? SMEM_USED + 1024 : 116 * 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S0 = 0, COL_O = 256;
  static constexpr uint32_t IDESC_S = ptx::idesc_bf16_f32(128, 128, false, false);
  static constexpr uint32_t IDESC_PV = ptx::idesc_bf16_f32(128, D, false, true);
  static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
};

struct FwdParams {
  int32_t* header;
  const int32_t* order;
  const int32_t* qt_seq;
  const int32_t* qt_idx;
  const int32_t* koff;
  const int32_t* kidx;
  const uint8_t* klabel;
  const int32_t* cu;
  MaskArgs mask;
  __nv_bfloat16* o;
  float* lse;
  int H, T;
  float scale_log2;  // scale * log2(e)
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

// Visibility bits of 32 consecutive keys (codes in shared memory) for one query code.
template <int KIND>
__device__ __forceinline__ uint32_t code_word(const int* kc, int qcode) {
  uint32_t w = 0;
#pragma unroll
  for (int c = 0; c < 32; c += 4) {
    const int4 k = *reinterpret_cast<const int4*>(kc + c);
    w |= (uint32_t(code_visible(KIND, qcode, k.x)) << c) | (uint32_t(code_visible(KIND, qcode, k.y)) << (c + 1)) |
         (uint32_t(code_visible(KIND, qcode, k.z)) << (c + 2)) | (uint32_t(code_visible(KIND, qcode, k.w)) << (c + 3));
  }
  return w;
}

// K-major operand (Q or K): k-step kk covers elements [16kk, 16kk+16) of D.
template <int D>
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile_addr, int kk) {
  using C = Cfg<D>;
  const uint32_t e = uint32_t(kk) * 16u;
  const uint32_t addr = tile_addr + (e / C::CE) * C::CHUNK + (e % C::CE) * 2u;
  return ptx::smem_desc(addr, 16u, C::SBO, C::SW);
}

// MN-major operand V (N = D across chunks, K = keys): k-step kk covers keys [16kk, 16kk+16).
template <int D>
__device__ __forceinline__ uint64_t v_desc(uint32_t tile_addr, int kk) {
  using C = Cfg<D>;
  const uint32_t addr = tile_addr + uint32_t(kk) * 16u * C::ROWB;
  return ptx::smem_desc(addr, C::CHUNK, C::SBO, C::SW);
}

template <int D>
__global__ void __launch_bounds__(192, 1)
    attn_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int n_qt = p.header[kHdrQtiles];
  const int item = blockIdx.x;
  if (item >= n_qt * p.H) return;
  int32_t* err = p.header + kHdrError;

  const int h = item / n_qt;
  const int g = p.order[item % n_qt];
  const int b = p.qt_seq[g], qa = p.qt_idx[g];
  const int s0 = p.cu[b], L = p.cu[b + 1] - s0;
  const int i0 = qa * kTile;                  // first query row, local to the sequence
  const int qn = min(kTile, L - i0);
  const int e0 = p.koff[g], n = p.koff[g + 1] - e0;

  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);
  const uint32_t sQ = base + C::OFF_Q, sK = base + C::OFF_K, sV = base + C::OFF_V;
  int* kcode = reinterpret_cast<int*>(sbase + C::OFF_KCODE);
  const uint32_t bars = base + C::OFF_BAR;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  uint32_t* misc = reinterpret_cast<uint32_t*>(sbase + C::OFF_MISC);
  volatile uint32_t* abort_flag = misc + 1;

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(C::B_Q), 1);
    for (int s = 0; s < C::NST; ++s) {
      ptx::mbar_init(bar(C::B_KFULL + s), 1);
      ptx::mbar_init(bar(C::B_VFULL + s), 1);
      ptx::mbar_init(bar(C::B_EMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(bar(C::B_SFULL + s), 1);
      ptx::mbar_init(bar(C::B_PFULL + s), 128);
    }
    ptx::mbar_init(bar(C::B_ODONE), 1);
    ptx::mbar_init(bar(C::B_DRAIN), 1);
    // An earlier CTA that gave up on a wait makes every later one skip its work.
    *abort_flag = (*reinterpret_cast<volatile int32_t*>(err) & kErrTimeout) ? 1u : 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(misc), C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = misc[0];
  const bool skip = *abort_flag != 0u;

  if (skip) {
    // nothing issued, nothing to drain
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    int n_issued = 0;
    const bool need_codes = p.mask.kind != ATTN_MASK_CAUSAL;
    if (lane == 0) {
      ptx::prefetch_tensormap(&tmQ);
      ptx::prefetch_tensormap(&tmK);
      ptx::prefetch_tensormap(&tmV);
      ptx::mbar_arrive_expect_tx(bar(C::B_Q), C::TILE);
      for (int c = 0; c < C::NCH; ++c)
        ptx::tma_load_3d(sQ + c * C::CHUNK, &tmQ, bar(C::B_Q), c * C::CE, h, s0 + i0);
    }
    for (int it = 0; it < n; ++it) {
      const int st = it % C::NST;
      const uint32_t ph = uint32_t(it / C::NST) & 1u;
      if (it >= C::NST && !warp_wait(bar(C::B_EMPTY + st), ph ^ 1u, abort_flag, err, 1)) break;
      const int kt = p.kidx[e0 + it];
      const int lab = p.klabel[e0 + it];
      const int j0 = kt * kTile;
      if (need_codes && lab == ATTN_TILE_PARTIAL) {
        for (int c = lane; c < kTile; c += 32)
          kcode[st * kTile + c] = (j0 + c < L) ? key_code(p.mask, s0 + j0 + c) : 0;
      }
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(bar(C::B_KFULL + st), C::TILE);
        for (int c = 0; c < C::NCH; ++c)
          ptx::tma_load_3d(sK + st * C::TILE + c * C::CHUNK, &tmK, bar(C::B_KFULL + st), c * C::CE,
                           h, s0 + j0);
        ptx::mbar_arrive_expect_tx(bar(C::B_VFULL + st), C::TILE);
        for (int c = 0; c < C::NCH; ++c)
          ptx::tma_load_3d(sV + st * C::TILE + c * C::CHUNK, &tmV, bar(C::B_VFULL + st), c * C::CE,
                           h, s0 + j0);
      }
      n_issued = it + 1;
    }
    // Do not leave while a load this CTA issued may still be writing shared memory.
    if (lane == 0) {
      for (int s = 0; s < C::NST; ++s) {
        if (n_issued <= s) continue;
        const int last = s + C::NST * ((n_issued - 1 - s) / C::NST);  // last load into stage s
        const uint32_t ph = uint32_t(last / C::NST) & 1u;
        drain_bar(bar(C::B_KFULL + s), ph, err);
        drain_bar(bar(C::B_VFULL + s), ph, err);
      }
      drain_bar(bar(C::B_Q), 0, err);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = wait_bar(bar(C::B_Q), 0, abort_flag, err, 3);
      for (int it = 0; ok && it <= n; ++it) {
        if (it < n) {
          const int st = it % C::NST;
          if (!wait_bar(bar(C::B_KFULL + st), uint32_t(it / C::NST) & 1u, abort_flag, err, 4)) break;
          ptx::tc_fence_after();
          const uint32_t dS = tmem + C::COL_S0 + uint32_t(it & 1) * 128u;
          const uint32_t kb = sK + st * C::TILE;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            ptx::mma_ss(dS, kmajor_desc<D>(sQ, kk), kmajor_desc<D>(kb, kk), C::IDESC_S, kk > 0);
          ptx::mma_commit(bar(C::B_SFULL + (it & 1)));
        }
        if (it >= 1) {
          const int j = it - 1, st = j % C::NST;
          if (!wait_bar(bar(C::B_PFULL + (j & 1)), uint32_t(j >> 1) & 1u, abort_flag, err, 5)) break;
          if (!wait_bar(bar(C::B_VFULL + st), uint32_t(j / C::NST) & 1u, abort_flag, err, 6)) break;
          ptx::tc_fence_after();
          const uint32_t aP = tmem + C::COL_S0 + uint32_t(j & 1) * 128u;
          const uint32_t vb = sV + st * C::TILE;
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            ptx::mma_ts(tmem + C::COL_O, aP + uint32_t(kk) * 8u, v_desc<D>(vb, kk), C::IDESC_PV,
                        (j > 0 || kk > 0) ? 1u : 0u);
          ptx::mma_commit(bar(C::B_EMPTY + st));
          ptx::mma_commit(bar(C::B_ODONE));
        }
      }
      // Every MMA issued above has finished once this commit arrives.
      ptx::mma_commit(bar(C::B_DRAIN));
      drain_bar(bar(C::B_DRAIN), 0, err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;              // TMEM lanes this warp may access
    const int r = quarter * 32 + lane;         // query row inside the tile
    const bool row_in = r < qn;
    const int il = i0 + r;                     // local query index
    const int qcode = (row_in && p.mask.kind != ATTN_MASK_CAUSAL) ? query_code(p.mask, s0 + il) : 0;
    const uint32_t lane_base = tmem + (uint32_t(quarter * 32) << 16);
    const float c2 = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int it = 0; it < n; ++it) {
      const int sb = it & 1, st = it % C::NST;
      const int kt = p.kidx[e0 + it];
      const int lab = p.klabel[e0 + it];
      const int j0 = kt * kTile;
      if (!warp_wait(bar(C::B_SFULL + sb), uint32_t(it >> 1) & 1u, abort_flag, err, 8)) { ok = false; break; }
      ptx::tc_fence_after();
      const int kn = min(kTile, L - j0);
      float s[128];
      {
        uint32_t v[4][32];
#pragma unroll
        for (int q = 0; q < 4; ++q) ptx::tmem_ld32(lane_base + C::COL_S0 + sb * 128 + q * 32, v[q]);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int c = 0; c < 32; ++c) s[q * 32 + c] = __uint_as_float(v[q][c]);
      }
      if (lab == ATTN_TILE_PARTIAL || kn < kTile) {
        // bit c of vis[c / 32]: key column c is visible to this row.  Causal part
        // and bounds together: columns c < upto.  PARTIAL tiles of the
        // metadata kinds also AND in the per-key predicate.
        const int upto = lab == ATTN_TILE_PARTIAL ? min(kn, il - j0 + 1) : kn;
        uint32_t vis[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) vis[q] = prefix_bits(upto - 32 * q);
        if (lab == ATTN_TILE_PARTIAL && p.mask.kind != ATTN_MASK_CAUSAL) {
          if (!warp_wait(bar(C::B_KFULL + st), uint32_t(it / C::NST) & 1u, abort_flag, err, 9)) { ok = false; break; }
          const int* kc = kcode + st * kTile;
          switch (p.mask.kind) {
            case ATTN_MASK_CAUSAL_DOCUMENT:
#pragma unroll
              for (int q = 0; q < 4; ++q) vis[q] &= code_word<ATTN_MASK_CAUSAL_DOCUMENT>(kc + 32 * q, qcode);
              break;
            case ATTN_MASK_SHARED_PREFIX:
#pragma unroll
              for (int q = 0; q < 4; ++q) vis[q] &= code_word<ATTN_MASK_SHARED_PREFIX>(kc + 32 * q, qcode);
              break;
            default:
#pragma unroll
              for (int q = 0; q < 4; ++q) vis[q] &= code_word<ATTN_MASK_STRIP_THINKING>(kc + 32 * q, qcode);
              break;
          }
        }
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = (vis[c >> 5] >> (c & 31)) & 1u ? s[c] : -INFINITY;
      }
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < 128; ++c) mx4[c & 3] = fmaxf(mx4[c & 3], s[c]);
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      const float m_new = fmaxf(m, mx * c2);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = ptx::ex2(m - m_use);
      float sum2[2] = {0.f, 0.f};
      uint32_t pk[2][32];
#pragma unroll
      for (int c = 0; c < 128; c += 2) {
        const float p0 = ptx::ex2(fmaf(s[c], c2, -m_use));
        const float p1 = ptx::ex2(fmaf(s[c + 1], c2, -m_use));
        sum2[(c >> 1) & 1] += p0 + p1;
        pk[c >> 6][(c & 63) >> 1] = ptx::pack_bf16(p0, p1);
      }
      const float sum = sum2[0] + sum2[1];
      l = l * alpha + sum;
      m = m_new;
      if (it > 0) {
        // O must hold exactly PV of tiles < it before it is rescaled.
        if (!warp_wait(bar(C::B_ODONE), uint32_t(it - 1) & 1u, abort_flag, err, 10)) { ok = false; break; }
        ptx::tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int q = 0; q < D / 32; ++q) {
            uint32_t v[32];
            ptx::tmem_ld32(lane_base + C::COL_O + q * 32, v);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * alpha);
            ptx::tmem_st32(lane_base + C::COL_O + q * 32, v);
          }
        }
      }
      ptx::tmem_st32(lane_base + C::COL_S0 + sb * 128, pk[0]);
      ptx::tmem_st32(lane_base + C::COL_S0 + sb * 128 + 32, pk[1]);
      if (kn < kTile) {
        // Rows past the sequence end were loaded from the next sequence (or
        // zero-filled past the tensor).  Their P is exactly 0, but 0 * inf is
        // NaN, so the V rows are zeroed before the P.V product reads them.
        if (!warp_wait(bar(C::B_VFULL + st), uint32_t(it / C::NST) & 1u, abort_flag, err, 12)) { ok = false; break; }
        if (r >= kn) {
#pragma unroll
          for (int c = 0; c < C::NCH; ++c) {
            uint4* row = reinterpret_cast<uint4*>(sbase + C::OFF_V + st * C::TILE + c * C::CHUNK + r * C::ROWB);
#pragma unroll
            for (int x = 0; x < C::ROWB / 16; ++x) row[x] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        ptx::fence_proxy_async_smem();
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(C::B_PFULL + sb));
    }
    // ------------------------------------------------------------ epilogue
    if (ok && n > 0) ok = warp_wait(bar(C::B_ODONE), uint32_t(n - 1) & 1u, abort_flag, err, 11);
    if (ok) {
      ptx::tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = p.o + (size_t(s0 + il) * p.H + h) * D;
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        uint32_t v[32];
        if (n > 0) {
          ptx::tmem_ld32(lane_base + C::COL_O + q * 32, v);
          ptx::tmem_wait_ld();
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = 0u;
        }
        uint32_t w[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          w[c] = ptx::pack_bf16(__uint_as_float(v[2 * c]) * inv_l, __uint_as_float(v[2 * c + 1]) * inv_l);
        if (row_in) {
          uint4* dst = reinterpret_cast<uint4*>(orow + q * 32);
#pragma unroll
          for (int c = 0; c < 4; ++c) dst[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
        }
      }
      if (row_in)
        p.lse[size_t(h) * p.T + s0 + il] = l > 0.f ? (m + ptx::lg2(l)) * 0.69314718055994531f : -INFINITY;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::TMEM_COLS);
  }
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
  using C = Cfg<D>;
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

template <int D>
attn_status launch(const FwdArgs& a, cudaStream_t s) {
  using C = Cfg<D>;
  CUtensorMap mq, mk, mv;
  if (!make_map<D>(&mq, a.q, a.total_tokens, a.num_heads) ||
      !make_map<D>(&mk, a.k, a.total_tokens, a.num_heads) ||
      !make_map<D>(&mv, a.v, a.total_tokens, a.num_heads))
    return ATTN_ERR_CUDA;
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(attn_fwd_bf16_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_ALLOC) != cudaSuccess)
      return ATTN_ERR_CUDA;
    configured = true;
  }
  FwdParams p;
  p.header = a.bm.header;
  p.order = a.bm.order;
  p.qt_seq = a.bm.qt_seq;
  p.qt_idx = a.bm.qt_idx;
  p.koff = a.bm.koff;
  p.kidx = a.bm.kidx;
  p.klabel = a.bm.klabel;
  p.cu = a.bm.cu;
  p.mask = a.mask;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.H = a.num_heads;
  p.T = a.total_tokens;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  const long long grid = (long long)a.bm.max_qt * a.num_heads;
  if (grid <= 0 || grid > INT_MAX) return ATTN_ERR_UNSUPPORTED;
  attn_fwd_bf16_kernel<D><<<unsigned(grid), 192, C::SMEM_ALLOC, s>>>(mq, mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

attn_status launch_attn_fwd_bf16(const FwdArgs& a, cudaStream_t s) {
  switch (a.head_dim) {
    case 32: return launch<32>(a, s);
    case 64: return launch<64>(a, s);
    case 128: return launch<128>(a, s);
  }
  return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attnmask
