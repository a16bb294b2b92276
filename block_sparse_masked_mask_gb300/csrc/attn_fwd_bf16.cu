// bf16 attention forward on the sm_103a tensor cores (tcgen05 + TMA + TMEM).
//
// The loop is the online-softmax flash attention of "Triton from first
// principles" Ch. 21, Section 21.1 (running max m, running sum l, accumulator
// rescaled by exp(m_old - m_new), one division at the end), with the causal /
// structured mask applied inside the loop as in Section 21.2, and only the
// k-tiles the block mask lists are visited (Ch. 9, Section 9.2: a skipped
// tile is never loaded).
//
// A work item is a pair of adjacent 128-row q-tiles of one sequence (the
// second may be absent) and one head; persistent CTAs (one per SM) loop over
// the items.  The pair walks the
// ascending union of its two k-tile lists; each K and V tile is loaded once
// and serves both q-tiles, and a q-tile skips the entries its own list does
// not hold (EMPTY for it).  Warp roles:
//   warps 0-3  softmax of q-tile 0, one thread per query row
//   warps 4-7  softmax of q-tile 1
//   warp 8     TMA producer: Q0/Q1 once, then K(j), V(j) into a ring of
//              four 128 x D slots; zeroes V rows past a sequence end
//   warps 9-10 tcgen05 issuers, one thread each: warp 9 for q-tile 0, warp 10
//              for q-tile 1 (warp 9 also owns the TMEM allocation).  They
//              take turns, PV0(j), S0(j+1) | PV1(j), S1(j+1) | ..., so the
//              tensor cores serve one q-tile while the other's softmax runs
//              (ping-pong), and each does its waits while the other issues.
//   warp 11    idle
// TMEM columns: S0 [0,128), S1 [128,256), O0 [256, 256+D), O1 [256+D, 256+2D).
// P (bf16) overwrites the first 64 columns of its S buffer.
//
// The row maximum used as the exponent reference only moves when a new tile
// raises it by more than 2^8 (factor 256 in p); O and l are then rescaled
// together, so the final O / l and LSE are unchanged in exact arithmetic.
// Every mbarrier wait is bounded: on timeout the CTA records kErrTimeout in the
// block-mask error word, drains what it issued, frees TMEM and exits.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "ptx.cuh"

namespace attnmask {
namespace {

constexpr uint64_t kWaitTimeoutNs = 1000000000ull;  // 1 s: far above any legitimate wait
constexpr uint64_t kDrainTimeoutNs = 200000000ull;  // bound on waiting for in-flight work
constexpr float kRescaleThreshold = 8.0f;           // log2 units: p stays <= 256
// 384 threads = 3 warpgroups, one warp of each on every SM sub-partition.
// Launched at kLaunchRegs per thread; the two softmax warpgroups then take
// kSoftmaxRegs and the producer / MMA warpgroup keeps kOtherRegs:
// 2 * 208 + 88 = 504 = 3 * 168, the launch budget of a sub-partition's warps.
constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168;
constexpr uint32_t kSoftmaxRegs = 208;
constexpr uint32_t kOtherRegs = 88;
static_assert(2 * kSoftmaxRegs + kOtherRegs <= 3 * kLaunchRegs, "register split exceeds the launch budget");

template <int D>
struct Cfg {
  static constexpr int NSLOT = 4;                     // K/V ring slots (one tile each)
  static constexpr int NCODE = 3;                     // key-code buffers, one per ring entry in flight
  static constexpr int CE = D >= 64 ? 64 : 32;        // bf16 elements per swizzled row chunk
  static constexpr int ROWB = CE * 2;                 // bytes per row chunk (128 or 64)
  static constexpr int NCH = D / CE;                  // row chunks per tile
  static constexpr int CHUNK = kTile * ROWB;          // bytes of one chunk of a 128-row tile
  static constexpr int TILE = NCH * CHUNK;            // 128 x D bf16
  static constexpr uint32_t SW = D >= 64 ? ptx::kSwizzle128B : ptx::kSwizzle64B;
  static constexpr int SBO = 8 * ROWB;                // 8-row core-matrix group stride
  static constexpr int OFF_Q0 = 0, OFF_Q1 = TILE, OFF_RING = 2 * TILE;
  static constexpr int B_Q = 0, B_QFREE = 1, B_FULL = 2, B_EMPTY = 2 + NSLOT, B_VTMA = 2 + 2 * NSLOT,
                       B_SFULL = B_VTMA + 1, B_PFULL = B_SFULL + 2, B_ODONE = B_PFULL + 2,
                       B_OFREE = B_ODONE + 2, B_IFULL = B_OFREE + 2, B_IEMPTY = B_IFULL + 2,
                       B_DRAIN = B_IEMPTY + 2, B_TURN = B_DRAIN + 1, B_CODE = B_TURN + 2, NBAR = B_CODE + NCODE;
  static constexpr int OFF_BAR = OFF_RING + NSLOT * TILE;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int OFF_RINGI = OFF_MISC + 16;    // two decoded work items, 8 ints each
  static constexpr int OFF_SINFO = OFF_RINGI + 2 * 8 * 4;  // per ring slot: labels / has-next
  static constexpr int OFF_CODES = (OFF_SINFO + NSLOT * 4 + 15) & ~15;  // per buffer: 128 key codes
  static constexpr int SMEM_USED = OFF_CODES + NCODE * kTile * 4;
  // + slack to align the base to 1024 B; at least 116 KB so that one CTA holds an SM
  // (and its 512 TMEM columns) alone.
  static constexpr int SMEM_ALLOC = SMEM_USED + 1024 > 116 * 1024 ? SMEM_USED + 1024 : 116 * 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t IDESC_S = ptx::idesc_bf16_f32(128, 128, false, false);
  static constexpr uint32_t IDESC_PV = ptx::idesc_bf16_f32(128, D, false, true);
  __host__ __device__ static constexpr uint32_t col_s(int t) { return uint32_t(t) * 128u; }
  __host__ __device__ static constexpr uint32_t col_o(int t) { return 256u + uint32_t(t) * D; }
  static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
};

struct FwdParams {
  int32_t* header;
  const int32_t* pair_order;
  const int32_t* pair_q0;
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

// Ascending union of the two q-tiles' k-tile lists, with each q-tile's label
// (EMPTY where its own list lacks the k-tile).  Every role walks it alike.
// Entries are positions in the CSR arrays: e0 .. end0 (q-tile 0), e1 .. end1.
struct PairWalk {
  int e0, end0, e1, end1;
  __device__ bool next(const int32_t* kidx, const uint8_t* klabel, int& kt, int& a, int& b) {
    const int x0 = e0 < end0 ? __ldg(kidx + e0) : INT_MAX;
    const int x1 = e1 < end1 ? __ldg(kidx + e1) : INT_MAX;
    kt = min(x0, x1);
    if (kt == INT_MAX) return false;
    a = ATTN_TILE_EMPTY;
    b = ATTN_TILE_EMPTY;
    if (x0 == kt) a = __ldg(klabel + e0++);
    if (x1 == kt) b = __ldg(klabel + e1++);
    return true;
  }
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

// Shared-memory descriptors: one base per tile; each k-step adds a constant to
// the start-address field (addresses stay below 2^18, so no carry leaves it).
// K-major operand (Q or K): k-step kk covers elements [16kk, 16kk+16) of D.
template <int D>
__device__ __forceinline__ uint64_t kmajor_base(uint32_t tile_addr) {
  using C = Cfg<D>;
  return ptx::smem_desc(tile_addr, 16u, C::SBO, C::SW);
}
template <int D>
__host__ __device__ constexpr uint64_t kmajor_step(int kk) {
  using C = Cfg<D>;
  return uint64_t(((16 * kk) / C::CE) * C::CHUNK + ((16 * kk) % C::CE) * 2) >> 4;
}
// MN-major operand V (N = D across chunks, K = keys): k-step kk covers keys [16kk, 16kk+16).
template <int D>
__device__ __forceinline__ uint64_t v_base(uint32_t tile_addr) {
  using C = Cfg<D>;
  return ptx::smem_desc(tile_addr, C::CHUNK, C::SBO, C::SW);
}
template <int D>
__host__ __device__ constexpr uint64_t v_step(int kk) {
  using C = Cfg<D>;
  return uint64_t(kk * 16 * C::ROWB) >> 4;
}

template <int D>
__device__ __forceinline__ void issue_s(uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc) {
  using C = Cfg<D>;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk)
    ptx::mma_ss(d_tmem, q_desc + kmajor_step<D>(kk), k_desc + kmajor_step<D>(kk), C::IDESC_S, kk > 0);
}

template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t v_desc, bool acc) {
  using C = Cfg<D>;
#pragma unroll
  for (int kk = 0; kk < kTile / 16; ++kk)
    ptx::mma_ts(d_tmem, p_tmem + uint32_t(kk) * 8u, v_desc + v_step<D>(kk), C::IDESC_PV,
                (acc || kk > 0) ? 1u : 0u);
}

// Per-slot note the producer leaves for the MMA issuer with every load:
// K loads carry the two q-tiles' labels, V loads whether the item has another entry.
constexpr uint32_t kInfoHasNext = 1u << 5;

// One work item: a q-tile pair of one sequence and one head.
struct Item {
  int h, s0, L, qi0;
  bool has1;
  PairWalk walk;
};

__device__ __forceinline__ Item decode_item(const FwdParams& p, int item, int n_pairs, int n_qt) {
  Item it;
  it.h = item / n_pairs;
  const int g0 = p.pair_q0[p.pair_order[item % n_pairs]];
  const int b = p.qt_seq[g0];
  it.has1 = g0 + 1 < n_qt && p.qt_seq[g0 + 1] == b;
  it.s0 = p.cu[b];
  it.L = p.cu[b + 1] - it.s0;
  it.qi0 = p.qt_idx[g0] * kTile;  // first query row of q-tile 0, local to the sequence
  it.walk.e0 = p.koff[g0];
  it.walk.end0 = p.koff[g0 + 1];
  it.walk.e1 = it.walk.end0;
  it.walk.end1 = it.has1 ? p.koff[g0 + 2] : it.walk.end0;
  return it;
}

// The producer publishes decoded items to the other roles as 8 ints.
__device__ __forceinline__ void store_item(volatile int* d, const Item& it, bool valid) {
  d[0] = valid ? 1 : 0;
  d[1] = it.h;
  d[2] = it.s0;
  d[3] = it.L;
  d[4] = it.qi0 | (it.has1 ? int(0x80000000) : 0);
  d[5] = it.walk.e0;
  d[6] = it.walk.end0;
  d[7] = it.walk.end1;
}
__device__ __forceinline__ bool load_item(const volatile int* d, Item& it) {
  if (!d[0]) return false;
  it.h = d[1];
  it.s0 = d[2];
  it.L = d[3];
  const int q = d[4];
  it.has1 = q < 0;
  it.qi0 = q & 0x7fffffff;
  it.walk.e0 = d[5];
  it.walk.end0 = d[6];
  it.walk.e1 = it.walk.end0;
  it.walk.end1 = d[7];
  return true;
}

// Producer warp: take a ticket, decode it and publish item k in ring slot k & 1
// (barriers iempty0 / ifull0 and the next ones 8 bytes on).  Returns 1 for an
// item, 0 when no work is left (an end marker is published), -1 on abort.
__device__ __forceinline__ int publish_item(const FwdParams& p, int k, int lane, int n_items, int n_pairs,
                                            int n_qt, Item& it, volatile int* item_ring, uint32_t iempty0,
                                            uint32_t ifull0, volatile uint32_t* abort_flag, int32_t* err) {
  int ticket = 0;
  if (lane == 0) ticket = atomicAdd(p.header + kHdrTicket, 1);
  ticket = __shfl_sync(0xffffffffu, ticket, 0);
  const bool valid = ticket < n_items;
  if (valid) it = decode_item(p, ticket, n_pairs, n_qt);
  const int slot_i = k & 1;
  if (k >= 2 && !warp_wait(iempty0 + 8u * slot_i, uint32_t((k >> 1) - 1) & 1u, abort_flag, err, 15))
    return -1;
  if (lane == 0) {
    store_item(item_ring + 8 * slot_i, it, valid);
    ptx::mbar_arrive(ifull0 + 8u * slot_i);
  }
  return valid ? 1 : 0;
}

// Persistent: each CTA takes work items from a global ticket counter (items
// are head-major, longest q-tile pair first inside a head, so tickets hand
// out the longest work first).  The producer takes the tickets, decodes them
// one item ahead and passes them to the MMA warp and the softmax groups
// through a two-slot ring in shared memory.  Barrier phases run on across
// items; the next item's Q load and first S MMAs overlap the current item's
// last P.V and O epilogue.  The last CTA to finish returns the counters to
// zero for the next launch.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int n_qt = p.header[kHdrQtiles];
  const int n_pairs = p.header[kHdrPairs];
  const int n_items = n_pairs * p.H;
  int32_t* err = p.header + kHdrError;

  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);
  const uint32_t sQ0 = base + C::OFF_Q0, sQ1 = base + C::OFF_Q1, sRing = base + C::OFF_RING;
  const uint32_t bars = base + C::OFF_BAR;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  uint32_t* misc = reinterpret_cast<uint32_t*>(sbase + C::OFF_MISC);
  volatile uint32_t* abort_flag = misc + 1;
  volatile int* item_ring = reinterpret_cast<volatile int*>(sbase + C::OFF_RINGI);  // 2 x 8 ints
  volatile uint32_t* slot_info = reinterpret_cast<volatile uint32_t*>(sbase + C::OFF_SINFO);
  int* slot_codes = reinterpret_cast<int*>(sbase + C::OFF_CODES);

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(C::B_Q), 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(bar(C::B_IFULL + s), 1);
      ptx::mbar_init(bar(C::B_IEMPTY + s), 2 + 256);  // both MMA issuers + both softmax groups
    }
    ptx::mbar_init(bar(C::B_QFREE), 2);  // both MMA issuers
    for (int s = 0; s < C::NSLOT; ++s) {
      ptx::mbar_init(bar(C::B_FULL + s), 1);
      ptx::mbar_init(bar(C::B_EMPTY + s), 2);  // both MMA issuers
    }
    ptx::mbar_init(bar(C::B_VTMA), 1);
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(bar(C::B_SFULL + t), 1);
      ptx::mbar_init(bar(C::B_PFULL + t), 128);
      ptx::mbar_init(bar(C::B_ODONE + t), 1);
      ptx::mbar_init(bar(C::B_OFREE + t), 128);
    }
    ptx::mbar_init(bar(C::B_DRAIN), 2);
    for (int t = 0; t < 2; ++t) ptx::mbar_init(bar(C::B_TURN + t), 1);
    for (int c = 0; c < C::NCODE; ++c) ptx::mbar_init(bar(C::B_CODE + c), 1);
    // An earlier CTA that gave up on a wait makes every later one skip its work.
    *abort_flag = (*reinterpret_cast<volatile int32_t*>(err) & kErrTimeout) ? 1u : 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 9) {
    ptx::tmem_alloc(ptx::smem_addr(misc), C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = misc[0];
  const bool skip = *abort_flag != 0u;

  if (warp >= 8) {
   ptx::regs_dec<kOtherRegs>();
   if (skip) {
    // nothing issued, nothing to drain
   } else if (warp == 8) {
    // ------------------------------------------------------------ producer
    int nload = 0, ntail = 0, nq = 0;
    bool tail_pending = false, ok = true;
    if (lane == 0) {
      ptx::prefetch_tensormap(&tmQ);
      ptx::prefetch_tensormap(&tmK);
      ptx::prefetch_tensormap(&tmV);
    }
    // Take a ticket, decode it and publish it in ring slot k & 1, one item
    // ahead of the loads, so the other roles never wait on the decoding.
    Item it_next;
    int st_next = publish_item(p, 0, lane, n_items, n_pairs, n_qt, it_next, item_ring,
                               bar(C::B_IEMPTY), bar(C::B_IFULL), abort_flag, err);
    for (int k = 0; ok && st_next == 1; ++k) {
      Item it = it_next;
      st_next = publish_item(p, k + 1, lane, n_items, n_pairs, n_qt, it_next, item_ring,
                             bar(C::B_IEMPTY), bar(C::B_IFULL), abort_flag, err);
      if (st_next < 0) break;
      // Q of this item, once the previous item's S MMAs no longer read Q.
      if (nq > 0 && !warp_wait(bar(C::B_QFREE), uint32_t(nq - 1) & 1u, abort_flag, err, 13)) break;
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(bar(C::B_Q), C::TILE * (it.has1 ? 2 : 1));
        for (int c = 0; c < C::NCH; ++c)
          ptx::tma_load_3d(sQ0 + c * C::CHUNK, &tmQ, bar(C::B_Q), c * C::CE, it.h, it.s0 + it.qi0);
        if (it.has1)
          for (int c = 0; c < C::NCH; ++c)
            ptx::tma_load_3d(sQ1 + c * C::CHUNK, &tmQ, bar(C::B_Q), c * C::CE, it.h,
                             it.s0 + it.qi0 + kTile);
      }
      ++nq;
      int kt, la, lb;
      bool have = it.walk.next(p.kidx, p.klabel, kt, la, lb);
      while (have) {
        int kt2, la2, lb2;
        const bool nxt = it.walk.next(p.kidx, p.klabel, kt2, la2, lb2);
        const int j0 = kt * kTile, kn = min(kTile, it.L - j0);
        // K(j)
        int slot = nload % C::NSLOT;
        if (nload >= C::NSLOT &&
            !warp_wait(bar(C::B_EMPTY + slot), uint32_t(nload / C::NSLOT - 1) & 1u, abort_flag, err, 1)) {
          ok = false;
          break;
        }
        // Keys' mask codes for the softmax of PARTIAL tiles, in buffer j % 3,
        // ready when S(j) is.  The buffer's previous entry, j - 3, is done with
        // it: K(j-2)'s slot is freed by each MMA thread after its P.V(j-3),
        // which it issues only once that q-tile's softmax of entry j-3 is over.
        {
          const int cb = (nload / 2) % C::NCODE;
          if (p.mask.kind != ATTN_MASK_CAUSAL && (la == ATTN_TILE_PARTIAL || lb == ATTN_TILE_PARTIAL)) {
            for (int c = lane; c < kTile; c += 32)
              slot_codes[cb * kTile + c] = key_code(p.mask, it.s0 + j0 + min(c, kn - 1));
            __syncwarp();
          }
          if (lane == 0) ptx::mbar_arrive(bar(C::B_CODE + cb));
        }
        if (lane == 0) {
          slot_info[slot] = uint32_t(la) | (uint32_t(lb) << 2);
          ptx::mbar_arrive_expect_tx(bar(C::B_FULL + slot), C::TILE);
          for (int c = 0; c < C::NCH; ++c)
            ptx::tma_load_3d(sRing + slot * C::TILE + c * C::CHUNK, &tmK, bar(C::B_FULL + slot),
                             c * C::CE, it.h, it.s0 + j0);
        }
        ++nload;
        // V(j)
        slot = nload % C::NSLOT;
        if (nload >= C::NSLOT &&
            !warp_wait(bar(C::B_EMPTY + slot), uint32_t(nload / C::NSLOT - 1) & 1u, abort_flag, err, 1)) {
          ok = false;
          break;
        }
        if (kn < kTile) {
          // Rows past the sequence end come from the next sequence (or are zero
          // past the tensor).  Their P is exactly 0, but 0 * inf is NaN, so they
          // are zeroed before the P.V product may read them.
          if (lane == 0) {
            ptx::mbar_arrive_expect_tx(bar(C::B_VTMA), C::TILE);
            for (int c = 0; c < C::NCH; ++c)
              ptx::tma_load_3d(sRing + slot * C::TILE + c * C::CHUNK, &tmV, bar(C::B_VTMA), c * C::CE,
                               it.h, it.s0 + j0);
          }
          tail_pending = true;
          if (!warp_wait(bar(C::B_VTMA), uint32_t(ntail) & 1u, abort_flag, err, 2)) {
            ok = false;
            break;
          }
          tail_pending = false;
          ++ntail;
          for (int rr = kn + lane; rr < kTile; rr += 32) {
#pragma unroll
            for (int c = 0; c < C::NCH; ++c) {
              uint4* row = reinterpret_cast<uint4*>(sbase + C::OFF_RING + slot * C::TILE + c * C::CHUNK +
                                                    rr * C::ROWB);
#pragma unroll
              for (int x = 0; x < C::ROWB / 16; ++x) row[x] = make_uint4(0u, 0u, 0u, 0u);
            }
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            slot_info[slot] = nxt ? kInfoHasNext : 0u;
            ptx::mbar_arrive(bar(C::B_FULL + slot));
          }
        } else if (lane == 0) {
          slot_info[slot] = nxt ? kInfoHasNext : 0u;
          ptx::mbar_arrive_expect_tx(bar(C::B_FULL + slot), C::TILE);
          for (int c = 0; c < C::NCH; ++c)
            ptx::tma_load_3d(sRing + slot * C::TILE + c * C::CHUNK, &tmV, bar(C::B_FULL + slot),
                             c * C::CE, it.h, it.s0 + j0);
        }
        ++nload;
        kt = kt2;
        la = la2;
        lb = lb2;
        have = nxt;
      }
    }
    // Do not leave while a load this CTA issued may still be writing shared memory.
    if (lane == 0) {
      for (int s = 0; s < C::NSLOT; ++s) {
        if (nload <= s) continue;
        const int last = s + C::NSLOT * ((nload - 1 - s) / C::NSLOT);  // last load into slot s
        drain_bar(bar(C::B_FULL + s), uint32_t(last / C::NSLOT) & 1u, err);
      }
      if (tail_pending) drain_bar(bar(C::B_VTMA), uint32_t(ntail) & 1u, err);
      if (nq > 0) drain_bar(bar(C::B_Q), uint32_t(nq - 1) & 1u, err);
    }
    __syncwarp();
   } else if (warp == 9 || warp == 10) {
    // ------------------------------------------------------------ MMA issuers
    // One thread of warp 9 issues q-tile 0's MMAs, one of warp 10 q-tile 1's.
    // They take turns: PV0(j), S0(j+1) | PV1(j), S1(j+1) | PV0(j+1), ... so the
    // tensor pipe serves the q-tiles alternately (one softmax group works while
    // the pipe runs the other's products).  An MMA issue blocks while the
    // pipe's short queue is full, so each issuer does its barrier waits and
    // commits while the other one is issuing, and the queue does not run dry.
    if (lane == 0) {
      const int t = warp - 9;
      const uint32_t colS = C::col_s(t), colO = C::col_o(t);
      int nload = 0, cnt = 0, nturn = 0;
      bool ok = true;
      const uint64_t qdesc = kmajor_base<D>(t == 0 ? sQ0 : sQ1);
      const uint64_t kdesc0 = kmajor_base<D>(sRing), vdesc0 = v_base<D>(sRing);
      // Turn n of issuer 0 follows turn n-1 of issuer 1; turn n of issuer 1
      // follows turn n of issuer 0.
      auto take_turn = [&]() -> bool {
        if (t == 0 && nturn == 0) return true;
        return wait_bar(bar(C::B_TURN + t), uint32_t(t == 0 ? nturn - 1 : nturn) & 1u, abort_flag, err, 18);
      };
      auto pass_turn = [&]() {
        ptx::mbar_arrive(bar(C::B_TURN + (1 - t)));
        ++nturn;
      };
      for (int k = 0; ok; ++k) {
        if (!wait_bar(bar(C::B_IFULL + (k & 1)), uint32_t(k >> 1) & 1u, abort_flag, err, 16)) break;
        Item it;
        const bool valid = load_item(item_ring + 8 * (k & 1), it);
        ptx::mbar_arrive(bar(C::B_IEMPTY + (k & 1)));
        if (!valid) break;
        if (!wait_bar(bar(C::B_Q), uint32_t(k) & 1u, abort_flag, err, 3)) { ok = false; break; }
        if (it.walk.e0 == it.walk.end0 && it.walk.e1 == it.walk.end1) {  // no entries
          ptx::mma_commit(bar(C::B_QFREE));
          continue;
        }
        bool first = true;  // no P.V of this item issued yet
        int lab;
        // entry 0: S from K(0)
        {
          const int slot = nload % C::NSLOT;
          if (!wait_bar(bar(C::B_FULL + slot), uint32_t(nload / C::NSLOT) & 1u, abort_flag, err, 4)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          lab = int((slot_info[slot] >> (2 * t)) & 3u);
          if (!take_turn()) { ok = false; break; }
          if (lab) issue_s<D>(tmem + colS, qdesc, kdesc0 + uint64_t(slot) * (C::TILE >> 4));
          pass_turn();
          if (lab) ptx::mma_commit(bar(C::B_SFULL + t));
          ptx::mma_commit(bar(C::B_EMPTY + slot));
          ++nload;
        }
        for (;;) {
          // V(j): its note says whether entry j+1 exists
          const int vslot = nload % C::NSLOT;
          if (!wait_bar(bar(C::B_FULL + vslot), uint32_t(nload / C::NSLOT) & 1u, abort_flag, err, 6)) {
            ok = false;
            break;
          }
          const bool nxt = (slot_info[vslot] & kInfoHasNext) != 0u;
          const int kslot = (nload + 1) % C::NSLOT;
          int nlab = 0;
          if (nxt) {
            // K(j+1), so that S(j+1) follows P.V(j) in the same turn
            if (!wait_bar(bar(C::B_FULL + kslot), uint32_t((nload + 1) / C::NSLOT) & 1u, abort_flag, err, 4)) {
              ok = false;
              break;
            }
            nlab = int((slot_info[kslot] >> (2 * t)) & 3u);
          } else {
            // every S of this item has been issued: Q may be replaced once they finish
            ptx::mma_commit(bar(C::B_QFREE));
          }
          if (lab) {
            if (!wait_bar(bar(C::B_PFULL + t), uint32_t(cnt) & 1u, abort_flag, err, 5)) { ok = false; break; }
            if (first && k > 0 &&
                !wait_bar(bar(C::B_OFREE + t), uint32_t(k - 1) & 1u, abort_flag, err, 14)) { ok = false; break; }
          }
          ptx::tc_fence_after();
          if (!take_turn()) { ok = false; break; }
          if (lab) issue_pv<D>(tmem + colO, tmem + colS, vdesc0 + uint64_t(vslot) * (C::TILE >> 4), !first);
          if (nlab) issue_s<D>(tmem + colS, qdesc, kdesc0 + uint64_t(kslot) * (C::TILE >> 4));
          pass_turn();
          if (lab) {
            first = false;
            ++cnt;
          }
          // The item's last P.V: O is final once this arrives.
          if (!nxt && !first) ptx::mma_commit(bar(C::B_ODONE + t));
          if (nlab) ptx::mma_commit(bar(C::B_SFULL + t));
          ptx::mma_commit(bar(C::B_EMPTY + vslot));
          ++nload;
          if (!nxt) break;
          ptx::mma_commit(bar(C::B_EMPTY + kslot));
          ++nload;
          lab = nlab;
        }
      }
      // Every MMA this thread issued has finished once this commit arrives.
      ptx::mma_commit(bar(C::B_DRAIN));
      drain_bar(bar(C::B_DRAIN), 0, err);
    }
    __syncwarp();
   }  // warp 11 idle
  } else if (!skip) {
    ptx::regs_inc<kSoftmaxRegs>();
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;                   // which q-tile of the pair
    const int quarter = warp & 3;              // TMEM lanes this warp may access
    const int r = quarter * 32 + lane;         // query row inside the tile
    const int kind = p.mask.kind;
    const uint32_t lane_base = tmem + (uint32_t(quarter * 32) << 16);
    const uint32_t colS = C::col_s(t), colO = C::col_o(t);
    const float c2 = p.scale_log2;
    int cnt = 0;     // entries processed by this q-tile slot over all items (barrier phases)
    int nodone = 0;  // items whose final O this slot has waited for
    int ue_next = 0; // union entries walked (both q-tiles), = K/V ring loads / 2
    bool ok = true;
    for (int k = 0; ok; ++k) {
      if (!warp_wait(bar(C::B_IFULL + (k & 1)), uint32_t(k >> 1) & 1u, abort_flag, err, 16)) break;
      Item it;
      const bool valid = load_item(item_ring + 8 * (k & 1), it);
      ptx::mbar_arrive(bar(C::B_IEMPTY + (k & 1)));
      if (!valid) break;
      const bool present = t == 0 || it.has1;
      const int it0 = it.qi0 + t * kTile;      // first row of this q-tile (local)
      const int qn = present ? min(kTile, it.L - it0) : 0;
      const bool row_in = r < qn;
      const int il = it0 + r;                  // local query index
      const int s0 = it.s0, L = it.L;
      const int qcode = (row_in && kind != ATTN_MASK_CAUSAL) ? query_code(p.mask, s0 + il) : 0;
      // The rows of a warp usually share one query code (one document, one
      // turn).  A key's visibility is then the same for all of them, and one
      // ballot over the keys' codes replaces 32 tests per row.
      const int qcode_w = __shfl_sync(0xffffffffu, qcode, 0);
      const bool uniform_q = __all_sync(0xffffffffu, !row_in || qcode == qcode_w);
      float m_ref = -INFINITY, l = 0.f;
      int cnt_item = 0;
      int kt, la, lb;
      // an absent second q-tile does not walk, but the ring still advanced by
      // the item's union entries (q-tile 0's list)
      if (!present) ue_next += it.walk.end0 - it.walk.e0;
      bool have = present && it.walk.next(p.kidx, p.klabel, kt, la, lb);
      while (have) {
        const int lab = t == 0 ? la : lb;
        const int j0 = kt * kTile;
        const int ue = ue_next++;  // union entry number over all items (ring position)
        // fetch the next entry now; its loads complete under this entry's work
        have = it.walk.next(p.kidx, p.klabel, kt, la, lb);
        if (lab == ATTN_TILE_EMPTY) continue;
        const int kn = min(kTile, L - j0);
        if (!warp_wait(bar(C::B_SFULL + t), uint32_t(cnt) & 1u, abort_flag, err, 8)) { ok = false; break; }
        ptx::tc_fence_after();
        float s[128];
        {
          uint32_t v[4][32];
#pragma unroll
          for (int q = 0; q < 4; ++q) ptx::tmem_ld32(lane_base + colS + q * 32, v[q]);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int c = 0; c < 32; ++c) s[q * 32 + c] = __uint_as_float(v[q][c]);
        }
        if (lab == ATTN_TILE_PARTIAL || kn < kTile) {
          // bit c of vis[c / 32]: key column c is visible to this row.  Causal part
          // and bounds: columns c < upto; PARTIAL tiles of the metadata kinds also
          // AND in the per-key predicate.
          const int upto = lab == ATTN_TILE_PARTIAL ? min(kn, il - j0 + 1) : kn;
          uint32_t vis[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) vis[q] = prefix_bits(upto - 32 * q);
          if (lab == ATTN_TILE_PARTIAL && kind != ATTN_MASK_CAUSAL) {
            // the producer wrote this entry's key codes before loading K(j)
            if (!warp_wait(bar(C::B_CODE + ue % C::NCODE), uint32_t(ue / C::NCODE) & 1u, abort_flag, err, 9)) {
              ok = false;
              break;
            }
            const int* codes = slot_codes + (ue % C::NCODE) * kTile;
            if (uniform_q) {
              int kc[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) kc[q] = codes[32 * q + lane];
              if (kind == ATTN_MASK_STRIP_THINKING) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  vis[q] &= __ballot_sync(0xffffffffu, code_visible(ATTN_MASK_STRIP_THINKING, qcode_w, kc[q]));
              } else if (kind == ATTN_MASK_SHARED_PREFIX) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  vis[q] &= __ballot_sync(0xffffffffu, code_visible(ATTN_MASK_SHARED_PREFIX, qcode_w, kc[q]));
              } else {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  vis[q] &= __ballot_sync(0xffffffffu, code_visible(ATTN_MASK_CAUSAL_DOCUMENT, qcode_w, kc[q]));
              }
            } else if (kind == ATTN_MASK_STRIP_THINKING) {
#pragma unroll
              for (int q = 0; q < 4; ++q)
                if (vis[q]) vis[q] &= code_word<ATTN_MASK_STRIP_THINKING>(codes, q, qcode);
            } else if (kind == ATTN_MASK_SHARED_PREFIX) {
#pragma unroll
              for (int q = 0; q < 4; ++q)
                if (vis[q]) vis[q] &= code_word<ATTN_MASK_SHARED_PREFIX>(codes, q, qcode);
            } else {
#pragma unroll
              for (int q = 0; q < 4; ++q)
                if (vis[q]) vis[q] &= code_word<ATTN_MASK_CAUSAL_DOCUMENT>(codes, q, qcode);
            }
          }
          // A word the whole warp sees needs no select (on a diagonal tile, the
          // words left of the warp's own rows).
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (__all_sync(0xffffffffu, vis[q] == 0xffffffffu)) continue;
#pragma unroll
            for (int c = 0; c < 32; ++c) s[32 * q + c] = (vis[q] >> c) & 1u ? s[32 * q + c] : -INFINITY;
          }
        }
        float mx8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          float mv = s[16 * u];
#pragma unroll
          for (int c = 1; c < 15; c += 2) mv = ptx::fmax3(mv, s[16 * u + c], s[16 * u + c + 1]);
          mx8[u] = fmaxf(mv, s[16 * u + 15]);
        }
        const float mxs = ptx::fmax3(ptx::fmax3(mx8[0], mx8[1], mx8[2]), ptx::fmax3(mx8[3], mx8[4], mx8[5]),
                                     fmaxf(mx8[6], mx8[7])) * c2;
        const bool raise = mxs > m_ref + kRescaleThreshold;  // always true on the first visible key
        const bool rescale = raise && m_ref != -INFINITY;   // O and l hold an older reference
        const float m_new = raise ? mxs : m_ref;
        const float alpha = rescale ? ptx::ex2(m_ref - m_new) : 1.f;
        if (cnt_item > 0 && __any_sync(0xffffffffu, rescale)) {
          // O holds exactly the P.V of earlier entries: this S was issued after
          // them by the same thread, and its commit arrives only once they are done.
          const float2 a2 = make_float2(alpha, alpha);
#pragma unroll 1
          for (int q = 0; q < D / 32; ++q) {
            uint32_t v[32];
            ptx::tmem_ld32(lane_base + colO + q * 32, v);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              const float2 x = ptx::fmul2(make_float2(__uint_as_float(v[c]), __uint_as_float(v[c + 1])), a2);
              v[c] = __float_as_uint(x.x);
              v[c + 1] = __float_as_uint(x.y);
            }
            ptx::tmem_st32(lane_base + colO + q * 32, v);
          }
        }
        l *= alpha;
        m_ref = m_new;
        const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
        const float2 c22 = make_float2(c2, c2), nm2 = make_float2(-m_use, -m_use);
        // four independent partial sums keep the additions off one serial chain
        float2 sum2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                          make_float2(0.f, 0.f)};
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const float2 x = ptx::ffma2(make_float2(s[32 * hh + c], s[32 * hh + c + 1]), c22, nm2);
            const float2 e = make_float2(ptx::ex2(x.x), ptx::ex2(x.y));
            sum2[(c >> 1) & 3] = ptx::fadd2(sum2[(c >> 1) & 3], e);
            pk[c >> 1] = ptx::pack_bf16(e.x, e.y);
          }
          ptx::tmem_st16(lane_base + colS + hh * 16, pk);
        }
        const float2 sa = ptx::fadd2(sum2[0], sum2[1]), sb = ptx::fadd2(sum2[2], sum2[3]);
        l += (sa.x + sb.x) + (sa.y + sb.y);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(C::B_PFULL + t));
        ++cnt;
        ++cnt_item;
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (present && cnt_item > 0) {
        if (!warp_wait(bar(C::B_ODONE + t), uint32_t(nodone) & 1u, abort_flag, err, 11)) {
          ok = false;
          break;
        }
        ++nodone;
      }
      if (present) {
        ptx::tc_fence_after();
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        __nv_bfloat16* orow = p.o + (size_t(s0 + il) * p.H + it.h) * D;
#pragma unroll 1
        for (int q = 0; q < D / 32; ++q) {
          uint32_t v[32];
          if (cnt_item > 0) {
            ptx::tmem_ld32(lane_base + colO + q * 32, v);
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
          p.lse[size_t(it.h) * p.T + s0 + il] =
              l > 0.f ? (m_ref + ptx::lg2(l)) * 0.69314718055994531f : -INFINITY;
      }
      // This q-tile slot's O columns may now take the next item's P.V.
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(C::B_OFREE + t));
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (threadIdx.x == 0) {
    // Every CTA has taken its last ticket before it counts itself finished, so
    // the last one can return both counters to zero for the next launch.
    __threadfence();
    if (atomicAdd(p.header + kHdrFinished, 1) == int(gridDim.x) - 1) {
      atomicExch(p.header + kHdrTicket, 0);
      atomicExch(p.header + kHdrFinished, 0);
    }
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
    return record_cuda_error(cudaErrorInvalidValue, "attn_fwd tensor map encoding");
  static bool configured = false;
  if (!configured) {
    // The warpgroups' register split assumes the kernel launches with exactly
    // kLaunchRegs per thread; anything else could leave setmaxnreg.inc waiting.
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, attn_fwd_bf16_kernel<D>);
    if (e != cudaSuccess) return record_cuda_error(e, "attn_fwd configure");
    if (fa.numRegs != kLaunchRegs) return ATTN_ERR_UNSUPPORTED;
    e = cudaFuncSetAttribute(attn_fwd_bf16_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) return record_cuda_error(e, "attn_fwd configure");
    configured = true;
  }
  FwdParams p;
  p.header = a.bm.header;
  p.pair_order = a.bm.pair_order;
  p.pair_q0 = a.bm.pair_q0;
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
  // Persistent: one CTA per SM (the pair count is only known on the device;
  // max_qt * H bounds it).
  static int num_sms = 0;
  if (num_sms == 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return record_cuda_error(e, "attn_fwd device query");
  }
  const long long items = (long long)a.bm.max_qt * a.num_heads;
  if (items <= 0 || items > INT_MAX) return ATTN_ERR_UNSUPPORTED;
  const long long grid = items < num_sms ? items : num_sms;
  attn_fwd_bf16_kernel<D><<<unsigned(grid), kThreads, C::SMEM_ALLOC, s>>>(mq, mk, mv, p);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? ATTN_OK : record_cuda_error(e, "attn_fwd launch");
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
