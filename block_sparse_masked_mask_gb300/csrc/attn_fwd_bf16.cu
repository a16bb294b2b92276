// bf16 attention forward on the sm_103a tensor cores (tcgen05 + TMA + TMEM).
//
// The loop is the online-softmax flash attention of "Triton from first
// principles" Ch. 21, Section 21.1 (running max m, running sum l, accumulator
// rescaled by exp(m_old - m_new), one division at the end), with the causal /
// structured mask applied inside the loop as in Section 21.2, and only the
// k-tiles the block mask lists are visited (Ch. 9, Section 9.2: a skipped
// tile is never loaded).
//
// A work item is one 128-row q-tile of one sequence and one head; persistent
// CTAs (one per SM) take the items longest first and walk each q-tile's k-tile
// list in ascending order.  Warp roles (512 threads):
//   warps 0-7  softmax, two threads per query row: warps 0-3 take score
//              columns 0-63 of every k-tile, warps 4-7 columns 64-127
//   warp 8     TMA producer of Q and of the K ring (three slots); stages the
//              keys' mask codes of PARTIAL tiles; takes the work tickets
//   warp 9     tcgen05 issuer of the P.V products (one thread; also owns the
//              TMEM allocation)
//   warp 10    TMA producer of the V ring (two slots); zeroes V rows past a
//              sequence end
//   warp 11    tcgen05 issuer of the S = Q K^T products (one thread)
//   warps 12-15 epilogue: one thread per query row reads the item's final O
//              from TMEM once (as bf16 pairs, divided by l), releases it, and
//              writes O and LSE while the softmax warps already work on the
//              next item
// The softmax warpgroups run with 160 registers a thread (144 for the dense
// kind), the producer / issuer warpgroup with 64 (96), the epilogue with the
// launch's 128 (setmaxnreg, within the 128 x 512 the block is launched with).
// The two issuers work independently: an MMA issue blocks while the tensor
// pipe's short queue is full, and with two threads one waits on its barriers
// while the other keeps the queue fed.
// TMEM columns: S0 [0,128), S1 [128,256), S2 [256,384) hold S of three
// consecutive k-tiles, O [384, 384+D) the accumulator.  Each half of a row
// writes its bf16 P over the first 32 of its own 64 S columns, so S(j) waits
// for P(j-3).V; the tensor cores compute S(j+1), S(j+2) and P(j-1).V while
// the softmax works on S(j).  The next item's first P.V waits for the
// epilogue's one read of O (a few hundred cycles), not for its stores.
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
#include "tile_pipeline.cuh"

namespace attnmask {
namespace {

constexpr float kRescaleThreshold = 8.0f;           // log2 units: p stays <= 256
constexpr int kThreads = 512;
constexpr int kWarpKLoad = 8, kWarpPV = 9, kWarpVLoad = 10, kWarpS = 11, kWarpEpi = 12;
// Registers per thread: the softmax warpgroups, the producer / issuer
// warpgroup and the epilogue warpgroup, which keeps the launch's 128 (a whole
// row of O in bf16).  The dense kind's softmax (its bit words) fits 144 without
// spills only if the producers get 96; the others run fastest with 160 / 64
// (measured).
template <bool kDense>
struct Regs {
  static constexpr int softmax = kDense ? 144 : 160, prod = kDense ? 96 : 64, epi = 128;
  static_assert(2 * 128 * softmax + 128 * prod + 128 * epi == kThreads * 128, "register split");
  static_assert(epi == 128, "the epilogue warpgroup runs with the launch's count");
};

template <int D>
struct Cfg : TileLayout<D> {
  using TileLayout<D>::TILE;
  using TileLayout<D>::CHUNK;
  using TileLayout<D>::CE;
  using TileLayout<D>::NCH;
  using TileLayout<D>::ROWB;
  // Q slots and K ring slots: a second Q slot (the next item's Q loaded under
  // this item's last k-tiles) in place of the third K slot measured slower
  // on every workload (0.950 vs 0.934 ms on the 32k mask, 0.108 vs 0.104 ms
  // on the 8-sequence varlen batch)
  static constexpr int NQ = 1;
  static constexpr int NK = 3;
  static constexpr int NV = 2;                        // V ring slots
  static constexpr int NCODE = 6;                     // key-code buffers (entries in flight)
  static constexpr int OFF_Q = 0, OFF_K = NQ * TILE, OFF_V = OFF_K + NK * TILE;
  // TMEM (512 columns): NS S buffers and NO O accumulators of 128 columns.
  // One O: the epilogue reads the item's O once into registers and releases
  // it at once, so the next item's first P.V waits only for that read; the
  // third S buffer keeps three k-tiles in flight (S(j) waits for P.V(j - 3)).
  static constexpr int NO = 1;
  static constexpr int NS = 4 - NO;
  // SFULL / PFULL / PDONE: per S buffer; XMAX: per entry parity; ODONE, OFREE,
  // STATS: per item parity
  static constexpr int B_Q = 0, B_QFREE = NQ, B_KFULL = 2 * NQ, B_KEMPTY = B_KFULL + NK, B_VFULL = B_KEMPTY + NK,
                       B_VEMPTY = B_VFULL + NV, B_VTMA = B_VEMPTY + NV, B_SFULL = B_VTMA + 1,
                       B_PFULL = B_SFULL + NS, B_PDONE = B_PFULL + NS, B_ODONE = B_PDONE + NS,
                       B_OFREE = B_ODONE + 2, B_IFULL = B_OFREE + 2, B_IEMPTY = B_IFULL + 2,
                       B_CODE = B_IEMPTY + 2, B_CODEFREE = B_CODE + NCODE, B_XMAX = B_CODEFREE + NCODE,
                       B_STATS = B_XMAX + 2, B_DRAIN = B_STATS + 2, NBAR = B_DRAIN + 1;
  static constexpr int OFF_BAR = OFF_V + NV * TILE;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int OFF_RINGI = OFF_MISC + 16;            // two decoded work items, 8 ints each
  static constexpr int OFF_CODES = (OFF_RINGI + 2 * 8 * 4 + 15) & ~15;  // per buffer: 128 key codes
  static constexpr int OFF_XMAX = OFF_CODES + NCODE * kTile * 4;  // [entry parity][half][row] floats
  static constexpr int OFF_STATS = OFF_XMAX + 2 * 2 * kTile * 4;  // [item parity][l0, l1, m][row] floats
  static constexpr int OFF_OSTAGE = (OFF_STATS + 2 * 3 * kTile * 4 + 127) & ~127;  // per epilogue warp
  static constexpr int OSTAGE_WARP = 4096;                                        // 16 rows of 256 bytes
  static constexpr int SMEM_USED = OFF_OSTAGE + 4 * OSTAGE_WARP;
  // + slack to align the base to 1024 B; at least 116 KB so that one CTA holds an SM
  // (and its 512 TMEM columns) alone.
  static constexpr int SMEM_ALLOC = SMEM_USED + 1024 > 116 * 1024 ? SMEM_USED + 1024 : 116 * 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  __host__ __device__ static constexpr uint32_t col_o(int b) { return 128u * uint32_t(NS) + uint32_t(b) * 128u; }
  __host__ __device__ static constexpr uint32_t col_s(int i) { return uint32_t(i) * 128u; }
  static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
};

struct FwdParams {
  int32_t* header;
  int sched;         // this launch's work-counter slot
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

// One work item: a q-tile of one sequence and one head; its k-tile list is
// entries e0 .. e1 of the CSR arrays.
struct Item {
  int h, s0, L, qi0, e0, e1, b;
};

// Items go by groups of kHeadGroup heads: inside a group, q-tiles longest
// list first, each q-tile for every head of the group in turn.  The group
// keeps the K / V tiles the CTAs read at once to a few heads (L2 locality),
// and the longest lists of the last group still start well before the end (a
// purely head-major order starts the last head's longest lists last).
constexpr int kHeadGroup = 8;
__device__ __forceinline__ Item decode_item(const FwdParams& p, int item, int n_qt) {
  Item it;
  const int grp = item / (n_qt * kHeadGroup), r = item - grp * (n_qt * kHeadGroup);
  const int hg = min(kHeadGroup, p.H - grp * kHeadGroup);  // heads in this group
  it.h = grp * kHeadGroup + r % hg;
  const int g = p.order[r / hg];
  const int b = p.qt_seq[g];
  it.s0 = p.cu[b];
  it.L = p.cu[b + 1] - it.s0;
  it.qi0 = p.qt_idx[g] * kTile;  // first query row of the q-tile, local to the sequence
  it.e0 = p.koff[g];
  it.e1 = p.koff[g + 1];
  it.b = b;
  return it;
}

// The K producer publishes decoded items to the other roles as 8 ints.
__device__ __forceinline__ void store_item(volatile int* d, const Item& it, bool valid) {
  d[0] = valid ? 1 : 0;
  d[1] = it.h;
  d[2] = it.s0;
  d[3] = it.L;
  d[4] = it.qi0;
  d[5] = it.e0;
  d[6] = it.e1;
  d[7] = it.b;
}
__device__ __forceinline__ bool load_item(const volatile int* d, Item& it) {
  if (!d[0]) return false;
  it.h = d[1];
  it.s0 = d[2];
  it.L = d[3];
  it.qi0 = d[4];
  it.e0 = d[5];
  it.e1 = d[6];
  it.b = d[7];
  return true;
}

// Take a ticket, decode it and publish item k in ring slot k & 1 (barriers
// iempty0 / ifull0 and the next ones 8 bytes on).  Returns 1 for an item, 0
// when no work is left (an end marker is published), -1 on abort.
__device__ __forceinline__ int publish_item(const FwdParams& p, int k, int lane, int n_items, int n_qt,
                                            Item& it, volatile int* item_ring, uint32_t iempty0,
                                            uint32_t ifull0, volatile uint32_t* abort_flag, int32_t* err) {
  int ticket = 0;
  if (lane == 0) ticket = take_ticket(p.sched);
  ticket = __shfl_sync(0xffffffffu, ticket, 0);
  const bool valid = ticket < n_items;
  if (valid) it = decode_item(p, ticket, n_qt);
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
// go by groups of heads, longest q-tile first inside a group, so tickets hand
// out the longest work first).  The K producer takes the tickets, decodes them one item
// ahead and passes them to the other roles through a two-slot ring in shared
// memory.  Barrier phases run on across items: the next item's Q load and
// first S MMAs overlap the current item's last P.V and O epilogue.  The
// counters are this launch's slot of the scheduler pool; the last CTA to
// finish returns them to zero.
// kDense: the instantiation for ATTN_MASK_DENSE; the others leave its code out
// (the softmax loop is sensitive to its own size).
template <int D, bool kDense>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int n_qt = p.header[kHdrQtiles];
  const int n_items = n_qt * p.H;
  int32_t* err = p.header + kHdrError;

  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);
  const uint32_t sQ = base + C::OFF_Q, sK = base + C::OFF_K, sV = base + C::OFF_V;
  const uint32_t bars = base + C::OFF_BAR;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  uint32_t* misc = reinterpret_cast<uint32_t*>(sbase + C::OFF_MISC);
  volatile uint32_t* abort_flag = misc + 1;
  volatile int* item_ring = reinterpret_cast<volatile int*>(sbase + C::OFF_RINGI);  // 2 x 8 ints
  int* key_codes = reinterpret_cast<int*>(sbase + C::OFF_CODES);

  if (threadIdx.x == 0) {
    for (int q = 0; q < C::NQ; ++q) {
      ptx::mbar_init(bar(C::B_Q + q), 1);
      ptx::mbar_init(bar(C::B_QFREE + q), 1);
    }
    for (int s = 0; s < C::NK; ++s) {
      ptx::mbar_init(bar(C::B_KFULL + s), 1);
      ptx::mbar_init(bar(C::B_KEMPTY + s), 1);
    }
    for (int s = 0; s < C::NV; ++s) {
      ptx::mbar_init(bar(C::B_VFULL + s), 1);
      ptx::mbar_init(bar(C::B_VEMPTY + s), 1);
    }
    ptx::mbar_init(bar(C::B_VTMA), 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bar(C::B_IFULL + i), 1);
      ptx::mbar_init(bar(C::B_IEMPTY + i), 256 + 3 + 128);  // softmax, MMA threads, V producer, epilogue
      ptx::mbar_init(bar(C::B_XMAX + i), 256);
      ptx::mbar_init(bar(C::B_STATS + i), 256);
      ptx::mbar_init(bar(C::B_ODONE + i), 1);
      ptx::mbar_init(bar(C::B_OFREE + i), 128);
    }
    for (int i = 0; i < C::NS; ++i) {
      ptx::mbar_init(bar(C::B_SFULL + i), 1);
      ptx::mbar_init(bar(C::B_PFULL + i), 256);
      ptx::mbar_init(bar(C::B_PDONE + i), 1);
    }
    for (int c = 0; c < C::NCODE; ++c) {
      ptx::mbar_init(bar(C::B_CODE + c), 1);
      ptx::mbar_init(bar(C::B_CODEFREE + c), 256);
    }
    ptx::mbar_init(bar(C::B_DRAIN), 2);  // both MMA threads
    // An earlier CTA that gave up on a wait makes every later one skip its work.
    *abort_flag = (*reinterpret_cast<volatile int32_t*>(err) & kErrTimeout) ? 1u : 0u;
    ptx::fence_mbar_init();
  }
  if (warp == kWarpPV) {
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
  } else if (warp >= kWarpEpi) {
    // ------------------------------------------------------------ epilogue
    // One thread per query row (TMEM lane): once the softmax has posted the
    // row's statistics and the item's last P.V is done, the row of O / l is
    // read once into registers as bf16 pairs and the O buffer released (the
    // next item's first P.V waits for it), then written as whole rows
    // through a 4 KB stage, 16 rows at a time.
    const int quarter = warp - kWarpEpi;       // TMEM lanes 32 quarter ..
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (uint32_t(quarter * 32) << 16);
    const float* stats = reinterpret_cast<const float*>(sbase + C::OFF_STATS);
    uint8_t* stage = sbase + C::OFF_OSTAGE + quarter * C::OSTAGE_WARP;
    constexpr int RB = D * 2;                  // bytes per output row
    constexpr int CPR = RB / 16;               // 16-byte pieces per row
    constexpr int RPI = 32 / CPR;              // rows per warp-wide store
    for (int k = 0;; ++k) {
      if (!warp_wait(bar(C::B_IFULL + (k & 1)), uint32_t(k >> 1) & 1u, abort_flag, err, 16)) break;
      Item it;
      const bool valid = load_item(item_ring + 8 * (k & 1), it);
      ptx::mbar_arrive(bar(C::B_IEMPTY + (k & 1)));
      if (!valid) break;
      const int ob = k & 1;  // item parity: statistics buffer and barriers
      if (!warp_wait(bar(C::B_STATS + ob), uint32_t(k >> 1) & 1u, abort_flag, err, 18)) break;
      const float* st = stats + ob * 3 * kTile;
      const float lt = st[r] + st[kTile + r];  // the halves' row sums, in a fixed order
      const float m = st[2 * kTile + r];
      const int qn = min(kTile, it.L - it.qi0);
      const bool has = it.e1 > it.e0;
      if (!warp_wait(bar(C::B_ODONE + ob), uint32_t(k >> 1) & 1u, abort_flag, err, 11)) break;
      ptx::tc_fence_after();
      const float inv_l = lt > 0.f ? 1.f / lt : 0.f;
      __nv_bfloat16* obase = p.o + (size_t(it.s0 + it.qi0 + quarter * 32) * p.H + it.h) * D;
      const size_t rstride = size_t(p.H) * D;
      const uint32_t ocol = C::col_o(k % C::NO);
      uint32_t pk[D / 2];  // the row as bf16 pairs
#pragma unroll
      for (int q32 = 0; q32 < (D + 31) / 32; ++q32) {
        constexpr int W = D < 32 ? D : 32;   // columns per TMEM read
        uint32_t v[32];
        if (has) {
          if constexpr (W == 32) ptx::tmem_ld32(lane_base + ocol + q32 * 32, v);
          else ptx::tmem_ld16(lane_base + ocol, *reinterpret_cast<uint32_t(*)[16]>(v));
          ptx::tmem_wait_ld();
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = 0u;
        }
#pragma unroll
        for (int x = 0; x < W / 2; ++x)
          pk[q32 * 16 + x] = ptx::pack_bf16(__uint_as_float(v[2 * x]) * inv_l, __uint_as_float(v[2 * x + 1]) * inv_l);
      }
      // every read of the buffer is done
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(C::B_OFREE + ob));
#pragma unroll
      for (int half16 = 0; half16 < 2; ++half16) {
        if ((lane >> 4) == half16) {
          const int q = lane & 15;
#pragma unroll
          for (int c = 0; c < CPR; ++c)  // 16-byte piece c of the row: pairs 4c .. 4c + 3
            *reinterpret_cast<uint4*>(stage + q * RB + ((c ^ q) & (CPR - 1)) * 16) =
                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 16 / RPI; ++i) {
          const int q = i * RPI + lane / CPR, c = lane % CPR;
          const int rr = half16 * 16 + q;
          const uint4 val = *reinterpret_cast<const uint4*>(stage + q * RB + ((c ^ q) & (CPR - 1)) * 16);
          if (quarter * 32 + rr < qn) *reinterpret_cast<uint4*>(obase + size_t(rr) * rstride + 8 * c) = val;
        }
        __syncwarp();
      }
      if (r < qn)
        p.lse[size_t(it.h) * p.T + it.s0 + it.qi0 + r] =
            lt > 0.f ? (m + ptx::lg2(lt)) * 0.69314718055994531f : -INFINITY;
    }
  } else if (warp >= 8) {
   ptx::regs_dec<Regs<kDense>::prod>();
   if (warp == kWarpKLoad) {
    // ------------------------------------------------------------ Q, K, key codes
    int nk = 0, nq = 0, up = 0;  // K loads, Q loads, PARTIAL entries given key codes
    bool ok = true;
    if (lane == 0) {
      ptx::prefetch_tensormap(&tmQ);
      ptx::prefetch_tensormap(&tmK);
    }
    // Take a ticket, decode it and publish it in ring slot k & 1, one item
    // ahead of the loads, so the other roles never wait on the decoding.
    Item it_next;
    int st_next = publish_item(p, 0, lane, n_items, n_qt, it_next, item_ring, bar(C::B_IEMPTY),
                               bar(C::B_IFULL), abort_flag, err);
    for (int k = 0; ok && st_next == 1; ++k) {
      const Item it = it_next;
      st_next = publish_item(p, k + 1, lane, n_items, n_qt, it_next, item_ring, bar(C::B_IEMPTY),
                             bar(C::B_IFULL), abort_flag, err);
      if (st_next < 0) break;
      // Q of this item into slot nq % NQ, once the S MMAs of the item that
      // last used the slot no longer read it.
      const int qsl = nq % C::NQ;
      if (nq >= C::NQ &&
          !warp_wait(bar(C::B_QFREE + qsl), uint32_t(nq / C::NQ - 1) & 1u, abort_flag, err, 13))
        break;
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(bar(C::B_Q + qsl), C::TILE);
        for (int c = 0; c < C::NCH; ++c)
          ptx::tma_load_3d(sQ + uint32_t(qsl) * C::TILE + c * C::CHUNK, &tmQ, bar(C::B_Q + qsl), c * C::CE,
                           it.h, it.s0 + it.qi0);
      }
      ++nq;
      for (int e = it.e0; e < it.e1; ++e) {
        const int j0 = __ldg(p.kidx + e) * kTile, kn = min(kTile, it.L - j0);
        const int lab = __ldg(p.klabel + e);
        if (kind_codes(p.mask.kind) && lab == ATTN_TILE_PARTIAL) {
          // Keys' mask codes for the softmax of a PARTIAL tile, in buffer up % NCODE
          // once the softmax is done with the buffer's previous PARTIAL entry.
          const int cb = up % C::NCODE;
          if (up >= C::NCODE &&
              !warp_wait(bar(C::B_CODEFREE + cb), uint32_t(up / C::NCODE - 1) & 1u, abort_flag, err, 10)) {
            ok = false;
            break;
          }
          for (int c = lane; c < kTile; c += 32)
            key_codes[cb * kTile + c] = key_code(p.mask, it.s0 + j0 + min(c, kn - 1));
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(bar(C::B_CODE + cb));
          ++up;
        }
        // K(j)
        const int slot = nk % C::NK;
        if (nk >= C::NK &&
            !warp_wait(bar(C::B_KEMPTY + slot), uint32_t(nk / C::NK - 1) & 1u, abort_flag, err, 1)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(bar(C::B_KFULL + slot), C::TILE);
          for (int c = 0; c < C::NCH; ++c)
            ptx::tma_load_3d(sK + slot * C::TILE + c * C::CHUNK, &tmK, bar(C::B_KFULL + slot), c * C::CE,
                             it.h, it.s0 + j0);
        }
        ++nk;
      }
    }
    // Do not leave while a load this CTA issued may still be writing shared memory.
    if (lane == 0) {
      for (int s = 0; s < C::NK; ++s) {
        if (nk <= s) continue;
        const int last = s + C::NK * ((nk - 1 - s) / C::NK);  // last load into slot s
        drain_bar(bar(C::B_KFULL + s), uint32_t(last / C::NK) & 1u, err);
      }
      for (int q = 0; q < C::NQ; ++q) {
        if (nq <= q) continue;
        const int last = q + C::NQ * ((nq - 1 - q) / C::NQ);  // last load into slot q
        drain_bar(bar(C::B_Q + q), uint32_t(last / C::NQ) & 1u, err);
      }
    }
    __syncwarp();
  } else if (warp == kWarpVLoad) {
    // ------------------------------------------------------------ V
    int nv = 0, ntail = 0;
    bool tail_pending = false, ok = true;
    if (lane == 0) ptx::prefetch_tensormap(&tmV);
    for (int k = 0; ok; ++k) {
      if (!warp_wait(bar(C::B_IFULL + (k & 1)), uint32_t(k >> 1) & 1u, abort_flag, err, 16)) break;
      Item it;
      const bool valid = load_item(item_ring + 8 * (k & 1), it);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(C::B_IEMPTY + (k & 1)));
      if (!valid) break;
      for (int e = it.e0; e < it.e1; ++e) {
        const int j0 = __ldg(p.kidx + e) * kTile, kn = min(kTile, it.L - j0);
        const int slot = nv % C::NV;
        if (nv >= C::NV &&
            !warp_wait(bar(C::B_VEMPTY + slot), uint32_t(nv / C::NV - 1) & 1u, abort_flag, err, 1)) {
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
              ptx::tma_load_3d(sV + slot * C::TILE + c * C::CHUNK, &tmV, bar(C::B_VTMA), c * C::CE, it.h,
                               it.s0 + j0);
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
              uint4* row = reinterpret_cast<uint4*>(sbase + C::OFF_V + slot * C::TILE + c * C::CHUNK +
                                                    rr * C::ROWB);
#pragma unroll
              for (int x = 0; x < C::ROWB / 16; ++x) row[x] = make_uint4(0u, 0u, 0u, 0u);
            }
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(bar(C::B_VFULL + slot));
        } else if (lane == 0) {
          ptx::mbar_arrive_expect_tx(bar(C::B_VFULL + slot), C::TILE);
          for (int c = 0; c < C::NCH; ++c)
            ptx::tma_load_3d(sV + slot * C::TILE + c * C::CHUNK, &tmV, bar(C::B_VFULL + slot), c * C::CE,
                             it.h, it.s0 + j0);
        }
        ++nv;
      }
    }
    if (lane == 0) {
      for (int s = 0; s < C::NV; ++s) {
        if (nv <= s) continue;
        const int last = s + C::NV * ((nv - 1 - s) / C::NV);
        drain_bar(bar(C::B_VFULL + s), uint32_t(last / C::NV) & 1u, err);
      }
      if (tail_pending) drain_bar(bar(C::B_VTMA), uint32_t(ntail) & 1u, err);
    }
    __syncwarp();
  } else if (warp == kWarpS) {
    // ------------------------------------------------------------ S issuer
    // S(j) into S buffer j % NS once P.V(j - NS) has read the P written over
    // S(j - NS) there.
    if (lane == 0) {
      int nkc = 0, ns = 0;  // K loads consumed, S issued (all items)
      bool ok = true;
      const uint64_t qdesc0 = kmajor_base<D>(sQ), kdesc0 = kmajor_base<D>(sK);
      for (int k = 0; ok; ++k) {
        if (!wait_bar(bar(C::B_IFULL + (k & 1)), uint32_t(k >> 1) & 1u, abort_flag, err, 16)) break;
        Item it;
        const bool valid = load_item(item_ring + 8 * (k & 1), it);
        ptx::mbar_arrive(bar(C::B_IEMPTY + (k & 1)));
        if (!valid) break;
        const int qsl = k % C::NQ;
        if (!wait_bar(bar(C::B_Q + qsl), uint32_t(k / C::NQ) & 1u, abort_flag, err, 3)) break;
        const uint64_t qdesc = qdesc0 + uint64_t(qsl) * (C::TILE >> 4);
        for (int e = it.e0; e < it.e1; ++e) {
          const int sb = ns % C::NS, ks = nkc % C::NK;
          if (ns >= C::NS && !wait_bar(bar(C::B_PDONE + sb), uint32_t(ns / C::NS - 1) & 1u, abort_flag, err, 7)) {
            ok = false;
            break;
          }
          if (!wait_bar(bar(C::B_KFULL + ks), uint32_t(nkc / C::NK) & 1u, abort_flag, err, 4)) { ok = false; break; }
          ptx::tc_fence_after();
          issue_s<D>(tmem + C::col_s(sb), qdesc, kdesc0 + uint64_t(ks) * (C::TILE >> 4));
          ptx::mma_commit(bar(C::B_SFULL + sb));
          ptx::mma_commit(bar(C::B_KEMPTY + ks));
          ++ns;
          ++nkc;
        }
        // every S of this item has been issued: its Q slot may be refilled once
        // they finish
        ptx::mma_commit(bar(C::B_QFREE + qsl));
      }
      // Every MMA this thread issued has finished once this commit arrives.
      ptx::mma_commit(bar(C::B_DRAIN));
      drain_bar(bar(C::B_DRAIN), 0, err);
    }
    __syncwarp();
  } else if (warp == kWarpPV) {
    // ------------------------------------------------------------ P.V issuer
    if (lane == 0) {
      int nvc = 0, np = 0;  // V loads consumed, P.V issued (all items)
      bool ok = true;
      const uint64_t vdesc0 = v_base<D>(sV);
      for (int k = 0; ok; ++k) {
        if (!wait_bar(bar(C::B_IFULL + (k & 1)), uint32_t(k >> 1) & 1u, abort_flag, err, 16)) break;
        Item it;
        const bool valid = load_item(item_ring + 8 * (k & 1), it);
        ptx::mbar_arrive(bar(C::B_IEMPTY + (k & 1)));
        if (!valid) break;
        const int n = it.e1 - it.e0;
        const int ob = k % C::NO;     // this item's O buffer, free once the epilogue of
        const int prev = k - C::NO;   // item k - NO (its last user) has read it
        if (n > 0 && prev >= 0 &&
            !wait_bar(bar(C::B_OFREE + (prev & 1)), uint32_t(prev >> 1) & 1u, abort_flag, err, 14)) {
          ok = false;
          break;
        }
        for (int j = 0; j < n; ++j) {
          const int pb = np % C::NS, vs = nvc % C::NV;
          if (!wait_bar(bar(C::B_VFULL + vs), uint32_t(nvc / C::NV) & 1u, abort_flag, err, 6)) { ok = false; break; }
          if (!wait_bar(bar(C::B_PFULL + pb), uint32_t(np / C::NS) & 1u, abort_flag, err, 5)) { ok = false; break; }
          ptx::tc_fence_after();
          issue_pv<D>(tmem + C::col_o(ob), tmem + C::col_s(pb), vdesc0 + uint64_t(vs) * (C::TILE >> 4), j > 0);
          // P(j) and V(j) are read by no later MMA
          ptx::mma_commit(bar(C::B_PDONE + pb));
          ptx::mma_commit(bar(C::B_VEMPTY + vs));
          ++np;
          ++nvc;
        }
        // The item's last P.V: O is final once this arrives (at once for an
        // item without entries).
        if (ok) ptx::mma_commit(bar(C::B_ODONE + (k & 1)));
      }
      ptx::mma_commit(bar(C::B_DRAIN));
      drain_bar(bar(C::B_DRAIN), 0, err);
    }
    __syncwarp();
   }
  } else {
    ptx::regs_inc<Regs<kDense>::softmax>();
    // ------------------------------------------------------------ softmax
    // Two threads per query row: warps 0-3 take score columns 0-63 of every
    // k-tile, warps 4-7 columns 64-127.  Both halves keep the same exponent
    // reference m (and each its own part of the row sum l); O is shared.  Per
    // k-tile each half posts its maximum for the other and takes its
    // exponentials with the current reference right away; only when the row
    // maximum rises by more than the threshold (rare after the first k-tile)
    // are they taken again with the new reference.
    const int hf = warp >> 2;                  // which half of the columns
    const int quarter = warp & 3;              // TMEM lanes this warp may access
    const int r = quarter * 32 + lane;         // query row inside the tile = TMEM lane
    const int kind = p.mask.kind;
    const uint32_t lane_base = tmem + (uint32_t(quarter * 32) << 16);
    constexpr int DH = D / 2;                  // O columns this half rescales and writes
    const uint32_t col_oh = uint32_t(DH * hf);  // this half's O columns, from its buffer's first
    const float c2 = p.scale_log2;
    const float2 c22 = make_float2(c2, c2);
    float* xmax = reinterpret_cast<float*>(sbase + C::OFF_XMAX);  // [entry parity][half][row]
    float* stats = reinterpret_cast<float*>(sbase + C::OFF_STATS);  // [item parity][l0, l1, m][row]
    int nsf = 0;     // k-tile entries processed (all items): S buffer nsf % NS
    int up = 0;      // PARTIAL entries with key codes (all items): code buffer up % NCODE
    bool ok = true;
    for (int k = 0; ok; ++k) {
      if (!warp_wait(bar(C::B_IFULL + (k & 1)), uint32_t(k >> 1) & 1u, abort_flag, err, 16)) break;
      Item it;
      const bool valid = load_item(item_ring + 8 * (k & 1), it);
      ptx::mbar_arrive(bar(C::B_IEMPTY + (k & 1)));
      if (!valid) break;
      const int qn = min(kTile, it.L - it.qi0);
      const bool row_in = r < qn;
      const int il = it.qi0 + r;               // local query index
      const int s0 = it.s0, L = it.L;
      const int qcode = (row_in && kind_codes(kind)) ? query_code(p.mask, s0 + il) : 0;
      // The rows of a warp usually share one query code (one document, one
      // turn).  A key's visibility is then the same for all of them, and one
      // ballot over the keys' codes replaces 32 tests per row.
      const int qcode_w = __shfl_sync(0xffffffffu, qcode, 0);
      const bool uniform_q = __all_sync(0xffffffffu, !row_in || qcode == qcode_w);
      float m_ref = -INFINITY, l = 0.f;
      int cnt_item = 0;
      for (int e = it.e0; e < it.e1; ++e) {
        const int j0 = __ldg(p.kidx + e) * kTile, kn = min(kTile, L - j0);
        const int lab = __ldg(p.klabel + e);
        // the dense kind's bits of this row for a PARTIAL tile, loaded before
        // the wait for the scores so that their latency hides behind it
        uint32_t dwords[2] = {0u, 0u};
        if constexpr (kDense) {
          if (lab == ATTN_TILE_PARTIAL && row_in) {
#pragma unroll
            for (int q = 0; q < 2; ++q)
              if (64 * hf + 32 * q < kn) dwords[q] = dense_word(p.mask, it.b, L, il, ((j0 + 64 * hf) >> 5) + q);
          }
        }
        const int sb = nsf % C::NS, xb = nsf & 1;
        const uint32_t col_s = C::col_s(sb) + 64u * hf;  // this half's 64 score columns; its P goes
                                                         // over the first 32 of them
        if (!warp_wait(bar(C::B_SFULL + sb), uint32_t(nsf / C::NS) & 1u, abort_flag, err, 8)) { ok = false; break; }
        ptx::tc_fence_after();
        float s[64];
        {
          uint32_t v[2][32];
          ptx::tmem_ld32(lane_base + col_s, v[0]);
          ptx::tmem_ld32(lane_base + col_s + 32, v[1]);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(v[c >> 5][c & 31]);
        }
        if (lab == ATTN_TILE_PARTIAL || kn < kTile) {
          // bit c of vis[c / 32]: key column 64 * hf + c is visible to this row.
          // Causal part and bounds: columns below upto; PARTIAL tiles of the
          // metadata kinds also AND in the per-key predicate, those of the
          // dense kind the caller's bits.
          const int upto = (lab == ATTN_TILE_PARTIAL && (!kDense && kind_causal(kind)) ? min(kn, il - j0 + 1) : kn) -
                           64 * hf;
          uint32_t vis[2] = {prefix_bits(upto), prefix_bits(upto - 32)};
          if (kDense && lab == ATTN_TILE_PARTIAL) {
            vis[0] &= dwords[0];  // zero for rows past the end
            vis[1] &= dwords[1];
          } else if (!kDense && lab == ATTN_TILE_PARTIAL && kind_codes(kind)) {
            // the K producer staged this entry's key codes
            const int cb = up % C::NCODE;
            if (!warp_wait(bar(C::B_CODE + cb), uint32_t(up / C::NCODE) & 1u, abort_flag, err, 9)) {
              ok = false;
              break;
            }
            const int* codes = key_codes + cb * kTile + 64 * hf;
            if (uniform_q) {
              const int kc0 = codes[lane], kc1 = codes[32 + lane];
              if (kind == ATTN_MASK_STRIP_THINKING) {
                vis[0] &= __ballot_sync(0xffffffffu, code_visible(ATTN_MASK_STRIP_THINKING, qcode_w, kc0));
                vis[1] &= __ballot_sync(0xffffffffu, code_visible(ATTN_MASK_STRIP_THINKING, qcode_w, kc1));
              } else if (kind == ATTN_MASK_SHARED_PREFIX) {
                vis[0] &= __ballot_sync(0xffffffffu, code_visible(ATTN_MASK_SHARED_PREFIX, qcode_w, kc0));
                vis[1] &= __ballot_sync(0xffffffffu, code_visible(ATTN_MASK_SHARED_PREFIX, qcode_w, kc1));
              } else if (kind == ATTN_MASK_STRIP_THINKING_DUP) {
                vis[0] &= __ballot_sync(0xffffffffu, dup_visible(qcode_w, kc0));
                vis[1] &= __ballot_sync(0xffffffffu, dup_visible(qcode_w, kc1));
              } else {
                vis[0] &= __ballot_sync(0xffffffffu, code_visible(ATTN_MASK_CAUSAL_DOCUMENT, qcode_w, kc0));
                vis[1] &= __ballot_sync(0xffffffffu, code_visible(ATTN_MASK_CAUSAL_DOCUMENT, qcode_w, kc1));
              }
            } else if (kind == ATTN_MASK_STRIP_THINKING) {
#pragma unroll
              for (int q = 0; q < 2; ++q)
                if (vis[q]) vis[q] &= code_word<ATTN_MASK_STRIP_THINKING>(codes, q, qcode);
            } else if (kind == ATTN_MASK_SHARED_PREFIX) {
#pragma unroll
              for (int q = 0; q < 2; ++q)
                if (vis[q]) vis[q] &= code_word<ATTN_MASK_SHARED_PREFIX>(codes, q, qcode);
            } else if (kind == ATTN_MASK_CAUSAL_DOCUMENT) {
#pragma unroll
              for (int q = 0; q < 2; ++q)
                if (vis[q]) vis[q] &= code_word<ATTN_MASK_CAUSAL_DOCUMENT>(codes, q, qcode);
            } else {
#pragma unroll
              for (int q = 0; q < 2; ++q)
                if (vis[q]) vis[q] &= code_word_rt(kind, codes, q, qcode);
            }
            // done with the buffer
            ptx::mbar_arrive(bar(C::B_CODEFREE + cb));
            ++up;
          }
          // A word the whole warp sees needs no select.
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            if (__all_sync(0xffffffffu, vis[q] == 0xffffffffu)) continue;
#pragma unroll
            for (int c = 0; c < 32; ++c) s[32 * q + c] = (vis[q] >> c) & 1u ? s[32 * q + c] : -INFINITY;
          }
        }
        float mx4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float mv = s[16 * u];
#pragma unroll
          for (int c = 1; c < 15; c += 2) mv = ptx::fmax3(mv, s[16 * u + c], s[16 * u + c + 1]);
          mx4[u] = fmaxf(mv, s[16 * u + 15]);
        }
        const float mh = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * c2;
        // post this half's maximum for the other half of the row
        xmax[(xb * 2 + hf) * kTile + r] = mh;
        ptx::mbar_arrive(bar(C::B_XMAX + xb));
        // p = 2^(s c2 - m) for the 64 columns, written as bf16 over this half's
        // first 32 S columns; returns the partial row sum.
        auto exp_pass = [&](float m) -> float {
          const float2 nm2 = make_float2(-m, -m);
          float2 sum2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                            make_float2(0.f, 0.f)};
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              const float2 x = ptx::ffma2(make_float2(s[32 * hh + c], s[32 * hh + c + 1]), c22, nm2);
              const float2 e2 = make_float2(ptx::ex2(x.x), ptx::ex2(x.y));
              sum2[(c >> 1) & 3] = ptx::fadd2(sum2[(c >> 1) & 3], e2);
              pk[c >> 1] = ptx::pack_bf16(e2.x, e2.y);
            }
            ptx::tmem_st16(lane_base + col_s + hh * 16, pk);
          }
          const float2 sa = ptx::fadd2(sum2[0], sum2[1]), sb2 = ptx::fadd2(sum2[2], sum2[3]);
          return (sa.x + sb2.x) + (sa.y + sb2.y);
        };
        // With a reference in every row of the warp, the exponentials need not
        // wait for the other half's maximum.
        const bool early = !__any_sync(0xffffffffu, m_ref == -INFINITY);
        float psum = early ? exp_pass(m_ref) : 0.f;
        if (!warp_wait(bar(C::B_XMAX + xb), uint32_t(nsf >> 1) & 1u, abort_flag, err, 17)) { ok = false; break; }
        const float mxs = fmaxf(mh, xmax[(xb * 2 + (1 - hf)) * kTile + r]);  // the same in both halves
        const bool raise = mxs > m_ref + kRescaleThreshold;  // always true on the first visible key
        if (!early || __any_sync(0xffffffffu, raise)) {
          const bool rescale = raise && m_ref != -INFINITY;  // O and l hold an older reference
          const float m_new = raise ? mxs : m_ref;
          const float alpha = rescale ? ptx::ex2(m_ref - m_new) : 1.f;
          if (cnt_item > 0 && __any_sync(0xffffffffu, rescale)) {
            // O must hold exactly the P.V of the earlier entries: wait for the
            // last of them.  Each half rescales its half of the O columns.
            const int pl = nsf - 1;
            if (!warp_wait(bar(C::B_PDONE + pl % C::NS), uint32_t(pl / C::NS) & 1u, abort_flag, err, 12)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const float2 a2 = make_float2(alpha, alpha);
#pragma unroll 1
            for (int q = 0; q < DH / 16; ++q) {
              uint32_t v[16];
              ptx::tmem_ld16(lane_base + C::col_o(k % C::NO) + col_oh + q * 16, v);
              ptx::tmem_wait_ld();
#pragma unroll
              for (int c = 0; c < 16; c += 2) {
                const float2 x = ptx::fmul2(make_float2(__uint_as_float(v[c]), __uint_as_float(v[c + 1])), a2);
                v[c] = __float_as_uint(x.x);
                v[c + 1] = __float_as_uint(x.y);
              }
              ptx::tmem_st16(lane_base + C::col_o(k % C::NO) + col_oh + q * 16, v);
            }
          }
          l *= alpha;
          m_ref = m_new;
          psum = exp_pass(m_ref == -INFINITY ? 0.f : m_ref);
        }
        l += psum;
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(C::B_PFULL + sb));
        ++nsf;
        ++cnt_item;
      }
      if (!ok) break;
      // ---------------------------------------------------------- row statistics
      // Post this half's row sum (and, from the first half, the reference m)
      // for the epilogue warps, once they have read the same buffer two items
      // ago; then straight on to the next item.
      {
        const int ob = k & 1;
        if (k >= 2 && !warp_wait(bar(C::B_OFREE + ob), uint32_t((k >> 1) - 1) & 1u, abort_flag, err, 19)) break;
        float* st = stats + ob * 3 * kTile;
        st[hf * kTile + r] = l;
        if (hf == 0) st[2 * kTile + r] = m_ref;
        ptx::mbar_arrive(bar(C::B_STATS + ob));
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kWarpPV) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (threadIdx.x == 0) finish_sched(p.sched);
}


template <int D, bool kDense>
attn_status launch(const FwdArgs& a, cudaStream_t s) {
  using C = Cfg<D>;
  CUtensorMap mq, mk, mv;
  if (!make_map<D>(&mq, a.q, a.total_tokens, a.num_heads) ||
      !make_map<D>(&mk, a.k, a.total_tokens, a.num_heads) ||
      !make_map<D>(&mv, a.v, a.total_tokens, a.num_heads))
    return record_cuda_error(cudaErrorInvalidValue, "attn_fwd tensor map encoding");
  // per launch, for the current device (the setting is per device and context)
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_bf16_kernel<D, kDense>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
  if (e != cudaSuccess) return record_cuda_error(e, "attn_fwd configure");
  int num_sms = 0;
  e = current_sm_count(&num_sms);
  if (e != cudaSuccess) return record_cuda_error(e, "attn_fwd device query");
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
  p.sched = next_sched_slot();
  // Persistent: one CTA per SM (the q-tile count is only known on the device;
  // max_qt * H bounds the item count).
  const long long items = (long long)a.bm.max_qt * a.num_heads;
  if (items <= 0 || items > INT_MAX) return ATTN_ERR_UNSUPPORTED;
  const long long grid = items < num_sms ? items : num_sms;
  attn_fwd_bf16_kernel<D, kDense><<<unsigned(grid), kThreads, C::SMEM_ALLOC, s>>>(mq, mk, mv, p);
  e = cudaGetLastError();
  return e == cudaSuccess ? ATTN_OK : record_cuda_error(e, "attn_fwd launch");
}

}  // namespace

attn_status launch_attn_fwd_bf16(const FwdArgs& a, cudaStream_t s) {
  const bool dense = a.mask.kind == ATTN_MASK_DENSE;
  switch (a.head_dim) {
    case 32: return dense ? launch<32, true>(a, s) : launch<32, false>(a, s);
    case 64: return dense ? launch<64, true>(a, s) : launch<64, false>(a, s);
    case 128: return dense ? launch<128, true>(a, s) : launch<128, false>(a, s);
  }
  return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attnmask
