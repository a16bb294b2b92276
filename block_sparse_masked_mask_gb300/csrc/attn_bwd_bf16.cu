// bf16 attention backward on the sm_103a tensor cores (tcgen05 + TMA + TMEM).
//
// Gradients of O = softmax(scale Q K^T, masked) V for an upstream dO, with the
// forward's LSE: P = exp(scale S - LSE) is recomputed tile by tile, and
//   dV = P^T dO,  dP = dO V^T,  D_i = sum_d dO_id O_id,  dS = P * (dP - D),
//   dQ = scale dS K,  dK = scale dS^T Q.
// The xorl issue (Verified FA4 gaps, items 1-3) asks for this backward over
// the block-sparse masks, walking the transposed (k-major) lists for dK and
// dV, and with a deterministic dQ.  Four kernels:
//   * delta: D = rowsum(dO * O) per (token, head), fp32;
//   * kpos: for every q-major entry, its position in the k-major lists;
//   * dK/dV: one work item per (k-tile, head) walks its k-major list of
//     q-tiles, recomputing S^T and dP^T, accumulating dK and dV in TMEM (K, V
//     stay in shared memory), and stores every dS tile once as a 32 KB bf16
//     block in the caller's workspace;
//   * dQ: one work item per (q-tile, head) walks its q-major list of k-tiles
//     and accumulates dQ = scale dS K in TMEM from the stored blocks.  dQ is a
//     sum over k-tiles in a fixed order inside one CTA, so it is
//     bit-reproducible, with no atomics.
// Five products per tile pair (S, dP, dV, dK, dQ); the masks are applied on
// PARTIAL tiles only and EMPTY tiles are never loaded.  Warp roles: dK/dV
// (384 threads) eight row warps (two per TMEM lane quarter, one per half of
// the queries), the TMA producer, the tcgen05 issuer, two idle; dQ (256
// threads) four epilogue warps, the producer and the issuer.  Every mbarrier
// wait is bounded as in the forward.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "ptx.cuh"
#include "tile_pipeline.cuh"

namespace attnmask {
namespace {

constexpr int kBwdThreads = 256;                        // dQ kernel: 4 epilogue warps, producer, MMA
constexpr int kDkdvThreads = 384;                       // dK/dV kernel: 8 row warps, producer, MMA, 2 idle
constexpr int kDkdvLoad = 8, kDkdvMma = 9;
// The producers copy an item's list to shared memory this many entries at a
// time, so that no list read sits between a free slot and the next copy.
constexpr int kPlist = 256;
constexpr int kWarpLoad = 4, kWarpMma = 5;

// ---------------------------------------------------------------------------
// D = rowsum(dO * O): D / 8 lanes per (token, head) row, 16 bytes of O and of
// dO per lane (eight bf16 each), so that every load moves whole sectors.
template <int D>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const __nv_bfloat16* __restrict__ o,
                                                        const __nv_bfloat16* __restrict__ dout,
                                                        float* __restrict__ delta, int T, int H) {
  constexpr int LPR = D / 8;                      // lanes per row: 16, 8 or 4
  constexpr int RPB = 256 / LPR;                  // rows per block
  const int sub = threadIdx.x % LPR;
  const long long row = (long long)blockIdx.x * RPB + threadIdx.x / LPR;  // t * H + h
  const bool in = row < (long long)T * H;
  float acc = 0.f;
  if (in) {
    const uint4 a = *reinterpret_cast<const uint4*>(o + row * D + 8 * sub);
    const uint4 g = *reinterpret_cast<const uint4*>(dout + row * D + 8 * sub);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&aw[i]));
      const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[i]));
      acc = fmaf(x.x, y.x, fmaf(x.y, y.y, acc));
    }
  }
#pragma unroll
  for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (in && sub == 0) {
    const int t = int(row / H), h = int(row % H);
    delta[size_t(h) * T + t] = acc;
  }
}

// ---------------------------------------------------------------------------
// Shared layout of the two list-walking kernels.
template <int D>
struct BwdCfg : TileLayout<D> {
  using TileLayout<D>::TILE;
  using TileLayout<D>::CHUNK;
  using TileLayout<D>::CE;
  using TileLayout<D>::NCH;
  using TileLayout<D>::ROWB;
  static constexpr int NSLOT = 4;  // ring of streamed tiles (two per list entry)
  // fixed tiles (Q and dO for dQ; K and V for dK/dV), then the ring
  static constexpr int OFF_A = 0, OFF_B = TILE, OFF_RING = 2 * TILE;
  static constexpr int B_FIX = 0, B_FIXFREE = 1, B_FULL = 2, B_EMPTY = 2 + NSLOT, B_VTMA = 2 + 2 * NSLOT,
                       B_SFULL = B_VTMA + 1, B_PFULL = B_SFULL + 1, B_ODONE = B_PFULL + 2,
                       B_OFREE = B_ODONE + 1, B_IFULL = B_OFREE + 1, B_IEMPTY = B_IFULL + 2,
                       B_DRAIN = B_IEMPTY + 2, B_YFREE = B_DRAIN + 1, NBAR = B_YFREE + 1;
  static constexpr int OFF_BAR = OFF_RING + NSLOT * TILE;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int OFF_RINGI = OFF_MISC + 16;                 // two decoded work items, 8 ints each
  // per ring slot: 128 ints of side data (key codes, or the q-tile's LSE, D and
  // query codes: 3 x 128 words for the dK/dV kernel's Q slots)
  static constexpr int OFF_SIDE = (OFF_RINGI + 2 * 8 * 4 + 15) & ~15;
  static constexpr int SIDE_WORDS = 3 * kTile;
  static constexpr int OFF_STAGE = OFF_SIDE + NSLOT * SIDE_WORDS * 4;  // per warp: 16 output rows
  static constexpr int STAGE_WARP = 2048;                       // per row warp: output rows in rounds
  static constexpr int OFF_PLIST = OFF_STAGE + 8 * STAGE_WARP;  // the producer's staged list
  static constexpr int SMEM_USED = OFF_PLIST + 2 * kPlist * 4;
  static constexpr int SMEM_ALLOC = SMEM_USED + 1024 > 116 * 1024 ? SMEM_USED + 1024 : 116 * 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
};

struct BwdParams {
  int32_t* header;
  int sched;              // this launch's work-counter slot
  const int32_t* order;   // items' tile order (q-major for dQ, k-major for dK/dV)
  const int32_t* qt_seq;
  const int32_t* qt_idx;
  const int32_t* off;     // CSR offsets of the walked lists
  const int32_t* idx;     // tile index inside the sequence
  const uint8_t* label;
  const int32_t* cu;
  MaskArgs mask;
  const float* lse;       // [H, T]
  const float* delta;     // [H, T]
  __nv_bfloat16* out0;    // dQ, or dK
  __nv_bfloat16* out1;    // unused, or dV
  uint8_t* ds;            // dS blocks of heads h0 .. h0+G-1: [G][entries][128 x 128 bf16]
  const int32_t* kpos;    // k-major position of every q-major entry
  int H, T;
  int h0, G;              // heads of this launch
  int e_bound;            // entries the dS blocks were sized for
  float scale;
  float scale_log2;
};

// Bytes of one stored dS block: 128 keys x 128 queries, bf16.
constexpr int kDsBlock = kTile * kTile * 2;

// One work item: a tile of one sequence and one head, and its list.
struct BwdItem {
  int h, s0, L, i0, e0, e1, b;  // i0: first row of the item's tile, local to the sequence
};

__device__ __forceinline__ BwdItem bwd_decode(const BwdParams& p, int item, int n_t) {
  BwdItem it;
  it.h = p.h0 + item / n_t;
  const int g = p.order[item % n_t];
  const int b = p.qt_seq[g];
  it.s0 = p.cu[b];
  it.L = p.cu[b + 1] - it.s0;
  it.i0 = p.qt_idx[g] * kTile;
  it.e0 = p.off[g];
  it.e1 = p.off[g + 1];
  it.b = b;
  return it;
}

__device__ __forceinline__ void bwd_store(volatile int* d, const BwdItem& it, bool valid) {
  d[0] = valid ? 1 : 0;
  d[1] = it.h;
  d[2] = it.s0;
  d[3] = it.L;
  d[4] = it.i0;
  d[5] = it.e0;
  d[6] = it.e1;
  d[7] = it.b;
}
__device__ __forceinline__ bool bwd_load(const volatile int* d, BwdItem& it) {
  if (!d[0]) return false;
  it.h = d[1];
  it.s0 = d[2];
  it.L = d[3];
  it.i0 = d[4];
  it.e0 = d[5];
  it.e1 = d[6];
  it.b = d[7];
  return true;
}

// The producer takes a ticket and publishes the item in ring slot k & 1.
__device__ __forceinline__ int bwd_publish(const BwdParams& p, int k, int lane, int n_items, int n_t, BwdItem& it,
                                           volatile int* ring, uint32_t iempty0, uint32_t ifull0,
                                           volatile uint32_t* abort_flag, int32_t* err) {
  int ticket = 0;
  if (lane == 0) ticket = take_ticket(p.sched);
  ticket = __shfl_sync(0xffffffffu, ticket, 0);
  const bool valid = ticket < n_items;
  if (valid) it = bwd_decode(p, ticket, n_t);
  const int slot_i = k & 1;
  if (k >= 2 && !warp_wait(iempty0 + 8u * slot_i, uint32_t((k >> 1) - 1) & 1u, abort_flag, err, 15)) return -1;
  if (lane == 0) {
    bwd_store(ring + 8 * slot_i, it, valid);
    ptx::mbar_arrive(ifull0 + 8u * slot_i);
  }
  return valid ? 1 : 0;
}

// Write this warp's 32 rows of COLS bf16 values (`w`, packed pairs) to rows
// 0 .. nrows-1 of `base` (row stride `rstride` elements) as whole 16-byte
// pieces, a few rows at a time through the warp's STAGE-byte shared-memory
// stage (pieces XOR-swizzled by row so that neither side has bank conflicts).
template <int COLS, int STAGE>
__device__ __forceinline__ void store_rows(uint8_t* stage, int lane, const uint32_t (&w)[COLS / 2],
                                           __nv_bfloat16* base, size_t rstride, int nrows) {
  constexpr int RB = COLS * 2;                              // bytes per row
  constexpr int CPR = RB / 16;                              // 16-byte pieces per row
  constexpr int RPI = 32 / CPR;                             // rows per warp-wide store
  constexpr int RR = STAGE / RB < 32 ? STAGE / RB : 32;     // rows per round
  static_assert(RR >= RPI && RR % RPI == 0 && 32 % RR == 0, "stage too small");
#pragma unroll
  for (int round = 0; round < 32 / RR; ++round) {
    if (lane / RR == round) {
      const int q = lane % RR;
#pragma unroll
      for (int c = 0; c < CPR; ++c)
        *reinterpret_cast<uint4*>(stage + q * RB + ((c ^ q) & (CPR - 1)) * 16) =
            make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < RR / RPI; ++i) {
      const int q = i * RPI + lane / CPR, c = lane % CPR;
      const int rr = round * RR + q;
      const uint4 val = *reinterpret_cast<const uint4*>(stage + q * RB + ((c ^ q) & (CPR - 1)) * 16);
      if (rr < nrows) *reinterpret_cast<uint4*>(base + size_t(rr) * rstride + 8 * c) = val;
    }
    __syncwarp();
  }
}

// A stored dS block is the image, in shared memory, of a 128-query x 128-key
// bf16 operand in the MN-major layout without swizzle: sixteen 2 KB chunks of
// eight queries; in chunk c, key k's eight queries q = 8c .. 8c+7 are the 16
// bytes at k * 16.  One bulk copy of the 32 KB gives the dQ kernel its A
// operand (8-key core matrices 128 bytes apart along K, chunks 2 KB apart
// along M), and a thread that holds one key's dS for 64 queries writes it
// straight from registers: for each chunk the 32 lanes of a warp (32
// consecutive keys) write 512 contiguous bytes.
constexpr int kDsChunk = 2048;  // bytes per eight-query chunk of a dS block

// TMEM -> registers: D fp32 columns of this thread's lane from `taddr`, times
// `mul`, rounded to bf16 pairs (zeros when `have` is false).
template <int D>
__device__ __forceinline__ void tmem_row_bf16(uint32_t taddr, float mul, bool have, uint32_t (&w)[D / 2]) {
#pragma unroll
  for (int q = 0; q < D / 32; ++q) {
    uint32_t v[32];
    if (have) {
      ptx::tmem_ld32(taddr + 32 * q, v);
      ptx::tmem_wait_ld();
    } else {
#pragma unroll
      for (int c = 0; c < 32; ++c) v[c] = 0u;
    }
#pragma unroll
    for (int c = 0; c < 16; ++c)
      w[16 * q + c] = ptx::pack_bf16(__uint_as_float(v[2 * c]) * mul, __uint_as_float(v[2 * c + 1]) * mul);
  }
}

// Producer: rows [row0, row0 + 128) of head h from maps ma and mb into ring
// slots sa and sb, completing FULL + slot.  When only `valid` < 128 rows
// belong to the sequence, both copies complete the tail barrier instead and
// the other rows are zeroed before FULL opens: they hold the next sequence's
// values (or the zero fill past the tensor), and an inf there would turn the
// zero weights these rows get in the products into NaN.
template <int D>
__device__ __forceinline__ bool load_pair(const CUtensorMap* ma, const CUtensorMap* mb, int h, int row0, int valid,
                                          uint32_t ring, uint8_t* ring_gen, int sa, int sb, uint32_t full0,
                                          uint32_t tail_bar, int& ntail, bool& tail_pending, int lane,
                                          volatile uint32_t* abort_flag, int32_t* err) {
  using C = BwdCfg<D>;
  const uint32_t da = ring + uint32_t(sa) * C::TILE, db = ring + uint32_t(sb) * C::TILE;
  const bool tail = valid < kTile;
  const uint32_t ba = tail ? tail_bar : full0 + 8u * uint32_t(sa);
  const uint32_t bb = tail ? tail_bar : full0 + 8u * uint32_t(sb);
  if (lane == 0) {
    if (tail) {
      ptx::mbar_arrive_expect_tx(tail_bar, 2 * C::TILE);
    } else {
      ptx::mbar_arrive_expect_tx(ba, C::TILE);
      ptx::mbar_arrive_expect_tx(bb, C::TILE);
    }
#pragma unroll
    for (int c = 0; c < C::NCH; ++c) {
      ptx::tma_load_3d(da + c * C::CHUNK, ma, ba, c * C::CE, h, row0);
      ptx::tma_load_3d(db + c * C::CHUNK, mb, bb, c * C::CE, h, row0);
    }
  }
  if (!tail) return true;
  tail_pending = true;
  if (!warp_wait(tail_bar, uint32_t(ntail) & 1u, abort_flag, err, 2)) return false;
  tail_pending = false;
  ++ntail;
  for (int rr = valid + lane; rr < kTile; rr += 32) {
#pragma unroll
    for (int c = 0; c < C::NCH; ++c) {
      uint4* ra = reinterpret_cast<uint4*>(ring_gen + sa * C::TILE + c * C::CHUNK + rr * C::ROWB);
      uint4* rb = reinterpret_cast<uint4*>(ring_gen + sb * C::TILE + c * C::CHUNK + rr * C::ROWB);
#pragma unroll
      for (int x = 0; x < C::ROWB / 16; ++x) {
        ra[x] = make_uint4(0u, 0u, 0u, 0u);
        rb[x] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
  ptx::fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    ptx::mbar_arrive(full0 + 8u * uint32_t(sa));
    ptx::mbar_arrive(full0 + 8u * uint32_t(sb));
  }
  return true;
}

// Half `hf` of a product over the 128 rows of a streamed tile: k-steps
// 4hf .. 4hf+3 of issue_pv (rows 64hf .. 64hf+63), so that the first half can
// run while the row threads still produce the second.
template <int D>
__device__ __forceinline__ void issue_pv_half(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, int hf, bool acc) {
  using C = BwdCfg<D>;
#pragma unroll
  for (int k4 = 0; k4 < 4; ++k4) {
    const int kk = 4 * hf + k4;
    ptx::mma_ts(d_tmem, a_tmem + uint32_t(hf) * 64u + uint32_t(k4) * 8u, b_desc + v_step<D>(kk), C::IDESC_PV,
                (acc || kk > 0) ? 1u : 0u);
  }
}

// ---------------------------------------------------------------------------
// dQ from the stored dS blocks: one item per (q-tile, head); per listed k-tile
// j, dQ += dS(i, j) K_j, with dS(i, j) the block the dK/dV kernel wrote for the
// pair (bulk-copied as the MN-major A operand) and K_j the MN-major B operand.
// Warps 0-3 are the epilogue (one thread per query row), warp 4 the producer,
// warp 5 the MMA issuer; dQ is double-buffered in TMEM so one item's epilogue
// runs under the next item's products.  Each dQ row is a sum over its k-tiles
// in ascending order inside one CTA: deterministic.
template <int D>
struct DqCfg : TileLayout<D> {
  using TileLayout<D>::TILE;
  using TileLayout<D>::CHUNK;
  using TileLayout<D>::CE;
  using TileLayout<D>::NCH;
  using TileLayout<D>::ROWB;
  static constexpr int SLOT = kDsBlock + TILE;  // dS block, then the K tile
  static constexpr int NSLOT = D == 128 ? 3 : 4;
  static constexpr int B_FULL = 0, B_EMPTY = NSLOT, B_TAIL = 2 * NSLOT, B_ODONE = B_TAIL + 1,
                       B_OFREE = B_ODONE + 2, B_IFULL = B_OFREE + 2, B_IEMPTY = B_IFULL + 2,
                       B_DRAIN = B_IEMPTY + 2, NBAR = B_DRAIN + 1;
  static constexpr int OFF_BAR = NSLOT * SLOT;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int OFF_RINGI = OFF_MISC + 16;
  static constexpr int OFF_STAGE = (OFF_RINGI + 2 * 8 * 4 + 15) & ~15;
  static constexpr int STAGE_WARP = 16 * 2 * D;
  static constexpr int OFF_PLIST = OFF_STAGE + 4 * STAGE_WARP;  // the producer's staged list
  static constexpr int SMEM_USED = OFF_PLIST + 2 * kPlist * 4;
  static constexpr int SMEM_ALLOC = SMEM_USED + 1024 > 116 * 1024 ? SMEM_USED + 1024 : 116 * 1024;
  static constexpr uint32_t DQ_COLS = D;                          // one dQ buffer
  static constexpr uint32_t TMEM_COLS = 2 * D < 32 ? 32 : 2 * D;  // two buffers
  // dS as the A operand: M = 128 queries (sixteen 8-query chunks), K = keys
  static constexpr uint32_t IDESC_DQ = ptx::idesc_bf16_f32(128, D, true, true);
  static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
};

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmK, const BwdParams p) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_t = p.header[kHdrQtiles];
  const int n_entries = p.header[kHdrEntries];
  const int n_items = n_t * p.G;
  int32_t* err = p.header + kHdrError;
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);
  const uint32_t sRing = base;
  const uint32_t bars = base + C::OFF_BAR;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  uint32_t* misc = reinterpret_cast<uint32_t*>(sbase + C::OFF_MISC);
  volatile uint32_t* abort_flag = misc + 1;
  volatile int* item_ring = reinterpret_cast<volatile int*>(sbase + C::OFF_RINGI);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NSLOT; ++s) {
      ptx::mbar_init(bar(C::B_FULL + s), 1);
      ptx::mbar_init(bar(C::B_EMPTY + s), 1);
    }
    ptx::mbar_init(bar(C::B_TAIL), 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bar(C::B_ODONE + i), 1);
      ptx::mbar_init(bar(C::B_OFREE + i), 128);
      ptx::mbar_init(bar(C::B_IFULL + i), 1);
      ptx::mbar_init(bar(C::B_IEMPTY + i), 128 + 1);  // epilogue threads, MMA thread
    }
    ptx::mbar_init(bar(C::B_DRAIN), 1);
    *abort_flag = (*reinterpret_cast<volatile int32_t*>(err) & (kErrTimeout | kErrCapacity)) ? 1u : 0u;
    if (n_entries > p.e_bound) {
      atomicOr(err, kErrCapacity);
      *abort_flag = 1u;
    }
    ptx::fence_mbar_init();
  }
  if (warp == kWarpMma) {
    ptx::tmem_alloc(ptx::smem_addr(misc), C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = misc[0];
  const bool skip = *abort_flag != 0u;

  if (skip) {
  } else if (warp == kWarpLoad) {
    // ---------------------------------------------------------- producer
    int nload = 0, ntail = 0;
    bool tail_pending = false, ok = true;
    BwdItem it_next;
    int st_next = bwd_publish(p, 0, lane, n_items, n_t, it_next, item_ring, bar(C::B_IEMPTY), bar(C::B_IFULL),
                              abort_flag, err);
    for (int k = 0; ok && st_next == 1; ++k) {
      const BwdItem it = it_next;
      st_next = bwd_publish(p, k + 1, lane, n_items, n_t, it_next, item_ring, bar(C::B_IEMPTY), bar(C::B_IFULL),
                            abort_flag, err);
      if (st_next < 0) break;
      const uint8_t* ds_head = p.ds + size_t(it.h - p.h0) * size_t(n_entries) * kDsBlock;
      int* s_idx = reinterpret_cast<int*>(sbase + C::OFF_PLIST);
      int* s_pos = s_idx + kPlist;
      for (int e = it.e0; e < it.e1; ++e) {
        const int r = (e - it.e0) & (kPlist - 1);
        if (r == 0) {  // the next kPlist entries of the list and their dS block positions
          __syncwarp();
          for (int x = lane; x < kPlist && e + x < it.e1; x += 32) {
            s_idx[x] = __ldg(p.idx + e + x);
            s_pos[x] = __ldg(p.kpos + e + x);
          }
          __syncwarp();
        }
        const int j0 = s_idx[r] * kTile, kn = min(kTile, it.L - j0);
        const uint8_t* blk = ds_head + size_t(s_pos[r]) * kDsBlock;
        const int slot = nload % C::NSLOT;
        if (nload >= C::NSLOT &&
            !warp_wait(bar(C::B_EMPTY + slot), uint32_t(nload / C::NSLOT - 1) & 1u, abort_flag, err, 1)) {
          ok = false;
          break;
        }
        const uint32_t dst = sRing + uint32_t(slot) * C::SLOT, kdst = dst + kDsBlock;
        const uint32_t full = bar(C::B_FULL + slot);
        if (kn == kTile) {
          if (lane == 0) {
            ptx::mbar_arrive_expect_tx(full, kDsBlock + C::TILE);
            ptx::bulk_load(dst, blk, kDsBlock, full);
            for (int c = 0; c < C::NCH; ++c)
              ptx::tma_load_3d(kdst + c * C::CHUNK, &tmK, full, c * C::CE, it.h, it.s0 + j0);
          }
        } else {
          // K rows past the sequence end are zeroed before FULL opens: their dS
          // is zero, but an inf there would make the product NaN
          if (lane == 0) {
            ptx::mbar_arrive_expect_tx(bar(C::B_TAIL), C::TILE);
            for (int c = 0; c < C::NCH; ++c)
              ptx::tma_load_3d(kdst + c * C::CHUNK, &tmK, bar(C::B_TAIL), c * C::CE, it.h, it.s0 + j0);
          }
          tail_pending = true;
          if (!warp_wait(bar(C::B_TAIL), uint32_t(ntail) & 1u, abort_flag, err, 2)) {
            ok = false;
            break;
          }
          tail_pending = false;
          ++ntail;
          uint8_t* kgen = sbase + size_t(slot) * C::SLOT + kDsBlock;
          for (int rr = kn + lane; rr < kTile; rr += 32) {
#pragma unroll
            for (int c = 0; c < C::NCH; ++c) {
              uint4* row = reinterpret_cast<uint4*>(kgen + c * C::CHUNK + rr * C::ROWB);
#pragma unroll
              for (int x = 0; x < C::ROWB / 16; ++x) row[x] = make_uint4(0u, 0u, 0u, 0u);
            }
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::mbar_arrive_expect_tx(full, kDsBlock);
            ptx::bulk_load(dst, blk, kDsBlock, full);
          }
        }
        ++nload;
      }
    }
    if (lane == 0) {
      for (int s = 0; s < C::NSLOT; ++s) {
        if (nload <= s) continue;
        const int last = s + C::NSLOT * ((nload - 1 - s) / C::NSLOT);
        drain_bar(bar(C::B_FULL + s), uint32_t(last / C::NSLOT) & 1u, err);
      }
      if (tail_pending) drain_bar(bar(C::B_TAIL), uint32_t(ntail) & 1u, err);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int nload = 0;
      bool ok = true;
      // dS: MN-major without swizzle, where the stride between eight-key core
      // matrices (K, 128 bytes) is the leading offset and the stride between
      // eight-query chunks (M, kDsChunk) the stride offset
      const uint64_t ds0 = ptx::smem_desc(sRing, 128u, kDsChunk, ptx::kSwizzleNone);
      const uint64_t k0 = v_base<D>(sRing + kDsBlock);
      for (int k = 0; ok; ++k) {
        if (!wait_bar(bar(C::B_IFULL + (k & 1)), uint32_t(k >> 1) & 1u, abort_flag, err, 16)) break;
        BwdItem it;
        const bool valid = bwd_load(item_ring + 8 * (k & 1), it);
        ptx::mbar_arrive(bar(C::B_IEMPTY + (k & 1)));
        if (!valid) break;
        const int b = k & 1;
        if (k >= 2 && !wait_bar(bar(C::B_OFREE + b), uint32_t((k >> 1) - 1) & 1u, abort_flag, err, 14)) break;
        const uint32_t dq_t = tmem + uint32_t(b) * C::DQ_COLS;
        const int n = it.e1 - it.e0;
        for (int j = 0; j < n; ++j) {
          const int slot = nload % C::NSLOT;
          if (!wait_bar(bar(C::B_FULL + slot), uint32_t(nload / C::NSLOT) & 1u, abort_flag, err, 4)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t so = uint64_t(slot) * (C::SLOT >> 4);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            ptx::mma_ss(dq_t, ds0 + so + uint64_t(kk * 16 * 16 >> 4), k0 + so + v_step<D>(kk), C::IDESC_DQ,
                        (j > 0 || kk > 0) ? 1u : 0u);
          ptx::mma_commit(bar(C::B_EMPTY + slot));
          ++nload;
        }
        if (!ok) break;
        ptx::mma_commit(bar(C::B_ODONE + b));
      }
      ptx::mma_commit(bar(C::B_DRAIN));
      drain_bar(bar(C::B_DRAIN), 0, err);
    }
    __syncwarp();
  } else if (warp < 4) {
    // ---------------------------------------------------------- epilogue
    const uint32_t lane_base = tmem + (uint32_t(warp * 32) << 16);
    for (int k = 0;; ++k) {
      if (!warp_wait(bar(C::B_IFULL + (k & 1)), uint32_t(k >> 1) & 1u, abort_flag, err, 16)) break;
      BwdItem it;
      const bool valid = bwd_load(item_ring + 8 * (k & 1), it);
      ptx::mbar_arrive(bar(C::B_IEMPTY + (k & 1)));
      if (!valid) break;
      const int b = k & 1;
      if (!warp_wait(bar(C::B_ODONE + b), uint32_t(k >> 1) & 1u, abort_flag, err, 11)) break;
      ptx::tc_fence_after();
      uint32_t w[D / 2];
      tmem_row_bf16<D>(lane_base + uint32_t(b) * C::DQ_COLS, p.scale, it.e1 > it.e0, w);
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(C::B_OFREE + b));
      const int qn = min(kTile, it.L - it.i0);
      store_rows<D, C::STAGE_WARP>(sbase + C::OFF_STAGE + warp * C::STAGE_WARP, lane, w,
                    p.out0 + (size_t(it.s0 + it.i0 + warp * 32) * p.H + it.h) * D, size_t(p.H) * D,
                    qn - warp * 32);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (threadIdx.x == 0) finish_sched(p.sched);
}

// k-major position of every q-major entry: for the pair (q-tile i, k-tile j),
// the rank of i in k-tile j's ascending list (one block per q-tile).
__global__ void __launch_bounds__(128) bwd_kpos_kernel(const int32_t* __restrict__ header,
                                                       const int32_t* __restrict__ qt_idx,
                                                       const int32_t* __restrict__ koff,
                                                       const int32_t* __restrict__ kidx,
                                                       const int32_t* __restrict__ qoff,
                                                       const int32_t* __restrict__ qidx, int32_t* kpos) {
  const int g = blockIdx.x;
  if (g >= header[kHdrQtiles]) return;
  const int i = qt_idx[g], g0 = g - i;  // tiles of one sequence are numbered contiguously
  for (int e = koff[g] + threadIdx.x; e < koff[g + 1]; e += blockDim.x) {
    const int gj = g0 + kidx[e];
    int lo = qoff[gj], hi = qoff[gj + 1];
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (qidx[mid] < i) lo = mid + 1;
      else hi = mid;
    }
    kpos[e] = lo;
  }
}

// ---------------------------------------------------------------------------
// dK, dV: one item per (k-tile, head); per listed q-tile i:
//   S^T = K Q_i^T, dP^T = V dO_i^T (TMEM, TMEM lane = key),
//   P^T = 2^(S^T c2 - LSE_i log2 e), dS^T = P^T (dP^T - D_i),
//   dV += P^T dO_i, dK += dS^T Q_i.
// TMEM: dV [0, D), dK [128, 128+D), and two 128-column regions [256,384),
// [384,512) that alternate by entry: S^T of entry j goes to region j % 2 and
// dP^T to the other; the row warps write bf16 P^T and dS^T over S^T's region
// (P^T over the first 32 columns of each 64-column half, dS^T over the other
// 32), so dP^T's region is free once they have read it, and S^T of entry j+1
// goes there while they are still working on entry j.
// Warps 0-7 are the row warps: warp w owns TMEM lanes (keys) 32 (w % 4) ..
// +31 and query columns 64 (w / 4) .. +63, so each half of the queries has its
// own four warps (two warps per SM sub-partition hide each other's latency);
// at the end of an item the first four store dV and the other four dK.  Warp 8
// is the TMA producer, warp 9 the tcgen05 issuer, warps 10-11 idle; the row
// warpgroups run with 192 registers a thread and the third with 112 (within
// the 168 x 384 the block is launched with).
template <int D>
__global__ void __launch_bounds__(kDkdvThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                         const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_t = p.header[kHdrQtiles];
  const int n_entries = p.header[kHdrEntries];
  const int n_items = n_t * p.G;
  int32_t* err = p.header + kHdrError;
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);
  const uint32_t sK = base + C::OFF_A, sV = base + C::OFF_B, sRing = base + C::OFF_RING;
  const uint32_t bars = base + C::OFF_BAR;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  uint32_t* misc = reinterpret_cast<uint32_t*>(sbase + C::OFF_MISC);
  volatile uint32_t* abort_flag = misc + 1;
  volatile int* item_ring = reinterpret_cast<volatile int*>(sbase + C::OFF_RINGI);
  int* side = reinterpret_cast<int*>(sbase + C::OFF_SIDE);
  constexpr uint32_t COL_DV = 0, COL_DK = 128, COL_R0 = 256;

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(C::B_FIX), 1);
    ptx::mbar_init(bar(C::B_FIXFREE), 1);
    for (int s = 0; s < C::NSLOT; ++s) {
      ptx::mbar_init(bar(C::B_FULL + s), (s & 1) ? 1 : 2);  // Q slots: copy + side words
      ptx::mbar_init(bar(C::B_EMPTY + s), 1);
    }
    ptx::mbar_init(bar(C::B_VTMA), 1);
    ptx::mbar_init(bar(C::B_SFULL), 1);
    ptx::mbar_init(bar(C::B_PFULL), 128);
    ptx::mbar_init(bar(C::B_PFULL + 1), 128);
    ptx::mbar_init(bar(C::B_ODONE), 1);
    ptx::mbar_init(bar(C::B_OFREE), 256);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bar(C::B_IFULL + i), 1);
      ptx::mbar_init(bar(C::B_IEMPTY + i), 256 + 1);  // row threads, MMA thread
    }
    ptx::mbar_init(bar(C::B_DRAIN), 1);
    ptx::mbar_init(bar(C::B_YFREE), 256);
    *abort_flag = (*reinterpret_cast<volatile int32_t*>(err) & kErrTimeout) ? 1u : 0u;
    if (n_entries > p.e_bound) {  // the dS blocks cannot hold this mask's entries
      atomicOr(err, kErrCapacity);
      *abort_flag = 1u;
    }
    ptx::fence_mbar_init();
  }
  if (warp == kDkdvMma) {
    ptx::tmem_alloc(ptx::smem_addr(misc), C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = misc[0];
  const bool skip = *abort_flag != 0u;

  if (skip) {
  } else if (warp >= 8) {
    ptx::regs_dec<112>();
    if (warp == kDkdvLoad) {
    // ---------------------------------------------------------- producer
    int nload = 0, ntail = 0, nfix = 0;
    bool tail_pending = false, ok = true;
    BwdItem it_next;
    int st_next = bwd_publish(p, 0, lane, n_items, n_t, it_next, item_ring, bar(C::B_IEMPTY), bar(C::B_IFULL),
                              abort_flag, err);
    for (int k = 0; ok && st_next == 1; ++k) {
      const BwdItem it = it_next;
      st_next = bwd_publish(p, k + 1, lane, n_items, n_t, it_next, item_ring, bar(C::B_IEMPTY), bar(C::B_IFULL),
                            abort_flag, err);
      if (st_next < 0) break;
      // K and V of this k-tile, once the previous item's MMAs no longer read
      // them (rows past the sequence end only reach their own dK, dV rows,
      // which are not stored)
      if (nfix > 0 && !warp_wait(bar(C::B_FIXFREE), uint32_t(nfix - 1) & 1u, abort_flag, err, 13)) break;
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(bar(C::B_FIX), 2 * C::TILE);
        for (int c = 0; c < C::NCH; ++c) {
          ptx::tma_load_3d(sK + c * C::CHUNK, &tmK, bar(C::B_FIX), c * C::CE, it.h, it.s0 + it.i0);
          ptx::tma_load_3d(sV + c * C::CHUNK, &tmV, bar(C::B_FIX), c * C::CE, it.h, it.s0 + it.i0);
        }
      }
      ++nfix;
      // Q(i) and dO(i) of every listed q-tile into two free slots.  Q's side
      // words get the q-tile's LSE (times log2 e; +inf for rows that see no
      // key or lie past the end), D and, on PARTIAL tiles, the query codes;
      // those come from global memory one entry ahead of their use, and the
      // list itself from the staged copy, so a free slot is refilled at once.
      int* s_idx = reinterpret_cast<int*>(sbase + C::OFF_PLIST);
      int* s_lab = s_idx + kPlist;
      float nl[4], ng[4];
      int nc[4];
      int a0 = 0, an = 0, lab = 0;
      auto fetch = [&](int e, int r) {  // list entry e (staged at r, if r >= 0) and its side values
        const int ix = r >= 0 ? s_idx[r] : __ldg(p.idx + e);
        lab = r >= 0 ? s_lab[r] : __ldg(p.label + e);
        a0 = ix * kTile;
        an = min(kTile, it.L - a0);
        const bool codes = kind_codes(p.mask.kind) && lab == ATTN_TILE_PARTIAL;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int c = lane + 32 * m;
          const size_t at = size_t(it.h) * p.T + it.s0 + a0 + c;
          nl[m] = c < an ? __ldg(p.lse + at) : -INFINITY;
          ng[m] = c < an ? __ldg(p.delta + at) : 0.f;
          nc[m] = codes ? query_code(p.mask, it.s0 + a0 + min(c, an - 1)) : 0;
        }
      };
      for (int e = it.e0; e < it.e1; ++e) {
        const int r = (e - it.e0) & (kPlist - 1);
        if (r == 0) {
          __syncwarp();
          for (int x = lane; x < kPlist && e + x < it.e1; x += 32) {
            s_idx[x] = __ldg(p.idx + e + x);
            s_lab[x] = __ldg(p.label + e + x);
          }
          __syncwarp();
          if (e == it.e0) fetch(e, 0);
        }
        const int ca0 = a0, can = an, clab = lab;
        float cl[4], cg[4];
        int cc[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          cl[m] = nl[m];
          cg[m] = ng[m];
          cc[m] = nc[m];
        }
        const int qs = nload % C::NSLOT, ds = (nload + 1) % C::NSLOT;
        if (nload >= C::NSLOT &&
            (!warp_wait(bar(C::B_EMPTY + qs), uint32_t(nload / C::NSLOT - 1) & 1u, abort_flag, err, 1) ||
             !warp_wait(bar(C::B_EMPTY + ds), uint32_t((nload + 1) / C::NSLOT - 1) & 1u, abort_flag, err, 1))) {
          ok = false;
          break;
        }
        if (!load_pair<D>(&tmQ, &tmDO, it.h, it.s0 + ca0, can, sRing, sbase + C::OFF_RING, qs, ds, bar(C::B_FULL),
                          bar(C::B_VTMA), ntail, tail_pending, lane, abort_flag, err)) {
          ok = false;
          break;
        }
        {
          float* sl = reinterpret_cast<float*>(side + qs * C::SIDE_WORDS);
          const bool codes = kind_codes(p.mask.kind) && clab == ATTN_TILE_PARTIAL;
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const int c = lane + 32 * m;
            sl[c] = cl[m] == -INFINITY ? INFINITY : cl[m] * 1.4426950408889634f;
            sl[kTile + c] = cg[m];
            if (codes) side[qs * C::SIDE_WORDS + 2 * kTile + c] = cc[m];
          }
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(bar(C::B_FULL + qs));
        }
        nload += 2;
        if (e + 1 < it.e1) fetch(e + 1, r + 1 < kPlist ? r + 1 : -1);
      }
    }
    if (lane == 0) {
      for (int s = 0; s < C::NSLOT; ++s) {
        if (nload <= s) continue;
        const int last = s + C::NSLOT * ((nload - 1 - s) / C::NSLOT);
        drain_bar(bar(C::B_FULL + s), uint32_t(last / C::NSLOT) & 1u, err);
      }
      if (tail_pending) drain_bar(bar(C::B_VTMA), uint32_t(ntail) & 1u, err);
      if (nfix > 0) drain_bar(bar(C::B_FIX), uint32_t(nfix - 1) & 1u, err);
    }
    __syncwarp();
  } else if (warp == kDkdvMma) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int nload = 0, nent = 0;
      bool ok = true;
      const uint64_t kdesc = kmajor_base<D>(sK), vdesc = kmajor_base<D>(sV);
      const uint64_t rk0 = kmajor_base<D>(sRing), rv0 = v_base<D>(sRing);
      for (int k = 0; ok; ++k) {
        if (!wait_bar(bar(C::B_IFULL + (k & 1)), uint32_t(k >> 1) & 1u, abort_flag, err, 16)) break;
        BwdItem it;
        const bool valid = bwd_load(item_ring + 8 * (k & 1), it);
        ptx::mbar_arrive(bar(C::B_IEMPTY + (k & 1)));
        if (!valid) break;
        if (!wait_bar(bar(C::B_FIX), uint32_t(k) & 1u, abort_flag, err, 3)) { ok = false; break; }
        const int n = it.e1 - it.e0;
        bool s_early = false;  // S^T of the current entry was issued during the previous one
        for (int j = 0; j < n; ++j) {
          const int qs = nload % C::NSLOT, ds = (nload + 1) % C::NSLOT;
          const uint32_t rs = tmem + COL_R0 + 128u * uint32_t(nent & 1);        // S^T, then P^T and dS^T
          const uint32_t rp = tmem + COL_R0 + 128u * uint32_t((nent & 1) ^ 1);  // dP^T
          if (!s_early) {
            if (!wait_bar(bar(C::B_FULL + qs), uint32_t(nload / C::NSLOT) & 1u, abort_flag, err, 4)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            issue_s<D>(rs, kdesc, rk0 + uint64_t(qs) * (C::TILE >> 4));  // S^T = K Q^T
          }
          if (!wait_bar(bar(C::B_FULL + ds), uint32_t((nload + 1) / C::NSLOT) & 1u, abort_flag, err, 4)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          issue_s<D>(rp, vdesc, rk0 + uint64_t(ds) * (C::TILE >> 4));  // dP^T = V dO^T
          ptx::mma_commit(bar(C::B_SFULL));
          if (j == 0 && k > 0 && !wait_bar(bar(C::B_OFREE), uint32_t(k - 1) & 1u, abort_flag, err, 14)) {
            ok = false;
            break;
          }
          // dV += P^T dO and dK += dS^T Q (dO, Q read MN-major), one half of the
          // queries at a time; between the halves, S^T of the next entry
          s_early = false;
          for (int hf = 0; hf < 2 && ok; ++hf) {
            if (!wait_bar(bar(C::B_PFULL + hf), uint32_t(nent) & 1u, abort_flag, err, 5)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            issue_pv_half<D>(tmem + COL_DV, rs, rv0 + uint64_t(ds) * (C::TILE >> 4), hf, j > 0);
            issue_pv_half<D>(tmem + COL_DK, rs + 32u, rv0 + uint64_t(qs) * (C::TILE >> 4), hf, j > 0);
            if (hf == 0 && j + 1 < n) {
              const int nq = (nload + 2) % C::NSLOT;
              if (!wait_bar(bar(C::B_YFREE), uint32_t(nent) & 1u, abort_flag, err, 6) ||
                  !wait_bar(bar(C::B_FULL + nq), uint32_t((nload + 2) / C::NSLOT) & 1u, abort_flag, err, 4)) {
                ok = false;
                break;
              }
              ptx::tc_fence_after();
              issue_s<D>(rp, kdesc, rk0 + uint64_t(nq) * (C::TILE >> 4));
              s_early = true;
            }
          }
          if (!ok) break;
          ptx::mma_commit(bar(C::B_EMPTY + qs));
          ptx::mma_commit(bar(C::B_EMPTY + ds));
          nload += 2;
          ++nent;
        }
        if (!ok) break;
        ptx::mma_commit(bar(C::B_FIXFREE));
        if (n > 0) ptx::mma_commit(bar(C::B_ODONE));
      }
      ptx::mma_commit(bar(C::B_DRAIN));
      drain_bar(bar(C::B_DRAIN), 0, err);
    }
    __syncwarp();
    }
  } else {
    ptx::regs_inc<192>();
    // ---------------------------------------------------------- P^T, dS^T (key rows)
    const int qd = warp & 3, hf = warp >> 2;  // lane quarter, query half
    const int r = qd * 32 + lane;
    const int kind = p.mask.kind;
    const uint32_t lane_base = tmem + (uint32_t(qd * 32) << 16);
    const float c2 = p.scale_log2;
    int nent = 0, nodone = 0, nload = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      if (!warp_wait(bar(C::B_IFULL + (k & 1)), uint32_t(k >> 1) & 1u, abort_flag, err, 16)) break;
      BwdItem it;
      const bool valid = bwd_load(item_ring + 8 * (k & 1), it);
      ptx::mbar_arrive(bar(C::B_IEMPTY + (k & 1)));
      if (!valid) break;
      const int kn = min(kTile, it.L - it.i0);
      const bool row_in = r < kn;
      const int kl = it.i0 + r;  // local key index
      const int kcode = (row_in && kind_codes(kind)) ? key_code(p.mask, it.s0 + kl) : 0;
      const int kbase = it.i0 + qd * 32;  // the warp's first key (local), a multiple of 32
      // keys of a warp usually share one code: then a query's visibility is the
      // same for all of them, and one ballot over the queries' codes gives a word
      const int kcode_w = __shfl_sync(0xffffffffu, kcode, 0);
      const bool uniform_k = __all_sync(0xffffffffu, !row_in || kcode == kcode_w);
      const bool all_in = __all_sync(0xffffffffu, row_in);
      const int n = it.e1 - it.e0;
      int nx_idx = n > 0 ? __ldg(p.idx + it.e0) : 0, nx_lab = n > 0 ? __ldg(p.label + it.e0) : 0;
      for (int jj = 0; jj < n; ++jj) {
        const int e = it.e0 + jj;
        const int a0 = nx_idx * kTile, an = min(kTile, it.L - a0);
        const int lab = nx_lab;
        if (jj + 1 < n) {  // the next entry's list values, one entry ahead
          nx_idx = __ldg(p.idx + e + 1);
          nx_lab = __ldg(p.label + e + 1);
        }
        const int qs = nload % C::NSLOT;
        nload += 2;
        // the dense kind: each lane loads the caller's word of query row
        // a0 + 64 hf + 32 m + lane over the warp's 32 keys, before the wait
        uint32_t dw[2] = {0u, 0u};
        if (kind == ATTN_MASK_DENSE && lab == ATTN_TILE_PARTIAL && kbase < it.L) {
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            const int qrow = a0 + 64 * hf + 32 * m + lane;
            if (qrow < it.L) dw[m] = dense_word(p.mask, it.b, it.L, qrow, kbase >> 5);
          }
        }
        if (!warp_wait(bar(C::B_SFULL), uint32_t(nent) & 1u, abort_flag, err, 8)) { ok = false; break; }
        ptx::tc_fence_after();
        // the q-tile's LSE, D and codes came with Q(i): its load has landed
        if (!warp_wait(bar(C::B_FULL + qs), uint32_t((nload - 2) / C::NSLOT) & 1u, abort_flag, err, 9)) {
          ok = false;
          break;
        }
        const float* sl = reinterpret_cast<const float*>(side + qs * C::SIDE_WORDS);
        // every pair of the warp's rows and columns visible: no masking at all
        const bool fast = lab == ATTN_TILE_FULL && an == kTile && all_in;
        // bit c of vis[m]: query column 64 hf + 32 m + c sees this key.  Causal
        // part and bounds: a0 + column >= kl and column < an.
        uint32_t vis[2] = {0xffffffffu, 0xffffffffu};
        if (!fast) {
          const int lo = kl - a0;  // first visible column
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            const int c0 = 64 * hf + 32 * m;
            vis[m] = lab == ATTN_TILE_PARTIAL && kind_causal(kind) ? ~prefix_bits(lo - c0) & prefix_bits(an - c0)
                                                                   : prefix_bits(an - c0);
          }
          if (lab == ATTN_TILE_PARTIAL && kind == ATTN_MASK_DENSE) {
            // transpose the 32 x 32 bit block: ballot j gathers bit j (key
            // lane j) of every lane's (query's) word, and lane j keeps it
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              uint32_t mine = 0u;
#pragma unroll 4
              for (int j = 0; j < 32; ++j) {
                const uint32_t t = __ballot_sync(0xffffffffu, (dw[m] >> j) & 1u);
                mine = lane == j ? t : mine;
              }
              vis[m] &= mine;
            }
          } else if (lab == ATTN_TILE_PARTIAL && kind_codes(kind)) {
            const int* qc = side + qs * C::SIDE_WORDS + 2 * kTile + 64 * hf;
            if (uniform_k) {
#pragma unroll
              for (int m = 0; m < 2; ++m) {
                vis[m] &= __ballot_sync(0xffffffffu, code_visible(kind, qc[32 * m + lane], kcode_w));
              }
            } else {
#pragma unroll
              for (int m = 0; m < 2; ++m) {
                uint32_t w = 0;
                for (int c = 0; c < 32; ++c) w |= uint32_t(code_visible(kind, qc[32 * m + c], kcode)) << c;
                vis[m] &= w;
              }
            }
          }
          if (!row_in) {
            // a key past the sequence end: its P and dS are exactly zero, so the
            // stored dS block holds no value from another sequence
            vis[0] = vis[1] = 0u;
          }
        }
        // this warp's 64 columns: S^T (both quarters) and dP^T (first quarter)
        // first; dP^T's second quarter loads while the first is computed, after
        // which dP^T's region is released for the next entry's S^T.  Quarter m
        // writes P^T to columns 64 hf + 16 m + [0,16) and dS^T to 64 hf + 32 +
        // 16 m + [0,16) of the S^T region, all of which this warp has read.
        const uint32_t rs = COL_R0 + 128u * uint32_t(nent & 1), rp = COL_R0 + 128u * uint32_t((nent & 1) ^ 1);
        uint32_t sv[2][32], dv0[32], dv1[32];
        uint32_t dsw[32];  // this half's dS (bf16 pairs), kept for the block store
        ptx::tmem_ld32(lane_base + rs + 64 * hf, sv[0]);
        ptx::tmem_ld32(lane_base + rs + 64 * hf + 32, sv[1]);
        ptx::tmem_ld32(lane_base + rp + 64 * hf, dv0);
        ptx::tmem_wait_ld();
        ptx::tmem_ld32(lane_base + rp + 64 * hf + 32, dv1);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const int cq = 64 * hf + 32 * m;
          if (m == 1) {
            ptx::tmem_wait_ld();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(C::B_YFREE));
          }
          const uint32_t(&dv)[32] = m ? dv1 : dv0;
          uint32_t pp[16], pd[16];
          if (fast) {
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              const float2 l = *reinterpret_cast<const float2*>(sl + cq + c);
              const float2 g = *reinterpret_cast<const float2*>(sl + kTile + cq + c);
              const float2 x = ptx::ffma2(make_float2(__uint_as_float(sv[m][c]), __uint_as_float(sv[m][c + 1])),
                                          make_float2(c2, c2), make_float2(-l.x, -l.y));
              const float2 pv = make_float2(ptx::ex2(x.x), ptx::ex2(x.y));
              pp[c >> 1] = ptx::pack_bf16(pv.x, pv.y);
              const float2 dd = ptx::fmul2(pv, ptx::fadd2(make_float2(__uint_as_float(dv[c]), __uint_as_float(dv[c + 1])),
                                                          make_float2(-g.x, -g.y)));
              pd[c >> 1] = ptx::pack_bf16(dd.x, dd.y);
            }
          } else {
            const uint32_t vw = vis[m];
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              const float2 l = *reinterpret_cast<const float2*>(sl + cq + c);
              const float2 g = *reinterpret_cast<const float2*>(sl + kTile + cq + c);
              const float2 x = ptx::ffma2(make_float2(__uint_as_float(sv[m][c]), __uint_as_float(sv[m][c + 1])),
                                          make_float2(c2, c2), make_float2(-l.x, -l.y));
              const bool v0 = (vw >> c) & 1u, v1 = (vw >> (c + 1)) & 1u;
              const float p0 = v0 ? ptx::ex2(x.x) : 0.f, p1 = v1 ? ptx::ex2(x.y) : 0.f;
              pp[c >> 1] = ptx::pack_bf16(p0, p1);
              const float d0 = v0 ? p0 * (__uint_as_float(dv[c]) - g.x) : 0.f;
              const float d1 = v1 ? p1 * (__uint_as_float(dv[c + 1]) - g.y) : 0.f;
              pd[c >> 1] = ptx::pack_bf16(d0, d1);
            }
          }
          ptx::tmem_st16(lane_base + rs + 64 * hf + 16 * m, pp);
          ptx::tmem_st16(lane_base + rs + 64 * hf + 32 + 16 * m, pd);
#pragma unroll
          for (int i = 0; i < 16; ++i) dsw[16 * m + i] = pd[i];
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(C::B_PFULL + hf));  // queries 64 hf .. +63 are ready for the products
        {
          // this half's dS, from registers (its TMEM columns may already be
          // the next entry's dP by now), to its chunk of the block the dQ
          // kernel multiplies by K
          uint8_t* kr = p.ds + (size_t(it.h - p.h0) * size_t(n_entries) + size_t(e)) * kDsBlock +
                        size_t(qd * 32 + lane) * 16;  // this key's piece of every chunk
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4*>(kr + (8 * hf + u) * kDsChunk) =
                make_uint4(dsw[4 * u], dsw[4 * u + 1], dsw[4 * u + 2], dsw[4 * u + 3]);
        }
        ++nent;
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (n > 0) {
        if (!warp_wait(bar(C::B_ODONE), uint32_t(nodone) & 1u, abort_flag, err, 11)) break;
        ++nodone;
      }
      ptx::tc_fence_after();
      // the first four warps store dV, the other four dK (times the scale)
      uint32_t w[D / 2];
      tmem_row_bf16<D>(lane_base + (hf ? COL_DK : COL_DV), hf ? p.scale : 1.f, n > 0, w);
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(C::B_OFREE));
      const size_t row0 = (size_t(it.s0 + it.i0 + qd * 32) * p.H + it.h) * D;
      store_rows<D, C::STAGE_WARP>(sbase + C::OFF_STAGE + warp * C::STAGE_WARP, lane, w,
                                   (hf ? p.out0 : p.out1) + row0, size_t(p.H) * D, kn - qd * 32);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kDkdvMma) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (threadIdx.x == 0) finish_sched(p.sched);
}

template <int D>
attn_status launch_bwd(const BwdArgs& a, cudaStream_t s) {
  using C = BwdCfg<D>;
  using Q = DqCfg<D>;
  CUtensorMap mq, mk, mv, mdo;
  if (!make_map<D>(&mq, a.q, a.total_tokens, a.num_heads) || !make_map<D>(&mk, a.k, a.total_tokens, a.num_heads) ||
      !make_map<D>(&mv, a.v, a.total_tokens, a.num_heads) ||
      !make_map<D>(&mdo, a.dout, a.total_tokens, a.num_heads))
    return record_cuda_error(cudaErrorInvalidValue, "attn_bwd tensor map encoding");
  // per launch, for the current device (the settings are per device and context)
  {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Q::SMEM_ALLOC);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) return record_cuda_error(e, "attn_bwd configure");
  }
  int num_sms = 0;
  {
    const cudaError_t e = current_sm_count(&num_sms);
    if (e != cudaSuccess) return record_cuda_error(e, "attn_bwd device query");
  }
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  float* delta = reinterpret_cast<float*>(ws + a.ws.delta);
  int32_t* kpos = reinterpret_cast<int32_t*>(ws + a.ws.kpos);
  const long long rows = (long long)a.total_tokens * a.num_heads;
  bwd_delta_kernel<D><<<unsigned((rows + (2048 / D) - 1) / (2048 / D)), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dout), delta, a.total_tokens,
      a.num_heads);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return record_cuda_error(e, "attn_bwd delta launch");
  bwd_kpos_kernel<<<unsigned(a.bm.max_qt), 128, 0, s>>>(a.bm.header, a.bm.qt_idx, a.bm.koff, a.bm.kidx,
                                                          a.bm.qoff, a.bm.qidx, kpos);
  e = cudaGetLastError();
  if (e != cudaSuccess) return record_cuda_error(e, "attn_bwd entry map launch");
  BwdParams p;
  p.header = a.bm.header;
  p.qt_seq = a.bm.qt_seq;
  p.qt_idx = a.bm.qt_idx;
  p.cu = a.bm.cu;
  p.mask = a.mask;
  p.lse = a.lse;
  p.delta = delta;
  p.ds = ws + a.ws.ds;
  p.kpos = kpos;
  p.e_bound = a.ws.e_bound;
  p.H = a.num_heads;
  p.T = a.total_tokens;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  // head groups whose dS blocks fit the workspace: dK, dV over the k-major
  // lists (writing dS), then dQ over the q-major lists (reading it)
  for (int h0 = 0; h0 < a.num_heads; h0 += a.heads_per_pass) {
    p.h0 = h0;
    p.G = a.num_heads - h0 < a.heads_per_pass ? a.num_heads - h0 : a.heads_per_pass;
    const long long items = (long long)a.bm.max_qt * p.G;
    if (items <= 0 || items > INT_MAX) return ATTN_ERR_UNSUPPORTED;
    const unsigned grid = unsigned(items < num_sms ? items : num_sms);
    p.order = a.bm.korder;
    p.off = a.bm.qoff;
    p.idx = a.bm.qidx;
    p.label = a.bm.qlabel;
    p.out0 = static_cast<__nv_bfloat16*>(a.dk);
    p.out1 = static_cast<__nv_bfloat16*>(a.dv);
    p.sched = next_sched_slot();
    attn_bwd_dkdv_kernel<D><<<grid, kDkdvThreads, C::SMEM_ALLOC, s>>>(mq, mk, mv, mdo, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return record_cuda_error(e, "attn_bwd dk/dv launch");
    p.order = a.bm.order;
    p.off = a.bm.koff;
    p.idx = a.bm.kidx;
    p.label = a.bm.klabel;
    p.out0 = static_cast<__nv_bfloat16*>(a.dq);
    p.out1 = nullptr;
    p.sched = next_sched_slot();
    attn_bwd_dq_kernel<D><<<grid, kBwdThreads, Q::SMEM_ALLOC, s>>>(mk, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return record_cuda_error(e, "attn_bwd dq launch");
  }
  return ATTN_OK;
}

}  // namespace

attn_status launch_attn_bwd_bf16(const BwdArgs& a, cudaStream_t s) {
  switch (a.head_dim) {
    case 32: return launch_bwd<32>(a, s);
    case 64: return launch_bwd<64>(a, s);
    case 128: return launch_bwd<128>(a, s);
  }
  return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attnmask
