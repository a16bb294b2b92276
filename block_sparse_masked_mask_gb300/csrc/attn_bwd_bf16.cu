// bf16 attention backward on the sm_103a tensor cores (tcgen05 + TMA + TMEM).
//
// Gradients of O = softmax(scale Q K^T, masked) V for an upstream dO, with the
// forward's LSE: P = exp(scale S - LSE) is recomputed tile by tile, and
//   dV = P^T dO,  dP = dO V^T,  D_i = sum_d dO_id O_id,  dS = P * (dP - D),
//   dQ = scale dS K,  dK = scale dS^T Q.
// The xorl issue (Verified FA4 gaps, items 1-3) asks for this backward over
// the block-sparse masks, walking the transposed (k-major) lists for dK and
// dV, and with a deterministic dQ.  Kernels:
//   * zero: clears the per-(sequence, head) bound words;
//   * mult: the per-row multipliers m_i, and the work order's head-group
//     size for this call;
//   * prep: per (q-tile, head): D = rowsum(dO * O) and ||dO_i|| of every row
//     in fp32, the largest ||V_j|| and |K_jd| of each (sequence, head), and
//     zeroes the q-tile's rows of the dQ accumulator;
//   * main: one work item per (k-tile, head) walks its k-major list of
//     q-tiles.  Per entry it forms S^T and dP^T in TMEM, P^T and dS^T in the
//     row warps, then dV += P^T dO and dK += dS^T Q (K, V stay in shared
//     memory for the item) and dQ_i^T = K^T dS^T (dS kept in shared memory,
//     never in HBM).  Eight reducer warps add each dQ^T tile into the
//     accumulator in HBM;
//   * convert: dQ = scale * accumulator * quantum, rounded to bf16.
// Five products per tile pair (S, dP, dV, dK, dQ), no per-pair HBM traffic:
// the workspace is O(T H D).
//
// Deterministic dQ without ordering: the accumulator is exact int32 fixed
// point.  Row i's contribution from one k-tile is added in quanta q_i =
// B_i 2^-30, where B_i bounds every partial sum of the row: with P_ij <= 1,
// sum_j P_ij = 1, |dP_ij| <= ||dO_i|| ||V_j|| and |D_i| = |sum_j P_ij dP_ij|
// <= ||dO_i|| max_j ||V_j||, every partial sum of dS_ij K_jd over keys j is
// at most 2 ||dO_i|| max_j ||V_j|| max_jd |K_jd| in magnitude, and B_i is
// twice that (headroom for the rounding of P and dS to bf16).  So the
// integer sums stay below 2^29 in magnitude, integer addition is exact and
// order-independent, and every call gives the same bits whatever order the
// CTAs add in (no atomics on floats, no turn-taking).  The quantum follows
// the row's own ||dO_i|| (rows with a small upstream gradient get a fine
// one) and is at most 2^-29 of the largest value the row's sum can reach;
// the rounding adds at most q_i / 2 per contribution.  The row warps scale
// the bf16 copy of dS that feeds dQ^T by m_i = 1 / q_i (rounded to bf16;
// the convert kernel divides by the same value), so the product comes out
// of the tensor cores already in quanta and the reducers only round and
// add.  The maxima over V and K use only the sequence's own tokens, so the
// result does not depend on what else is packed with it.
//
// Items are taken by groups of heads (eight, or more when a mask has few long
// lists), longest list first inside a group, so at any time the CTAs add into
// the accumulator rows of a few heads (17 MB per head on the 32k workload).
//
// Each entry (q-tile) runs as two units of 64 queries, one per TMEM buffer,
// so that the tensor pipe works on one unit while the row warps work on the
// other.  Two threads issue the products: one the scores of each unit, the
// other (once the row warps are done with a unit) its dV, dK and dQ^T, so
// that the tensor pipe has work from one while the other waits for a buffer.
// Warp roles of the main kernel (896 threads): warps 0-15 the row warps (warp
// w owns TMEM lanes, i.e. keys, 32 (w % 4) .. +31 and, in each unit, query
// columns 16 (w / 4) .. +15, read by halves of 16 lanes so that a thread
// holds four keys at four query columns; warps 0-7 also write dV and dK),
// warp 16 the TMA
// producer, warps 17 and 18 the tcgen05 issuers (scores; dV, dK and dQ^T),
// warps 20-27 the dQ reducers (warp 20 + r + 4 c owns TMEM lanes, i.e. head
// dims, 32 r .. +31 and query columns 32 c .. +31 of each unit), warp 19
// idle.  The row warpgroups run with kRegsRow registers a thread, the others
// with kRegsLoad and kRegsRed (setmaxnreg, within the 896 x 72 of the
// launch).
// TMEM: dV [0, D), dK [128, 128 + D), then per buffer h: S^T [256 + 128 h,
// +64) (then P^T and dS^T in bf16 over it) and dP^T [320 + 128 h, +64) (then
// dQ^T over it).  Every mbarrier wait is bounded as in the forward.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "ptx.cuh"
#include "tile_pipeline.cuh"

namespace attnmask {
namespace {

constexpr int kBwdThreads = 896;
constexpr int kRowWarps = 16;
constexpr int kWarpLoad = 16, kWarpMma = 17, kWarpTail = 18, kWarpRed = 20;  // reducers: warps 20-27
// registers a thread per warpgroup: rows (four warpgroups), producer + MMA,
// reducers (two warpgroups); the launch gives 72 a thread (896 x 72 <= 65536),
// 4 x 128 x kRegsRow + 128 x kRegsLoad + 2 x 128 x kRegsRed <= 896 x 72
constexpr int kRegsLaunch = 72;
constexpr int kRegsRow = 80, kRegsLoad = 64, kRegsRed = 56;
static_assert(4 * kRegsRow + kRegsLoad + 2 * kRegsRed <= 7 * kRegsLaunch, "register budget of the launch");
static_assert(kRegsRow > kRegsLaunch && kRegsLoad < kRegsLaunch && kRegsRed < kRegsLaunch,
              "the row warps grow, the others shrink");
constexpr int kItemInts = 12;
// dS of one entry as it sits in shared memory: 128 keys x 128 queries bf16,
// in sixteen 2 KB chunks of eight queries; in chunk c, key k's eight queries
// q = 8c .. 8c+7 are the 16 bytes at k * 16 (the MN-major operand layout
// without swizzle: eight-key core matrices 128 bytes apart along K, chunks
// 2 KB apart along N).  A row-warp thread, which holds one key's dS for 32
// queries at a time, writes it as four 16-byte pieces, and the 32 lanes of a
// warp (32 consecutive keys) write 512 contiguous bytes per chunk.
constexpr int kDsBlock = kTile * kTile * 2;
constexpr int kDsChunk = 2048;
// Bound words per (sequence, head): max ||V_j||, max |K_jd| (non-negative
// floats, so their bit patterns order like ints), two words unused except
// word 2 of the first (sequence, head): the item order's head-group size.
constexpr int kBoundWords = 4;
constexpr int kHeadGroupWord = 2;
constexpr int kHeadGroupMin = 8;
constexpr float kFixScale = 1073741824.0f;  // 2^30: the quantum is B_i / 2^30

// B_i / ||dO_i|| of a (sequence, head) from its bound words.
__device__ __forceinline__ float fixed_base(const float* w) { return 4.0f * (w[0] * w[1]); }

// Row i's fixed-point multiplier m_i = 1 / quantum_i = 2^30 / B_i, rounded to
// bf16 (the row warps scale the bf16 dS that feeds dQ^T by it, so that the
// product comes out in quanta), zero for a row whose dO is zero (its dS is
// zero too) and capped at 2^100 (a smaller multiplier only coarsens the
// quantum).  The producer and the convert kernel compute it the same way.
__device__ __forceinline__ float row_multiplier(const float* bound_words, float dnorm_i) {
  const float fb = fixed_base(bound_words) * dnorm_i;
  const float m = fb > 0.f ? fminf(kFixScale / fb, 0x1p100f) : 0.f;
  return __bfloat162float(__float2bfloat16_rn(m));
}

// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) bwd_zero_kernel(int32_t* __restrict__ x, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) x[i] = 0;
}

// Per (q-tile, head): the tile's side values LSE * log2 e and D = rowsum(dO *
// O), ||dO_i|| (D / 8 lanes per row, 16 bytes of each tensor per lane), the
// tile's largest ||V_i|| and |K_id| folded into its sequence's bound words,
// and the tile's rows of the dQ accumulator zeroed.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const int32_t* __restrict__ header,
                                                       const int32_t* __restrict__ qt_seq,
                                                       const int32_t* __restrict__ qt_idx,
                                                       const int32_t* __restrict__ cu,
                                                       const __nv_bfloat16* __restrict__ o,
                                                       const __nv_bfloat16* __restrict__ dout,
                                                       const __nv_bfloat16* __restrict__ k,
                                                       const __nv_bfloat16* __restrict__ v,
                                                       const float* __restrict__ lse, float* __restrict__ side,
                                                       float* __restrict__ dnorm, float* __restrict__ bounds,
                                                       int32_t* __restrict__ dqacc, int T, int H, int G) {
  constexpr int LPR = D / 8;        // lanes per row: 16, 8 or 4
  constexpr int RPP = 256 / LPR;    // rows per pass
  __shared__ float s_max[8][2];
  const int g = blockIdx.x, h = blockIdx.y;
  if (g >= header[kHdrQtiles]) return;
  const int b = qt_seq[g];
  const int s0 = cu[b], L = cu[b + 1] - s0;
  const int a0 = qt_idx[g] * kTile;
  const int qn = min(kTile, L - a0);
  const int sub = threadIdx.x % LPR, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // the tile's side values; rows past the sequence end see no key
  float* sd = side + (size_t(h) * G + g) * kBwdSideFloats;
  for (int r = qn + int(threadIdx.x); r < kTile; r += blockDim.x) {
    sd[r] = INFINITY;
    sd[kTile + r] = 0.f;
  }
  float mv = 0.f, mk = 0.f;
  for (int r0 = 0; r0 < qn; r0 += RPP) {
    const int r = r0 + int(threadIdx.x) / LPR;
    const bool in = r < qn;
    float acc = 0.f, sdo = 0.f, sv = 0.f, ak = 0.f;
    const size_t row = (size_t(s0 + a0 + r) * H + h) * D + 8 * sub;
    if (in) {
      const uint4 ow = *reinterpret_cast<const uint4*>(o + row);
      const uint4 gw = *reinterpret_cast<const uint4*>(dout + row);
      const uint4 kw = *reinterpret_cast<const uint4*>(k + row);
      const uint4 vw = *reinterpret_cast<const uint4*>(v + row);
      const uint32_t oa[4] = {ow.x, ow.y, ow.z, ow.w}, ga[4] = {gw.x, gw.y, gw.z, gw.w};
      const uint32_t ka[4] = {kw.x, kw.y, kw.z, kw.w}, va[4] = {vw.x, vw.y, vw.z, vw.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&oa[i]));
        const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ga[i]));
        const float2 kk = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ka[i]));
        const float2 vv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&va[i]));
        acc = fmaf(x.x, y.x, fmaf(x.y, y.y, acc));
        sdo = fmaf(y.x, y.x, fmaf(y.y, y.y, sdo));
        sv = fmaf(vv.x, vv.x, fmaf(vv.y, vv.y, sv));
        ak = fmaxf(ak, fmaxf(fabsf(kk.x), fabsf(kk.y)));
      }
      int32_t* z = dqacc + row;
      *reinterpret_cast<uint4*>(z) = make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(z + 4) = make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) {
      acc += __shfl_xor_sync(0xffffffffu, acc, off);
      sdo += __shfl_xor_sync(0xffffffffu, sdo, off);
      sv += __shfl_xor_sync(0xffffffffu, sv, off);
      ak = fmaxf(ak, __shfl_xor_sync(0xffffffffu, ak, off));
    }
    if (in && sub == 0) {
      const size_t at = size_t(h) * T + s0 + a0 + r;
      const float l = __ldg(lse + at);
      sd[r] = l == -INFINITY ? INFINITY : l * 1.4426950408889634f;
      sd[kTile + r] = acc;
      // norms rounded up by a relative 2^-20, so that the bound holds for the
      // exact norms too
      dnorm[at] = sqrtf(sdo) * 1.000001f;
      mv = fmaxf(mv, sqrtf(sv) * 1.000001f);
      mk = fmaxf(mk, ak);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, off));
    mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, off));
  }
  if (lane == 0) {
    s_max[warp][0] = mv;
    s_max[warp][1] = mk;
  }
  __syncthreads();
  if (threadIdx.x < 2) {
    float m = 0.f;
    for (int w = 0; w < 8; ++w) m = fmaxf(m, s_max[w][threadIdx.x]);
    atomicMax(reinterpret_cast<int*>(bounds + (size_t(b) * H + h) * kBoundWords + threadIdx.x), __float_as_int(m));
  }
}

// Per (q-tile, head), once every tile's bound words are in: the rows'
// fixed-point multipliers m_i (zero past the sequence end) into the side
// values.
__global__ void __launch_bounds__(kTile) bwd_mult_kernel(const int32_t* __restrict__ header,
                                                         const int32_t* __restrict__ qt_seq,
                                                         const int32_t* __restrict__ qt_idx,
                                                         const int32_t* __restrict__ cu,
                                                         const int32_t* __restrict__ korder,
                                                         const int32_t* __restrict__ qoff,
                                                         const float* __restrict__ bounds,
                                                         const float* __restrict__ dnorm, float* __restrict__ side,
                                                         int32_t* __restrict__ hgroup, int T, int H, int G,
                                                         int num_sms) {
  const int g = blockIdx.x, h = blockIdx.y, c = threadIdx.x;
  if (g >= header[kHdrQtiles]) return;
  if (g == 0 && h == 0) {
    // The head-group size of the main kernel's item order (k-tiles longest
    // list first inside a group of heads): a group holds at least one long
    // item (a list of at least half the longest) per SM, or the SMs left over
    // take short items while the long ones of the next group wait for their
    // tickets and end late.  kHeadGroupMin heads at least (the K, V and
    // accumulator rows in use at once stay within a few heads), doubled
    // until the long items cover the SMs.
    const int nt = header[kHdrQtiles];
    const int lmax = qoff[korder[0] + 1] - qoff[korder[0]];
    int nlong = 0;
    for (int i0 = 0; i0 < nt; i0 += kTile) {
      const int i = i0 + c;
      const bool lg = i < nt && 2 * (qoff[korder[i] + 1] - qoff[korder[i]]) >= lmax;
      const int cnt = __syncthreads_count(lg);
      nlong += cnt;
      if (cnt < kTile) break;  // longest first: no long list further on
    }
    if (c == 0) {
      int grp = kHeadGroupMin;
      while (grp < H && grp * nlong < num_sms) grp *= 2;
      *hgroup = grp;
    }
  }
  const int b = qt_seq[g];
  const int s0 = cu[b], L = cu[b + 1] - s0;
  const int a0 = qt_idx[g] * kTile;
  const float* bw = bounds + (size_t(b) * H + h) * kBoundWords;
  side[(size_t(h) * G + g) * kBwdSideFloats + 2 * kTile + c] =
      a0 + c < L ? row_multiplier(bw, __ldg(dnorm + size_t(h) * T + s0 + a0 + c)) : 0.f;
}

// dQ = scale * accumulator / m_i in bf16, per (q-tile, head).
template <int D>
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const int32_t* __restrict__ header,
                                                             const int32_t* __restrict__ qt_seq,
                                                             const int32_t* __restrict__ qt_idx,
                                                             const int32_t* __restrict__ cu,
                                                             const float* __restrict__ bounds,
                                                             const float* __restrict__ dnorm,
                                                             const int32_t* __restrict__ acc,
                                                             __nv_bfloat16* __restrict__ dq, int T, int H,
                                                             float scale) {
  const int g = blockIdx.x, h = blockIdx.y;
  if (g >= header[kHdrQtiles]) return;
  const int b = qt_seq[g];
  const int s0 = cu[b], L = cu[b + 1] - s0;
  const int a0 = qt_idx[g] * kTile;
  const int qn = min(kTile, L - a0);
  const float* bw = bounds + (size_t(b) * H + h) * kBoundWords;
  constexpr int V4 = D / 4;  // four-int pieces per row
  for (int x = threadIdx.x; x < qn * V4; x += blockDim.x) {
    const int r = x / V4, c = x % V4;
    const float m = row_multiplier(bw, __ldg(dnorm + size_t(h) * T + s0 + a0 + r));
    const float mul = m > 0.f ? scale / m : 0.f;
    const size_t off = (size_t(s0 + a0 + r) * H + h) * D + 4 * c;
    const int4 v = __ldcg(reinterpret_cast<const int4*>(acc + off));
    uint2 w;
    w.x = ptx::pack_bf16(float(v.x) * mul, float(v.y) * mul);
    w.y = ptx::pack_bf16(float(v.z) * mul, float(v.w) * mul);
    *reinterpret_cast<uint2*>(dq + off) = w;
  }
}

// ---------------------------------------------------------------------------
template <int D>
struct BwdCfg : TileLayout<D> {
  using TileLayout<D>::TILE;
  using TileLayout<D>::CHUNK;
  using TileLayout<D>::CE;
  using TileLayout<D>::NCH;
  using TileLayout<D>::ROWB;
  static constexpr int NSLOT = 4;  // ring of streamed tiles: Q and dO of two entries
  static constexpr int OFF_K = 0, OFF_V = TILE, OFF_RING = 2 * TILE;
  static constexpr int OFF_DS = OFF_RING + NSLOT * TILE;  // dS of the entry; the dK/dV output stage
  // barriers with two instances are per 64-query half (TMEM buffer) h
  static constexpr int B_FIX = 0, B_FIXFREE = 1, B_KTAIL = 2, B_FULL = 3, B_EMPTY = B_FULL + NSLOT,
                       B_QTAIL = B_EMPTY + NSLOT, B_SFULL = B_QTAIL + 1, B_PFULL = B_SFULL + 2,
                       B_AFREE = B_PFULL + 2, B_DQFULL = B_AFREE + 2, B_DQFREE = B_DQFULL + 2,
                       B_ODONE = B_DQFREE + 2, B_OFREE = B_ODONE + 1, B_IFULL = B_OFREE + 1,
                       B_IEMPTY = B_IFULL + 2, B_DRAIN = B_IEMPTY + 2, B_DRAIN2 = B_DRAIN + 1,
                       B_STAGE = B_DRAIN2 + 1, NBAR = B_STAGE + 1;
  static constexpr int OFF_BAR = OFF_DS + kDsBlock;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int OFF_RINGI = OFF_MISC + 16;  // two decoded work items
  static constexpr int SMEM_USED = OFF_RINGI + 2 * kItemInts * 4;
  static constexpr int SMEM_MAX = 232448;
  // up to 1 KB of slack to align the base to 1024 bytes, within the limit; at
  // least 116 KB so that one CTA holds an SM (and its 512 TMEM columns) alone
  static constexpr int SMEM_ALLOC = SMEM_USED + 1024 > SMEM_MAX ? SMEM_MAX
                                    : (SMEM_USED + 1024 > 116 * 1024 ? SMEM_USED + 1024 : 116 * 1024);
  static constexpr int STAGE_WARP = 2048;  // per row warp: output rows in rounds (in the dS buffer)
  static constexpr uint32_t TMEM_COLS = 512;
  // dV and dK accumulators, then per half h: S^T (64 columns, then P^T and
  // dS^T in bf16 over it) and dP^T (64 columns, then dQ^T over it)
  static constexpr uint32_t COL_DV = 0, COL_DK = 128, COL_BUF = 256;
  static constexpr uint32_t col_s(int h) { return COL_BUF + 128u * uint32_t(h); }
  static constexpr uint32_t col_p(int h) { return COL_BUF + 128u * uint32_t(h) + 64u; }
  // S^T = K Q_h^T and dP^T = V dO_h^T: M = 128 keys, N = 64 queries, K-major
  static constexpr uint32_t IDESC_S64 = ptx::idesc_bf16_f32(128, 64, false, false);
  // dQ_h^T = K^T dS_h^T: M = 128 head-dim rows (for D < 128 the rows past D
  // read other shared memory and land in TMEM lanes nobody reads), N = 64
  // queries, K = 128 keys, both operands MN-major
  static constexpr uint32_t IDESC_DQT64 = ptx::idesc_bf16_f32(128, 64, true, true);
  // byte offset of a streamed tile's rows 64 .. 127 (the second half)
  static constexpr uint32_t HALF_ROWS = 64u * ROWB;
  static_assert(SMEM_USED <= SMEM_MAX, "shared memory budget");
  static_assert(8 * STAGE_WARP <= kDsBlock, "output stage");
  static_assert(OFF_K % 1024 == 0 && OFF_V % 1024 == 0 && OFF_RING % 1024 == 0 && TILE % 1024 == 0,
                "swizzled tiles need 1024-byte alignment");
};

struct BwdParams {
  int32_t* header;
  int sched;                // this launch's work-counter slot
  const int32_t* korder;    // k-tiles by descending list length
  const int32_t* qt_seq;
  const int32_t* qt_idx;
  const int32_t* qoff;      // k-major lists
  const int32_t* qidx;
  const uint8_t* qlabel;
  const int32_t* cu;
  MaskArgs mask;
  const float* side;        // [H][G][kBwdSideFloats]: LSE * log2 e, D, m_i of each q-tile's rows
  const int32_t* hgroup;    // heads per group of the item order (bwd_mult_kernel writes it)
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int32_t* dqacc;           // [T, H, D] fixed point
  int H, T, G;
  float scale;
  float scale_log2;
};

// One work item: one k-tile of one sequence and one head, and its list.
struct BwdItem {
  int h, s0, L, i0, e0, e1, b, gbase;  // i0: first key of the tile (local); gbase: tile 0 of the sequence
};

// Items go by groups of `group` heads (set per call by bwd_mult_kernel, at
// least kHeadGroupMin): inside a group, k-tiles longest list first, each
// k-tile for every head of the group in turn.  A group keeps the accumulator
// rows and Q / dO tiles that the CTAs touch at once to a few heads (L2
// locality), and the longest lists of the last group still start well
// before the end (a purely head-major order would start the last head's
// longest lists last and leave a tail of one list's duration).
__device__ __forceinline__ BwdItem bwd_decode(const BwdParams& p, int item, int n_t, int group) {
  BwdItem it;
  const int grp = item / (n_t * group), r = item - grp * (n_t * group);
  const int hg = min(group, p.H - grp * group);  // heads in this group
  it.h = grp * group + r % hg;
  const int g = p.korder[r / hg];
  const int b = p.qt_seq[g];
  it.s0 = p.cu[b];
  it.L = p.cu[b + 1] - it.s0;
  const int m = p.qt_idx[g];
  it.i0 = m * kTile;
  it.e0 = p.qoff[g];
  it.e1 = p.qoff[g + 1];
  it.b = b;
  it.gbase = g - m;
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
  d[8] = it.gbase;
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
  it.gbase = d[8];
  return true;
}

// The producer takes a ticket and publishes the item in ring slot k & 1.
__device__ __forceinline__ int bwd_publish(const BwdParams& p, int k, int lane, int n_items, int n_t, int group,
                                           BwdItem& it,
                                           volatile int* ring, uint32_t iempty0, uint32_t ifull0,
                                           volatile uint32_t* abort_flag, int32_t* err) {
  int ticket = 0;
  if (lane == 0) ticket = take_ticket(p.sched);
  ticket = __shfl_sync(0xffffffffu, ticket, 0);
  const bool valid = ticket < n_items;
  if (valid) it = bwd_decode(p, ticket, n_t, group);
  const int slot_i = k & 1;
  if (k >= 2 && !warp_wait(iempty0 + 8u * slot_i, uint32_t((k >> 1) - 1) & 1u, abort_flag, err, 15)) return -1;
  if (lane == 0) {
    bwd_store(ring + kItemInts * slot_i, it, valid);
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

// The issuing thread's loops are unrolled with compile-time descriptor
// offsets and accumulate flags: the tensor pipe finishes a 128 x 64 x 16
// product in ~48 cycles, so a few instructions more per issue would leave it
// idle.
//
// Half h of a product over the 128 rows of a streamed tile (dV += P^T dO or
// dK += dS^T Q over rows 64h .. 64h+63, four k-steps of 16; b_desc already
// points at row 64h).  The A operand (P^T or dS^T, bf16) sits over buffer h's
// S^T columns: the row warps write each 16-query group g over its own 16
// score columns, P^T in the first 8, dS^T in the next 8 (a_tmem is the
// buffer's first column for P^T, that + 8 for dS^T), so k-step k4 is at
// column 16 k4.
template <int D>
__device__ __forceinline__ void issue_pv_half(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, bool acc) {
  using C = BwdCfg<D>;
  ptx::mma_ts(d_tmem, a_tmem, b_desc, C::IDESC_PV, acc ? 1u : 0u);
#pragma unroll
  for (int k4 = 1; k4 < 4; ++k4)
    ptx::mma_ts_c<true>(d_tmem, a_tmem + uint32_t(k4) * 16u, b_desc + v_step<D>(k4), C::IDESC_PV);
}

// Scores-like product D = A B^T over K = D, N = 64 (both operands K-major).
template <int D>
__device__ __forceinline__ void issue_scores64(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc) {
  using C = BwdCfg<D>;
  ptx::mma_ss_c<false>(d_tmem, a_desc, b_desc, C::IDESC_S64);
#pragma unroll
  for (int kk = 1; kk < D / 16; ++kk)
    ptx::mma_ss_c<true>(d_tmem, a_desc + kmajor_step<D>(kk), b_desc + kmajor_step<D>(kk), C::IDESC_S64);
}

// dQ_h^T = K^T dS_h^T over the k-tile's 128 keys (eight k-steps of 16 keys).
template <int D>
__device__ __forceinline__ void issue_dqt64(uint32_t d_tmem, uint64_t kt_desc, uint64_t ds_desc) {
  using C = BwdCfg<D>;
  ptx::mma_ss_c<false>(d_tmem, kt_desc, ds_desc, C::IDESC_DQT64);
#pragma unroll
  for (int kk = 1; kk < kTile / 16; ++kk)
    ptx::mma_ss_c<true>(d_tmem, kt_desc + v_step<D>(kk), ds_desc + uint64_t((kk * 256) >> 4), C::IDESC_DQT64);
}

// The products of one unit after its P^T and dS^T are in TMEM: dV and dK
// (starting the accumulators when the unit opens its item), then dQ_h^T into
// buffer h's dP^T columns.  Returns false when the CTA is aborting.
template <int D>
__device__ __forceinline__ bool bwd_tail(uint32_t tmem, uint32_t bars, int h, int ent, int qs, int ds, bool first,
                                         int nitem, uint64_t rv0, uint64_t ktdesc, uint64_t dsdesc0,
                                         volatile uint32_t* abort_flag, int32_t* err) {
  using C = BwdCfg<D>;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  if (!wait_bar(bar(C::B_PFULL + h), uint32_t(ent) & 1u, abort_flag, err, 5)) return false;
  // an item's first products overwrite dV and dK: the previous item's
  // epilogue has read them out (it precedes this unit's P^T in every row
  // warp, so this wait never holds)
  if (first && nitem > 0 && !wait_bar(bar(C::B_OFREE), uint32_t(nitem - 1) & 1u, abort_flag, err, 14)) return false;
  ptx::tc_fence_after();
  const uint32_t ts = tmem + C::col_s(h);
  const uint64_t hrow = uint64_t(h) * (C::HALF_ROWS >> 4);  // rows 64h .. of a slot
  issue_pv_half<D>(tmem + C::COL_DV, ts, rv0 + uint64_t(ds) * (C::TILE >> 4) + hrow, !first);
  issue_pv_half<D>(tmem + C::COL_DK, ts + 8u, rv0 + uint64_t(qs) * (C::TILE >> 4) + hrow, !first);
  ptx::mma_commit(bar(C::B_AFREE + h));
  if (h == 1) {  // the entry's last products that read Q and dO
    ptx::mma_commit(bar(C::B_EMPTY + qs));
    ptx::mma_commit(bar(C::B_EMPTY + ds));
  }
  // dQ_h^T over this k-tile into dP^T's columns (every row warp has read them
  // before it signalled the unit)
  issue_dqt64<D>(tmem + C::col_p(h), ktdesc, dsdesc0 + uint64_t(h) * uint64_t((kDsBlock / 2) >> 4));
  ptx::mma_commit(bar(C::B_DQFULL + h));
  return true;
}

// ---------------------------------------------------------------------------
// dK, dV and the dQ contributions: one item per (k-tile, head); per listed
// q-tile i, in two units of 64 queries (h = 0, 1; TMEM buffer h):
//   S^T = K Q_ih^T, dP^T = V dO_ih^T (TMEM, TMEM lane = key),
//   P^T = 2^(S^T c2 - LSE_i log2 e), dS^T = P^T (dP^T - D_i),
//   dV += P^T dO_ih, dK += dS^T Q_ih, dQ_ih^T (+)= K^T dS^T (over this k-tile).
// The tensor pipe runs one unit ahead of the row warps: while they turn unit
// u's scores into P^T and dS^T, it runs unit u-1's dV, dK and dQ^T products
// and unit u+1's scores, each in the other buffer.
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_t = p.header[kHdrQtiles];
  const int n_items = n_t * p.H;
  int32_t* err = p.header + kHdrError;
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);
  const uint32_t sK = base + C::OFF_K, sV = base + C::OFF_V, sRing = base + C::OFF_RING, sDS = base + C::OFF_DS;
  const uint32_t bars = base + C::OFF_BAR;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  uint32_t* misc = reinterpret_cast<uint32_t*>(sbase + C::OFF_MISC);
  volatile uint32_t* abort_flag = misc + 1;
  volatile int* item_ring = reinterpret_cast<volatile int*>(sbase + C::OFF_RINGI);
  // the aligned layout must fit the allocation (it always does when the
  // dynamic shared memory starts 1024-byte aligned); otherwise fail closed
  if (base - raw + uint32_t(C::SMEM_USED) > uint32_t(C::SMEM_ALLOC)) {
    if (threadIdx.x == 0) {
      atomicOr(err, kErrTimeout | (31 << 9));
      finish_sched(p.sched);
    }
    return;
  }

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(C::B_FIX), 1);
    ptx::mbar_init(bar(C::B_FIXFREE), 2);  // tails issuer's commit + scores issuer's arrival
    ptx::mbar_init(bar(C::B_KTAIL), 1);
    for (int s = 0; s < C::NSLOT; ++s) {
      ptx::mbar_init(bar(C::B_FULL + s), 1);
      ptx::mbar_init(bar(C::B_EMPTY + s), 1);
    }
    ptx::mbar_init(bar(C::B_QTAIL), 1);
    for (int h = 0; h < 2; ++h) {
      ptx::mbar_init(bar(C::B_SFULL + h), 1);
      ptx::mbar_init(bar(C::B_PFULL + h), kRowWarps);
      ptx::mbar_init(bar(C::B_AFREE + h), 1);
      ptx::mbar_init(bar(C::B_DQFULL + h), 1);
      ptx::mbar_init(bar(C::B_DQFREE + h), 8);
    }
    ptx::mbar_init(bar(C::B_ODONE), 1);
    ptx::mbar_init(bar(C::B_OFREE), 8);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bar(C::B_IFULL + i), 1);
      ptx::mbar_init(bar(C::B_IEMPTY + i), kRowWarps + 2 + 8);  // row warps, two MMA threads, reducer warps
    }
    ptx::mbar_init(bar(C::B_DRAIN), 1);
    ptx::mbar_init(bar(C::B_DRAIN2), 1);
    ptx::mbar_init(bar(C::B_STAGE), 8);
    *abort_flag = (*reinterpret_cast<volatile int32_t*>(err) & kErrTimeout) ? 1u : 0u;
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
  } else if (warp >= kRowWarps) {
    if (warp < kWarpRed) ptx::regs_dec<kRegsLoad>();
    else ptx::regs_dec<kRegsRed>();
    if (warp == kWarpLoad) {
      // ---------------------------------------------------------- producer
      int nload = 0, ntail = 0, nfix = 0, nktail = 0;
      bool tail_pending = false, ktail_pending = false, ok = true;
      BwdItem it_next;
      const int group = *p.hgroup;  // written by bwd_mult_kernel before this launch
      int st_next = bwd_publish(p, 0, lane, n_items, n_t, group, it_next, item_ring, bar(C::B_IEMPTY),
                                bar(C::B_IFULL), abort_flag, err);
      for (int k = 0; ok && st_next == 1; ++k) {
        const BwdItem it = it_next;
        st_next = bwd_publish(p, k + 1, lane, n_items, n_t, group, it_next, item_ring, bar(C::B_IEMPTY),
                              bar(C::B_IFULL), abort_flag, err);
        if (st_next < 0) break;
        // K and V of this k-tile, once the previous item's products no longer
        // read them.  K and V rows past the sequence end are zeroed: their P
        // and dS are zero, but an inf there would make dQ^T = K^T dS^T or dP
        // (hence 0 * dP) NaN.
        if (nfix > 0 && !warp_wait(bar(C::B_FIXFREE), uint32_t(nfix - 1) & 1u, abort_flag, err, 13)) break;
        const int kn = min(kTile, it.L - it.i0);
        if (kn == kTile) {
          if (lane == 0) {
            ptx::mbar_arrive_expect_tx(bar(C::B_FIX), 2 * C::TILE);
            for (int c = 0; c < C::NCH; ++c) {
              ptx::tma_load_3d(sK + c * C::CHUNK, &tmK, bar(C::B_FIX), c * C::CE, it.h, it.s0 + it.i0);
              ptx::tma_load_3d(sV + c * C::CHUNK, &tmV, bar(C::B_FIX), c * C::CE, it.h, it.s0 + it.i0);
            }
          }
        } else {
          if (lane == 0) {
            ptx::mbar_arrive_expect_tx(bar(C::B_KTAIL), 2 * C::TILE);
            for (int c = 0; c < C::NCH; ++c) {
              ptx::tma_load_3d(sK + c * C::CHUNK, &tmK, bar(C::B_KTAIL), c * C::CE, it.h, it.s0 + it.i0);
              ptx::tma_load_3d(sV + c * C::CHUNK, &tmV, bar(C::B_KTAIL), c * C::CE, it.h, it.s0 + it.i0);
            }
          }
          ktail_pending = true;
          if (!warp_wait(bar(C::B_KTAIL), uint32_t(nktail) & 1u, abort_flag, err, 12)) break;
          ktail_pending = false;
          ++nktail;
          for (int rr = kn + lane; rr < kTile; rr += 32) {
#pragma unroll
            for (int c = 0; c < C::NCH; ++c) {
              uint4* krow = reinterpret_cast<uint4*>(sbase + C::OFF_K + c * C::CHUNK + rr * C::ROWB);
              uint4* vrow = reinterpret_cast<uint4*>(sbase + C::OFF_V + c * C::CHUNK + rr * C::ROWB);
#pragma unroll
              for (int x = 0; x < C::ROWB / 16; ++x) {
                krow[x] = make_uint4(0u, 0u, 0u, 0u);
                vrow[x] = make_uint4(0u, 0u, 0u, 0u);
              }
            }
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(bar(C::B_FIX));
        }
        ++nfix;
        // Q(i) and dO(i) of every listed q-tile into two free slots; the list
        // entry comes from global memory one entry ahead of its use, so a free
        // slot is refilled at once
        int nx = it.e0 < it.e1 ? __ldg(p.qidx + it.e0) : 0;
        for (int e = it.e0; e < it.e1; ++e) {
          const int ca0 = nx * kTile, can = min(kTile, it.L - ca0);
          if (e + 1 < it.e1) nx = __ldg(p.qidx + e + 1);
          const int qs = nload % C::NSLOT, ds = (nload + 1) % C::NSLOT;
          if (nload >= C::NSLOT &&
              (!warp_wait(bar(C::B_EMPTY + qs), uint32_t(nload / C::NSLOT - 1) & 1u, abort_flag, err, 1) ||
               !warp_wait(bar(C::B_EMPTY + ds), uint32_t((nload + 1) / C::NSLOT - 1) & 1u, abort_flag, err, 1))) {
            ok = false;
            break;
          }
          if (!load_pair<D>(&tmQ, &tmDO, it.h, it.s0 + ca0, can, sRing, sbase + C::OFF_RING, qs, ds,
                            bar(C::B_FULL), bar(C::B_QTAIL), ntail, tail_pending, lane, abort_flag, err)) {
            ok = false;
            break;
          }
          nload += 2;
        }
      }
      if (lane == 0) {
        for (int s = 0; s < C::NSLOT; ++s) {
          if (nload <= s) continue;
          const int last = s + C::NSLOT * ((nload - 1 - s) / C::NSLOT);
          drain_bar(bar(C::B_FULL + s), uint32_t(last / C::NSLOT) & 1u, err);
        }
        if (tail_pending) drain_bar(bar(C::B_QTAIL), uint32_t(ntail) & 1u, err);
        if (ktail_pending) drain_bar(bar(C::B_KTAIL), uint32_t(nktail) & 1u, err);
        if (nfix > 0) drain_bar(bar(C::B_FIX), uint32_t(nfix - 1) & 1u, err);
      }
      __syncwarp();
    } else if (warp == kWarpMma) {
      // ---------------------------------------------------------- scores issuer
      // Per unit u = (entry, half h): S^T and dP^T into buffer h.  The tails
      // (dV, dK, dQ^T) come from a second issuing thread, so that the tensor
      // pipe has work from one while the other waits for a buffer.
      if (lane == 0) {
        int nload = 0, nent = 0;
        bool ok = true;
        const uint64_t kdesc = kmajor_base<D>(sK), vdesc = kmajor_base<D>(sV);
        const uint64_t rk0 = kmajor_base<D>(sRing);
        for (int k = 0; ok; ++k) {
          if (!wait_bar(bar(C::B_IFULL + (k & 1)), uint32_t(k >> 1) & 1u, abort_flag, err, 16)) break;
          BwdItem it;
          const bool valid = bwd_load(item_ring + kItemInts * (k & 1), it);
          ptx::mbar_arrive(bar(C::B_IEMPTY + (k & 1)));
          if (!valid) break;
          if (!wait_bar(bar(C::B_FIX), uint32_t(k) & 1u, abort_flag, err, 3)) { ok = false; break; }
          const int n = it.e1 - it.e0;
          for (int j = 0; j < n && ok; ++j) {
            const int qs = nload % C::NSLOT, ds = (nload + 1) % C::NSLOT;
            for (int h = 0; h < 2; ++h) {
              const uint64_t hrow = uint64_t(h) * (C::HALF_ROWS >> 4);
              // S^T into buffer h once the previous entry's dV and dK products
              // of this half have read the P^T and dS^T written there
              if (nent > 0 && !wait_bar(bar(C::B_AFREE + h), uint32_t(nent - 1) & 1u, abort_flag, err, 7)) {
                ok = false;
                break;
              }
              if (h == 0 && !wait_bar(bar(C::B_FULL + qs), uint32_t(nload / C::NSLOT) & 1u, abort_flag, err, 4)) {
                ok = false;
                break;
              }
              ptx::tc_fence_after();
              issue_scores64<D>(tmem + C::col_s(h), kdesc, rk0 + uint64_t(qs) * (C::TILE >> 4) + hrow);
              // dP^T into buffer h once the reducers have read the dQ^T there
              if (nent > 0 && !wait_bar(bar(C::B_DQFREE + h), uint32_t(nent - 1) & 1u, abort_flag, err, 10)) {
                ok = false;
                break;
              }
              if (h == 0 &&
                  !wait_bar(bar(C::B_FULL + ds), uint32_t((nload + 1) / C::NSLOT) & 1u, abort_flag, err, 4)) {
                ok = false;
                break;
              }
              ptx::tc_fence_after();
              issue_scores64<D>(tmem + C::col_p(h), vdesc, rk0 + uint64_t(ds) * (C::TILE >> 4) + hrow);
              ptx::mma_commit(bar(C::B_SFULL + h));
            }
            nload += 2;
            ++nent;
          }
          // done with this item's K and V (its products' completion is the
          // tails issuer's half of the barrier): the next item's copy may only
          // start after this thread has seen the present one, or a phase of
          // the copy barrier could pass unseen
          if (ok) ptx::mbar_arrive(bar(C::B_FIXFREE));
        }
        ptx::mma_commit(bar(C::B_DRAIN));
        drain_bar(bar(C::B_DRAIN), 0, err);
      }
      __syncwarp();
    } else if (warp == kWarpTail) {
      // ---------------------------------------------------------- tails issuer
      // Per unit, once the row warps have written its P^T and dS^T: dV, dK and
      // dQ^T.  Its commits also free K and V (after the item's last unit) and
      // close dV and dK for the epilogue; both cover the scores issuer's
      // products too, which finished before the row warps signalled.
      if (lane == 0) {
        int nload = 0, nent = 0;
        bool ok = true;
        const uint64_t rv0 = v_base<D>(sRing);
        // dQ^T operands: K^T (the K tile read MN-major, like V in P.V) and dS^T
        // (MN-major without swizzle: 128 bytes between eight-key core matrices
        // along K, 2 KB between eight-query chunks along N; half h starts at
        // chunk 8h)
        const uint64_t ktdesc = v_base<D>(sK);
        const uint64_t dsdesc0 = ptx::smem_desc(sDS, 128u, kDsChunk, ptx::kSwizzleNone);
        for (int k = 0; ok; ++k) {
          if (!wait_bar(bar(C::B_IFULL + (k & 1)), uint32_t(k >> 1) & 1u, abort_flag, err, 16)) break;
          BwdItem it;
          const bool valid = bwd_load(item_ring + kItemInts * (k & 1), it);
          ptx::mbar_arrive(bar(C::B_IEMPTY + (k & 1)));
          if (!valid) break;
          const int n = it.e1 - it.e0;
          for (int j = 0; j < n && ok; ++j) {
            const int qs = nload % C::NSLOT, ds = (nload + 1) % C::NSLOT;
            for (int h = 0; h < 2 && ok; ++h)
              ok = bwd_tail<D>(tmem, bars, h, nent, qs, ds, j == 0 && h == 0, k, rv0, ktdesc, dsdesc0, abort_flag,
                               err);
            nload += 2;
            ++nent;
          }
          if (!ok) break;
          // K and V are free and (with n > 0) dV and dK final once the item's
          // products have finished; that includes the last dQ^T, so the dS
          // buffer is free for the output stage too
          ptx::mma_commit(bar(C::B_FIXFREE));
          if (n > 0) ptx::mma_commit(bar(C::B_ODONE));
        }
        ptx::mma_commit(bar(C::B_DRAIN2));
        drain_bar(bar(C::B_DRAIN2), 0, err);
      }
      __syncwarp();
    } else if (warp >= kWarpRed) {
      // ---------------------------------------------------------- dQ reducers
      // Warps 20-27: warp 20 + rq + 4 ch owns TMEM lanes 32 rq .. +31 of dQ^T,
      // i.e. head dims d = 32 rq + lane, and query columns 32 ch .. +31 of each
      // unit (64 queries of buffer h): its 32 columns into registers, the
      // buffer released at once, then for each of its query rows q,
      // dQacc[q, h, d] += round(dQ^T[d, q]): the product already comes out in
      // the row's quanta (its dS was scaled by m_q), so this is an exact
      // integer add at L2, each warp instruction covering 128 contiguous bytes.
      const int rq = (warp - kWarpRed) & 3, ch = (warp - kWarpRed) >> 2;
      const bool active = 32 * rq < D;
      const uint32_t lane_off = uint32_t(rq * 32) << 16;
      int nent = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        if (!warp_wait(bar(C::B_IFULL + (k & 1)), uint32_t(k >> 1) & 1u, abort_flag, err, 16)) break;
        BwdItem it;
        const bool valid = bwd_load(item_ring + kItemInts * (k & 1), it);
        warp_arrive(bar(C::B_IEMPTY + (k & 1)), lane);
        if (!valid) break;
        const size_t rstride = size_t(p.H) * D;
        int nx = it.e0 < it.e1 ? __ldg(p.qidx + it.e0) : 0;
        for (int e = it.e0; e < it.e1 && ok; ++e) {
          const int a0 = nx * kTile, qn = min(kTile, it.L - a0);
          if (e + 1 < it.e1) nx = __ldg(p.qidx + e + 1);  // one entry ahead
          for (int h = 0; h < 2; ++h) {
            if (!warp_wait(bar(C::B_DQFULL + h), uint32_t(nent) & 1u, abort_flag, err, 11)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            uint32_t v[32];
            if (active) {
              ptx::tmem_ld32(tmem + C::col_p(h) + lane_off + 32 * ch, v);
              ptx::tmem_wait_ld();
            }
            ptx::tc_fence_before();
            warp_arrive(bar(C::B_DQFREE + h), lane);
            const int q0 = 64 * h + 32 * ch;  // first query row of this warp's columns
            if (active && q0 < qn) {
              int32_t* row = p.dqacc + (size_t(it.s0 + a0 + q0) * p.H + it.h) * D + 32 * rq + lane;
              if (q0 + 32 <= qn) {
#pragma unroll
                for (int q = 0; q < 32; ++q, row += rstride)
                  ptx::red_add_s32(row, __float2int_rn(__uint_as_float(v[q])));
              } else {
                // rows past the sequence end hold zeros and are skipped by the
                // instruction's predicate
#pragma unroll
                for (int q = 0; q < 32; ++q, row += rstride)
                  ptx::red_add_s32_if(row, __float2int_rn(__uint_as_float(v[q])), q0 + q < qn);
              }
            }
          }
          ++nent;
        }
      }
    }
  } else {
    ptx::regs_inc<kRegsRow>();
    // ---------------------------------------------------------- P^T, dS^T (key rows)
    // Warp w owns TMEM lanes (keys) 32 (w % 4) .. +31 and, in every unit, the
    // unit's query columns 16 (w / 4) .. +15; the first eight warps also write
    // the item's dV (w / 4 = 0) or dK (w / 4 = 1) rows.
    const int qd = warp & 3, cg = warp >> 2;  // lane quarter, 16-column group
    const int r = qd * 32 + lane;             // the key whose mask word this lane works out
    const int kg = lane >> 2, qi = lane & 3;  // the P and dS arithmetic: keys kg + 8k, columns 2 qi (+8)
    const int kind = p.mask.kind;
    const uint32_t lane_base = tmem + (uint32_t(qd * 32) << 16);
    const float c2 = p.scale_log2;
    uint8_t* dsbuf = sbase + C::OFF_DS;
    const bool epi = cg < 2;
    int nent = 0, nodone = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      if (!warp_wait(bar(C::B_IFULL + (k & 1)), uint32_t(k >> 1) & 1u, abort_flag, err, 16)) break;
      BwdItem it;
      const bool valid = bwd_load(item_ring + kItemInts * (k & 1), it);
      warp_arrive(bar(C::B_IEMPTY + (k & 1)), lane);
      if (!valid) break;
      // the dS buffer doubles as the output stage of the item's epilogue: no
      // warp writes this item's dS before every epilogue warp has stored the
      // previous item's rows
      if (k > 0 && !warp_wait(bar(C::B_STAGE), uint32_t(k - 1) & 1u, abort_flag, err, 6)) break;
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
      int nx_idx = n > 0 ? __ldg(p.qidx + it.e0) : 0, nx_lab = n > 0 ? __ldg(p.qlabel + it.e0) : 0;
      // the side values of a q-tile (1.5 KB, twelve lines) go into L1 one entry
      // ahead of their loads
      const float* side_h = p.side + (size_t(it.h) * p.G + it.gbase) * kBwdSideFloats;
      if (warp == 0 && lane < kBwdSideFloats / 32 && n > 0)
        ptx::prefetch_l1(side_h + size_t(nx_idx) * kBwdSideFloats + 32 * lane);
      for (int jj = 0; jj < n && ok; ++jj) {
        const int e = it.e0 + jj;
        const int ti = nx_idx;  // the entry's q-tile within the sequence
        const int a0 = ti * kTile, an = min(kTile, it.L - a0);
        const int lab = nx_lab;
        if (jj + 1 < n) {  // the next entry's list values, one entry ahead
          nx_idx = __ldg(p.qidx + e + 1);
          nx_lab = __ldg(p.qlabel + e + 1);
          if (warp == 0 && lane < kBwdSideFloats / 32)
            ptx::prefetch_l1(side_h + size_t(nx_idx) * kBwdSideFloats + 32 * lane);
        }
        // the q-tile's side values (LSE * log2 e, D, m_i), from global memory:
        // the tensor cores have priority on shared memory, global loads do not
        // wait for them
        const float* sl = side_h + size_t(ti) * kBwdSideFloats;
        // every pair of the warp's rows and columns visible: no masking at all
        const bool fast = lab == ATTN_TILE_FULL && an == kTile && all_in;
        for (int h = 0; h < 2; ++h) {
          const int cq = 64 * h + 16 * cg;  // the warp's first query column of the entry
          const int cl = lane & 15;         // the masking's query column: lanes 16-31 repeat 0-15
          // before the wait: the dense kind's word of query row a0 + cq + cl
          // over the warp's 32 keys, or (code kinds) that query's code
          uint32_t dw = 0u;
          int qc = 0;
          if (lab == ATTN_TILE_PARTIAL && kbase < it.L) {
            const int qrow = a0 + cq + cl;
            if (kind == ATTN_MASK_DENSE) {
              if (qrow < it.L && lane < 16) dw = dense_word(p.mask, it.b, it.L, qrow, kbase >> 5);
            } else if (kind_codes(kind)) {
              qc = query_code(p.mask, it.s0 + min(qrow, a0 + an - 1));
            }
          }
          // the side values of this thread's four query columns, cq + 2 qi,
          // cq + 2 qi + 1 and the same 8 columns on (the TMEM layout below)
          const float* slc = sl + cq + 2 * qi;
          const float2 l_a = __ldg(reinterpret_cast<const float2*>(slc)),
                       l_b = __ldg(reinterpret_cast<const float2*>(slc + 8));
          const float2 g_a = __ldg(reinterpret_cast<const float2*>(slc + kTile)),
                       g_b = __ldg(reinterpret_cast<const float2*>(slc + kTile + 8));
          const float2 m_a = __ldg(reinterpret_cast<const float2*>(slc + 2 * kTile)),
                       m_b = __ldg(reinterpret_cast<const float2*>(slc + 2 * kTile + 8));
          if (!warp_wait(bar(C::B_SFULL + h), uint32_t(nent) & 1u, abort_flag, err, 8)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          // bit c of vis: query column cq + c sees this key (bits 0-15).
          // Causal part and bounds: a0 + column >= kl and column < an.
          uint32_t vis = 0xffffu;
          if (!fast) {
            vis = (lab == ATTN_TILE_PARTIAL && kind_causal(kind) ? ~prefix_bits(kl - a0 - cq) & prefix_bits(an - cq)
                                                                 : prefix_bits(an - cq)) &
                  0xffffu;
            if (lab == ATTN_TILE_PARTIAL && kind == ATTN_MASK_DENSE) {
              // transpose the 32-key x 16-query bit block: ballot j gathers bit
              // j (key lane j) of every lane's (query's) word, and lane j keeps it
              uint32_t mine = 0u;
#pragma unroll 4
              for (int j = 0; j < 32; ++j) {
                const uint32_t t = __ballot_sync(0xffffffffu, (dw >> j) & 1u);
                mine = lane == j ? t : mine;
              }
              vis &= mine;
            } else if (lab == ATTN_TILE_PARTIAL && kind_codes(kind)) {
              if (uniform_k) {
                vis &= __ballot_sync(0xffffffffu, code_visible(kind, qc, kcode_w));
              } else {
                uint32_t w = 0;
                for (int c = 0; c < 16; ++c)
                  w |= uint32_t(code_visible(kind, __shfl_sync(0xffffffffu, qc, c), kcode)) << c;
                vis &= w;
              }
            }
            // a key past the sequence end: its P and dS are exactly zero
            if (!row_in) vis = 0u;
          }
          // The warp's 32 keys x 16 query columns of S^T and dP^T, read by
          // halves of 16 TMEM lanes: this thread takes keys kg, kg + 8 (first
          // half) and kg + 16, kg + 24 (second) at the query columns 2 qi,
          // 2 qi + 1, 8 + 2 qi, 9 + 2 qi, so it needs the side values of four
          // columns only.  vk[k]: the visibility word of its key k.
          uint32_t vk[4] = {vis, vis, vis, vis};
          if (!fast) {
#pragma unroll
            for (int k = 0; k < 4; ++k) vk[k] = __shfl_sync(0xffffffffu, vis, kg + 8 * k);
          }
          const uint32_t half2 = 16u << 16;  // TMEM lane offset of the second half
          uint32_t sa[8], sb[8], da[8], db[8];
          ptx::tmem_ld16x256_x2(lane_base + C::col_s(h) + 16 * cg, sa);
          ptx::tmem_ld16x256_x2(lane_base + half2 + C::col_s(h) + 16 * cg, sb);
          ptx::tmem_ld16x256_x2(lane_base + C::col_p(h) + 16 * cg, da);
          ptx::tmem_ld16x256_x2(lane_base + half2 + C::col_p(h) + 16 * cg, db);
          ptx::tmem_wait_ld();
          // P^T and dS^T back to TMEM, packed bf16 pairs over the first 8 and
          // the next 8 of the warp's score columns: column j holds query
          // columns 2j, 2j + 1, so this thread's pairs land at columns qi and
          // 4 + qi of its keys.  The copy of dS for the dQ^T product goes to
          // shared memory scaled by each query's fixed-point multiplier m_i,
          // 4 bytes per (key, column pair) in the key's 16-byte row of the
          // eight-query chunk (the dQ^T that last read these chunks, the
          // previous entry's of this half, was issued before this unit's
          // scores, whose completion this warp waited for).
          uint32_t pa[4], pb[4], qa[4], qb[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {  // column pair (c, c + 1), c = 8 u + 2 qi
              const uint32_t* sv = k < 2 ? sa : sb;
              const uint32_t* dv = k < 2 ? da : db;
              const int ri = (k & 1) * 2 + u * 4;  // the pair's registers
              const int c = 8 * u + 2 * qi;
              const float2 l = u ? l_b : l_a, g = u ? g_b : g_a, mf = u ? m_b : m_a;
              float2 x = ptx::ffma2(make_float2(__uint_as_float(sv[ri]), __uint_as_float(sv[ri + 1])),
                                    make_float2(c2, c2), make_float2(-l.x, -l.y));
              // branch-free (vk is all ones on unmasked tiles), so that the
              // compiler interleaves the independent pairs: a hidden pair's
              // exponent is -inf, so its P is exactly zero, and so is its
              // dS = P (dP - D) (dP and D are finite)
              x = make_float2((vk[k] >> c) & 1u ? x.x : -INFINITY, (vk[k] >> (c + 1)) & 1u ? x.y : -INFINITY);
              const float2 pv = make_float2(ptx::ex2(x.x), ptx::ex2(x.y));
              const float2 dd =
                  ptx::fmul2(pv, ptx::fadd2(make_float2(__uint_as_float(dv[ri]), __uint_as_float(dv[ri + 1])),
                                            make_float2(-g.x, -g.y)));
              const int oi = (k & 1) + 2 * u;  // its place in the 16-lane store
              (k < 2 ? pa : pb)[oi] = ptx::pack_bf16(pv.x, pv.y);
              (k < 2 ? qa : qb)[oi] = ptx::pack_bf16(dd.x, dd.y);
              const float2 dm = ptx::fmul2(dd, mf);
              *reinterpret_cast<uint32_t*>(dsbuf + ((cq >> 3) + u) * kDsChunk + (32 * qd + kg + 8 * k) * 16 +
                                           4 * qi) = ptx::pack_bf16(dm.x, dm.y);
            }
          }
          ptx::tmem_st16x128_x2(lane_base + C::col_s(h) + 16 * cg, pa);
          ptx::tmem_st16x128_x2(lane_base + half2 + C::col_s(h) + 16 * cg, pb);
          ptx::tmem_st16x128_x2(lane_base + C::col_s(h) + 16 * cg + 8, qa);
          ptx::tmem_st16x128_x2(lane_base + half2 + C::col_s(h) + 16 * cg + 8, qb);
          ptx::tmem_wait_st();
          ptx::fence_proxy_async_smem();
          ptx::tc_fence_before();
          warp_arrive(bar(C::B_PFULL + h), lane);  // unit (entry, h) is ready for its products
        }
        ++nent;
      }
      if (!ok) break;
      if (!epi) continue;
      // ---------------------------------------------------------- epilogue
      if (n > 0) {
        if (!warp_wait(bar(C::B_ODONE), uint32_t(nodone) & 1u, abort_flag, err, 11)) break;
        ++nodone;
      }
      ptx::tc_fence_after();
      // warps 0-3 store dV, warps 4-7 dK (times the scale), 64 columns at a
      // time (the row warps' register budget holds half a row)
      constexpr int PART = D < 64 ? D : 64;
      const size_t row0 = (size_t(it.s0 + it.i0 + qd * 32) * p.H + it.h) * D;
#pragma unroll 1
      for (int pc = 0; pc < D; pc += PART) {
        uint32_t w[PART / 2];
        tmem_row_bf16<PART>(lane_base + (cg ? C::COL_DK : C::COL_DV) + pc, cg ? p.scale : 1.f, n > 0, w);
        store_rows<PART, C::STAGE_WARP>(dsbuf + warp * C::STAGE_WARP, lane, w, (cg ? p.dk : p.dv) + row0 + pc,
                                        size_t(p.H) * D, kn - qd * 32);
      }
      ptx::tc_fence_before();
      warp_arrive(bar(C::B_OFREE), lane);
      warp_arrive(bar(C::B_STAGE), lane);
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

template <int D>
attn_status launch_bwd(const BwdArgs& a, cudaStream_t s) {
  using C = BwdCfg<D>;
  CUtensorMap mq, mk, mv, mdo;
  if (!make_map<D>(&mq, a.q, a.total_tokens, a.num_heads) || !make_map<D>(&mk, a.k, a.total_tokens, a.num_heads) ||
      !make_map<D>(&mv, a.v, a.total_tokens, a.num_heads) ||
      !make_map<D>(&mdo, a.dout, a.total_tokens, a.num_heads))
    return record_cuda_error(cudaErrorInvalidValue, "attn_bwd tensor map encoding");
  // per launch, for the current device (the settings are per device and context)
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_ALLOC);
  if (e != cudaSuccess) return record_cuda_error(e, "attn_bwd configure");
  int num_sms = 0;
  e = current_sm_count(&num_sms);
  if (e != cudaSuccess) return record_cuda_error(e, "attn_bwd device query");
  const long long items = (long long)a.bm.max_qt * a.num_heads;
  if (items <= 0 || items > INT_MAX || a.num_heads > 65535) return ATTN_ERR_UNSUPPORTED;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  float* side = reinterpret_cast<float*>(ws + a.ws.side);
  float* dnorm = reinterpret_cast<float*>(ws + a.ws.dnorm);
  float* bounds = reinterpret_cast<float*>(ws + a.ws.bounds);
  int32_t* dqacc = reinterpret_cast<int32_t*>(ws + a.ws.dqacc);
  const int G = a.bm.max_qt;

  const int nbound = a.bm.batch * a.num_heads * kBoundWords;
  bwd_zero_kernel<<<unsigned((nbound + 255) / 256 < 1024 ? (nbound + 255) / 256 : 1024), 256, 0, s>>>(
      reinterpret_cast<int32_t*>(bounds), nbound);
  e = cudaGetLastError();
  if (e != cudaSuccess) return record_cuda_error(e, "attn_bwd zero launch");
  const dim3 tiles(unsigned(a.bm.max_qt), unsigned(a.num_heads));
  bwd_prep_kernel<D><<<tiles, 256, 0, s>>>(a.bm.header, a.bm.qt_seq, a.bm.qt_idx, a.bm.cu,
                                           static_cast<const __nv_bfloat16*>(a.o),
                                           static_cast<const __nv_bfloat16*>(a.dout),
                                           static_cast<const __nv_bfloat16*>(a.k),
                                           static_cast<const __nv_bfloat16*>(a.v), a.lse, side, dnorm, bounds, dqacc,
                                           a.total_tokens, a.num_heads, G);
  e = cudaGetLastError();
  if (e != cudaSuccess) return record_cuda_error(e, "attn_bwd prep launch");
  int32_t* hgroup = reinterpret_cast<int32_t*>(bounds) + kHeadGroupWord;
  bwd_mult_kernel<<<tiles, kTile, 0, s>>>(a.bm.header, a.bm.qt_seq, a.bm.qt_idx, a.bm.cu, a.bm.korder, a.bm.qoff,
                                          bounds, dnorm, side, hgroup, a.total_tokens, a.num_heads, G, num_sms);
  e = cudaGetLastError();
  if (e != cudaSuccess) return record_cuda_error(e, "attn_bwd multiplier launch");

  BwdParams p;
  p.header = a.bm.header;
  p.korder = a.bm.korder;
  p.qt_seq = a.bm.qt_seq;
  p.qt_idx = a.bm.qt_idx;
  p.qoff = a.bm.qoff;
  p.qidx = a.bm.qidx;
  p.qlabel = a.bm.qlabel;
  p.cu = a.bm.cu;
  p.mask = a.mask;
  p.side = side;
  p.hgroup = hgroup;
  p.G = G;
  p.dk = static_cast<__nv_bfloat16*>(a.dk);
  p.dv = static_cast<__nv_bfloat16*>(a.dv);
  p.dqacc = dqacc;
  p.H = a.num_heads;
  p.T = a.total_tokens;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.sched = next_sched_slot();
  const unsigned grid = unsigned(items < num_sms ? items : num_sms);
  attn_bwd_kernel<D><<<grid, kBwdThreads, C::SMEM_ALLOC, s>>>(mq, mk, mv, mdo, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return record_cuda_error(e, "attn_bwd launch");
  bwd_dq_convert_kernel<D><<<tiles, 256, 0, s>>>(a.bm.header, a.bm.qt_seq, a.bm.qt_idx, a.bm.cu, bounds, dnorm,
                                                 dqacc, static_cast<__nv_bfloat16*>(a.dq), a.total_tokens,
                                                 a.num_heads, a.scale);
  e = cudaGetLastError();
  if (e != cudaSuccess) return record_cuda_error(e, "attn_bwd dq convert launch");
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
