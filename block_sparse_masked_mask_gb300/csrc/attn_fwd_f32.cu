// fp32 attention forward on the CUDA cores.
//
// Same work decomposition, block-mask lists and masking rules as the bf16
// tensor-core kernel; the arithmetic is plain fp32 FMA so that fp32 inputs
// keep fp32 score precision ("Triton from first principles" Ch. 21,
// Section 21.1 computes its scores with an fp32 dot).  One CTA per
// (q-tile, head) work item, one thread per query row; keys are staged in
// shared memory 32 at a time and the online-softmax update runs per chunk.
#include "common.cuh"

namespace attnmask {
namespace {

constexpr int kChunk = 32;

struct F32Params {
  const int32_t* header;
  const int32_t* order;
  const int32_t* qt_seq;
  const int32_t* qt_idx;
  const int32_t* koff;
  const int32_t* kidx;
  const uint8_t* klabel;
  const int32_t* cu;
  MaskArgs mask;
  const float* q;
  const float* k;
  const float* v;
  float* o;
  float* lse;
  int H, T;
  float scale_log2;
};

template <int D>
__global__ void __launch_bounds__(128) attn_fwd_f32_kernel(const F32Params p) {
  constexpr int DP = D + 1;  // padded row stride: conflict-free per-row reads
  extern __shared__ float fsm[];
  float* sQ = fsm;                       // [128][DP]
  float* sK = sQ + kTile * DP;           // [kChunk][D]
  float* sV = sK + kChunk * D;           // [kChunk][D]
  float* sS = sV + kChunk * D;           // [128][kChunk + 1] scaled scores of the chunk
  int* sCode = reinterpret_cast<int*>(sS + kTile * (kChunk + 1));  // [kChunk]

  const int n_qt = p.header[kHdrQtiles];
  const int item = blockIdx.x;
  if (item >= n_qt * p.H) return;
  const int h = item / n_qt;
  const int g = p.order[item % n_qt];
  const int b = p.qt_seq[g], qa = p.qt_idx[g];
  const int s0 = p.cu[b], L = p.cu[b + 1] - s0;
  const int i0 = qa * kTile, qn = min(kTile, L - i0);
  const int e0 = p.koff[g], n = p.koff[g + 1] - e0;
  const int r = threadIdx.x;
  const bool row_in = r < qn;
  const int il = i0 + r;

  // stage the q-tile (rows past the sequence are zero)
  for (int x = threadIdx.x; x < kTile * D; x += blockDim.x) {
    const int rr = x / D, d = x % D;
    sQ[rr * DP + d] = rr < qn ? p.q[(size_t(s0 + i0 + rr) * p.H + h) * D + d] : 0.f;
  }
  const int qcode = (row_in && kind_codes(p.mask.kind)) ? query_code(p.mask, s0 + il) : 0;
  const bool causal = kind_causal(p.mask.kind), dense = p.mask.kind == ATTN_MASK_DENSE;
  const float c2 = p.scale_log2;
  float m = -INFINITY, l = 0.f;
  float acc[D];
#pragma unroll
  for (int d = 0; d < D; ++d) acc[d] = 0.f;

  for (int e = 0; e < n; ++e) {
    const int kt = p.kidx[e0 + e];
    const bool partial = p.klabel[e0 + e] == ATTN_TILE_PARTIAL;
    const int j0 = kt * kTile, kn = min(kTile, L - j0);
    for (int c0 = 0; c0 < kn; c0 += kChunk) {
      const int cn = min(kChunk, kn - c0);
      __syncthreads();
      for (int x = threadIdx.x; x < kChunk * D; x += blockDim.x) {
        const int c = x / D, d = x % D;
        const size_t src = (size_t(s0 + j0 + c0 + c) * p.H + h) * D + d;
        sK[x] = c < cn ? p.k[src] : 0.f;
        sV[x] = c < cn ? p.v[src] : 0.f;
      }
      if (threadIdx.x < kChunk)
        sCode[threadIdx.x] = (partial && threadIdx.x < cn && kind_codes(p.mask.kind))
                                 ? key_code(p.mask, s0 + j0 + c0 + threadIdx.x) : 0;
      __syncthreads();
      float* srow = sS + r * (kChunk + 1);
      float mx = -INFINITY;
      for (int c = 0; c < kChunk; ++c) {
        float dot = 0.f;
#pragma unroll
        for (int d = 0; d < D; ++d) dot = fmaf(sQ[r * DP + d], sK[c * D + d], dot);
        bool vis = c < cn;
        if (partial && dense) {
          vis = vis && row_in && ((dense_word(p.mask, b, L, il, (j0 + c0 + c) >> 5) >> ((j0 + c0 + c) & 31)) & 1u);
        } else if (partial) {
          vis = vis && (!causal || j0 + c0 + c <= il) && code_visible(p.mask.kind, qcode, sCode[c]);
        }
        const float sc = vis ? dot * c2 : -INFINITY;
        srow[c] = sc;
        mx = fmaxf(mx, sc);
      }
      const float m_new = fmaxf(m, mx);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = exp2f(m - m_use);
      l *= alpha;
#pragma unroll
      for (int d = 0; d < D; ++d) acc[d] *= alpha;
      for (int c = 0; c < kChunk; ++c) {
        const float pc = exp2f(srow[c] - m_use);
        l += pc;
#pragma unroll
        for (int d = 0; d < D; ++d) acc[d] = fmaf(pc, sV[c * D + d], acc[d]);
      }
      m = m_new;
    }
  }
  if (row_in) {
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    float* orow = p.o + (size_t(s0 + il) * p.H + h) * D;
#pragma unroll
    for (int d = 0; d < D; ++d) orow[d] = acc[d] * inv_l;
    p.lse[size_t(h) * p.T + s0 + il] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
  }
}

template <int D>
attn_status launch(const FwdArgs& a, cudaStream_t s) {
  const size_t smem = (size_t(kTile) * (D + 1) + 2 * kChunk * D + size_t(kTile) * (kChunk + 1)) * sizeof(float) +
                      kChunk * sizeof(int);
  // per launch, for the current device (the setting is per device and context)
  cudaError_t e =
      cudaFuncSetAttribute(attn_fwd_f32_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return record_cuda_error(e, "attn_fwd configure");
  F32Params p;
  p.header = a.bm.header;
  p.order = a.bm.order;
  p.qt_seq = a.bm.qt_seq;
  p.qt_idx = a.bm.qt_idx;
  p.koff = a.bm.koff;
  p.kidx = a.bm.kidx;
  p.klabel = a.bm.klabel;
  p.cu = a.bm.cu;
  p.mask = a.mask;
  p.q = static_cast<const float*>(a.q);
  p.k = static_cast<const float*>(a.k);
  p.v = static_cast<const float*>(a.v);
  p.o = static_cast<float*>(a.o);
  p.lse = a.lse;
  p.H = a.num_heads;
  p.T = a.total_tokens;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  const long long grid = (long long)a.bm.max_qt * a.num_heads;
  if (grid <= 0 || grid > INT_MAX) return ATTN_ERR_UNSUPPORTED;
  attn_fwd_f32_kernel<D><<<unsigned(grid), 128, smem, s>>>(p);
  e = cudaGetLastError();
  return e == cudaSuccess ? ATTN_OK : record_cuda_error(e, "attn_fwd launch");
}

}  // namespace

attn_status launch_attn_fwd_f32(const FwdArgs& a, cudaStream_t s) {
  switch (a.head_dim) {
    case 32: return launch<32>(a, s);
    case 64: return launch<64>(a, s);
    case 128: return launch<128>(a, s);
  }
  return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attnmask
