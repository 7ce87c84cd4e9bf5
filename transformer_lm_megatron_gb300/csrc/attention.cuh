// Row-wise kernels of the attention core (HBM-bound).
//
// Softmax:  P[r, :] = softmax(S[r, :]) for scores S (fp32) that already carry the
//           1/sqrt(d) scale and -inf above the causal diagonal; P is stored bf16.
// Rows of `cols` elements, cols % 8 == 0: one warp per row for cols <= 2048 (the
// row held in registers, read once), else one CTA per row (grid-stride over rows).
// The rows are causal: row r is query q = r % cols of its sequence and only keys
// c <= q carry probability.  The kernels read the first roundup8(q + 1) entries
// (the scores beyond q there are -inf) and write exact zeros for the rest of the
// row, so the masked half of S is never read.
// Softmax gradient: the row sums delta = sum_k P dP = dO . O (k_attn_delta); the
// rest, dS = P (dO V^T - delta) / sqrt(d), is the epilogue of the dO V^T GEMM.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace gbmlp {

constexpr int kSoftmaxThreads = 256;

__device__ __forceinline__ float block_reduce_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  v = (l < kSoftmaxThreads / 32) ? red[l] : -INFINITY;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Fixed-order block sum (deterministic).
__device__ __forceinline__ float block_reduce_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  v = (l < kSoftmaxThreads / 32) ? red[l] : 0.0f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(kSoftmaxThreads)
    k_softmax_rows(const float* __restrict__ S, uint16_t* __restrict__ P, int64_t rows, int cols) {
  __shared__ float red[kSoftmaxThreads / 32];
  grid_dependency_wait();
  grid_launch_dependents();
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const float* s = S + r * cols;
    uint16_t* p = P + r * cols;
    const int active = ((int)(r % cols) + 8) & ~7;  // roundup8(q + 1)
    float mx = -INFINITY;
    for (int c = threadIdx.x * 8; c < active; c += kSoftmaxThreads * 8) {
      const float4 a = reinterpret_cast<const float4*>(s + c)[0];
      const float4 b = reinterpret_cast<const float4*>(s + c)[1];
      mx = fmaxf(mx, fmaxf(fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)), fmaxf(fmaxf(b.x, b.y), fmaxf(b.z, b.w))));
    }
    mx = block_reduce_max(mx, red);
    float sum = 0.0f;
    for (int c = threadIdx.x * 8; c < active; c += kSoftmaxThreads * 8) {
      const float4 a = reinterpret_cast<const float4*>(s + c)[0];
      const float4 b = reinterpret_cast<const float4*>(s + c)[1];
      sum += __expf(a.x - mx) + __expf(a.y - mx) + __expf(a.z - mx) + __expf(a.w - mx) + __expf(b.x - mx) +
             __expf(b.y - mx) + __expf(b.z - mx) + __expf(b.w - mx);
    }
    sum = block_reduce_sum(sum, red);
    const float inv = 1.0f / sum;
    for (int c = threadIdx.x * 8; c < cols; c += kSoftmaxThreads * 8) {
      if (c >= active) {
        *reinterpret_cast<uint4*>(p + c) = make_uint4(0, 0, 0, 0);
        continue;
      }
      const float4 a = reinterpret_cast<const float4*>(s + c)[0];
      const float4 b = reinterpret_cast<const float4*>(s + c)[1];
      uint4 o;
      o.x = pack_bf16x2(__expf(a.x - mx) * inv, __expf(a.y - mx) * inv);
      o.y = pack_bf16x2(__expf(a.z - mx) * inv, __expf(a.w - mx) * inv);
      o.z = pack_bf16x2(__expf(b.x - mx) * inv, __expf(b.y - mx) * inv);
      o.w = pack_bf16x2(__expf(b.z - mx) * inv, __expf(b.w - mx) * inv);
      *reinterpret_cast<uint4*>(p + c) = o;
    }
  }
}

// Warp-per-row variants for rows of up to 256 * CHUNKS columns: each lane keeps its
// 8-column pieces of the row in registers, so the row is read from HBM once, and
// the reductions are warp shuffles in a fixed butterfly order (deterministic).
// A CTA works on kSoftmaxRowsPerCta rows at a time.
constexpr int kSoftmaxRowsPerCta = 8;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int CHUNKS>
__global__ void __launch_bounds__(kSoftmaxRowsPerCta * 32)
    k_softmax_rows_warp(const float* __restrict__ S, uint16_t* __restrict__ P, int64_t rows, int cols) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * kSoftmaxRowsPerCta;
  for (int64_t r = (int64_t)blockIdx.x * kSoftmaxRowsPerCta + (threadIdx.x >> 5); r < rows; r += stride) {
    const float* s = S + r * cols;
    uint16_t* p = P + r * cols;
    const int active = ((int)(r % cols) + 8) & ~7;  // roundup8(q + 1)
    float v[CHUNKS][8];
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < CHUNKS; ++i) {
      const int c = (i * 32 + lane) * 8;
      if (c < active) {
        const float4 a = __ldcs(reinterpret_cast<const float4*>(s + c));
        const float4 b = __ldcs(reinterpret_cast<const float4*>(s + c) + 1);
        v[i][0] = a.x; v[i][1] = a.y; v[i][2] = a.z; v[i][3] = a.w;
        v[i][4] = b.x; v[i][5] = b.y; v[i][6] = b.z; v[i][7] = b.w;
#pragma unroll
        for (int j = 0; j < 8; ++j) mx = fmaxf(mx, v[i][j]);
      }
    }
    mx = warp_max(mx);
    float sum = 0.0f;
#pragma unroll
    for (int i = 0; i < CHUNKS; ++i) {
      if ((i * 32 + lane) * 8 < active) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          v[i][j] = __expf(v[i][j] - mx);
          sum += v[i][j];
        }
      }
    }
    const float inv = 1.0f / warp_sum(sum);
#pragma unroll
    for (int i = 0; i < CHUNKS; ++i) {
      const int c = (i * 32 + lane) * 8;
      if (c >= cols) continue;
      uint4 o = make_uint4(0, 0, 0, 0);
      if (c < active) {
        o.x = pack_bf16x2(v[i][0] * inv, v[i][1] * inv);
        o.y = pack_bf16x2(v[i][2] * inv, v[i][3] * inv);
        o.z = pack_bf16x2(v[i][4] * inv, v[i][5] * inv);
        o.w = pack_bf16x2(v[i][6] * inv, v[i][7] * inv);
      }
      *reinterpret_cast<uint4*>(p + c) = o;
    }
  }
}

// delta[s, j, q] = sum_c dO[s L + q, j d + c] * O[s L + q, j d + c], the row sums
// sum_k P dP of the softmax gradient (sum_k P_qk (dO_q . V_k) = dO_q . O_q), in fp32.
// One warp per (token, head): lanes take 8-column pieces, then a fixed-order
// butterfly sum.  d % 8 == 0.
constexpr int kDeltaWarps = 8;

__global__ void __launch_bounds__(kDeltaWarps * 32)
    k_attn_delta(const uint16_t* __restrict__ dO, const uint16_t* __restrict__ O, float* __restrict__ delta,
                 int64_t tokens, int h, int nh, int L) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int d = h / nh;
  const int64_t n = tokens * nh;
  const int64_t stride = (int64_t)gridDim.x * kDeltaWarps;
  for (int64_t w = (int64_t)blockIdx.x * kDeltaWarps + (threadIdx.x >> 5); w < n; w += stride) {
    const int64_t tok = w / nh;
    const int j = (int)(w - tok * nh);
    const uint16_t* a = dO + tok * h + (int64_t)j * d;
    const uint16_t* b = O + tok * h + (int64_t)j * d;
    float acc = 0.0f;
    for (int c = lane * 8; c < d; c += 256) {
      const uint4 qa = *reinterpret_cast<const uint4*>(a + c);
      const uint4 qb = *reinterpret_cast<const uint4*>(b + c);
      acc += bf16lo(qa.x) * bf16lo(qb.x) + bf16hi(qa.x) * bf16hi(qb.x) + bf16lo(qa.y) * bf16lo(qb.y) +
             bf16hi(qa.y) * bf16hi(qb.y) + bf16lo(qa.z) * bf16lo(qb.z) + bf16hi(qa.z) * bf16hi(qb.z) +
             bf16lo(qa.w) * bf16lo(qb.w) + bf16hi(qa.w) * bf16hi(qb.w);
    }
    acc = warp_sum(acc);
    if (lane == 0) {
      const int64_t sq = tok / L, q = tok - sq * L;
      delta[(sq * nh + j) * L + q] = acc;
    }
  }
}

}  // namespace gbmlp
