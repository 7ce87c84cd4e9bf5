// HBM-bound kernels of the MLP block that do not fuse into a GEMM epilogue:
//   * dropout backward + bias gradient:  dZ = dO * m / (1-p) (bf16),  db (+)= sum_tok dZ
//   * column sums:                        da_i (+)= sum_tok dU_i
//   (+)= adds to the accumulator, or overwrites it for the first micro-batch of a step
//   * gradient-accumulator reset, transposed copies of bf16 matrices, the dropout
//     mask itself, and a GeLU probe.
//
// Column sums are deterministic: a cluster of 1 to 8 CTAs (as many as keep the
// grid resident in one wave) owns 64 columns, each CTA a fixed share of the rows; each of a
// CTA's 64 row-lanes sums a fixed row subset, the lanes' sums are added in a fixed
// order, and CTA 0 adds the CTAs' sums in rank order through distributed shared
// memory.  Loads and stores are
// 16-byte vectors; a warp covers four 128-byte row segments per instruction.
#pragma once
#include <cstdint>

#include "block_math.cuh"
#include "ptx.cuh"

namespace gbmlp {

constexpr int kColRowLanes = 64;                 // threads along the rows of a column strip
constexpr int kColThreads = 8 * kColRowLanes;    // 8 column groups (8 bf16 = 16 B each) x row lanes
constexpr int kColsPerCta = 64;
constexpr int kColRowSplitMax = 8;               // most CTAs of a cluster splitting the rows

// Deterministic column sums over a cluster of gridDim.y CTAs (grid y = rank):
// every CTA reduces its row range to 64 partial sums in a fixed order, then CTA 0
// adds the partial vectors, in rank order, through distributed shared memory.
// part is [kColRowLanes][kColsPerCta + 1]; returns the total for thread
// threadIdx.x < kColsPerCta of CTA rank 0 (0 elsewhere).
__device__ __forceinline__ float cluster_colsum(float (*part)[kColsPerCta + 1], float* psum) {
  if (threadIdx.x < kColsPerCta) {
    float tot = 0.0f;
    for (int k = 0; k < kColRowLanes; ++k) tot += part[k][threadIdx.x];
    psum[threadIdx.x] = tot;
  }
  cluster_sync();  // every CTA's partial vector is complete
  float tot = 0.0f;
  if (cluster_ctarank() == 0 && threadIdx.x < kColsPerCta) {
    for (unsigned r = 0; r < gridDim.y; ++r) {
      const float* peer = static_cast<const float*>(__cluster_map_shared_rank(static_cast<void*>(psum), r));
      tot += peer[threadIdx.x];
    }
  }
  cluster_sync();  // the peers' shared memory stays alive until CTA 0 has read it
  return tot;
}

// dZ = dO * keep * scale (rounded to bf16); db[c] (+)= sum over rows of the rounded dZ.
// Grid (ceil(cols / 64), split), clusters of (1, split, 1), split <= kColRowSplitMax.
__global__ void __launch_bounds__(kColThreads)
    k_dropout_bwd_colsum(const uint16_t* __restrict__ dO, uint16_t* __restrict__ dZ, float* __restrict__ db,
                         int64_t rows, int cols, DropoutParams drop, int accumulate) {
  __shared__ float part[kColRowLanes][kColsPerCta + 1];
  __shared__ float psum[kColsPerCta];
  grid_dependency_wait();
  grid_launch_dependents();
  const int cg = threadIdx.x & 7;
  const int rl = threadIdx.x >> 3;
  const int col = blockIdx.x * kColsPerCta + cg * 8;
  const int64_t r_begin = rows * (int64_t)blockIdx.y / gridDim.y;
  const int64_t r_end = rows * (int64_t)(blockIdx.y + 1) / gridDim.y;
  float s[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  // One row's 8 columns: dZ out, the rounded values into the running sums.
  auto row_step = [&](int64_t r, const uint4& q) {
    float v[8] = {bf16lo(q.x), bf16hi(q.x), bf16lo(q.y), bf16hi(q.y),
                  bf16lo(q.z), bf16hi(q.z), bf16lo(q.w), bf16hi(q.w)};
    const uint32_t keep = dropout_keep8(drop, r, col);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[j] = round_bf16_f(((keep >> j) & 1u) ? v[j] * drop.scale : 0.0f);
      s[j] += v[j];
    }
    uint4 o;
    o.x = pack_bf16x2(v[0], v[1]);
    o.y = pack_bf16x2(v[2], v[3]);
    o.z = pack_bf16x2(v[4], v[5]);
    o.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4*>(dZ + r * cols + col) = o;
  };
  if (col < cols) {
    // rows in increasing order, the loads of four rows issued together
    int64_t r = r_begin + rl;
    for (; r + 3 * kColRowLanes < r_end; r += 4 * kColRowLanes) {
      uint4 q[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) q[u] = *reinterpret_cast<const uint4*>(dO + (r + u * kColRowLanes) * cols + col);
#pragma unroll
      for (int u = 0; u < 4; ++u) row_step(r + u * kColRowLanes, q[u]);
    }
    for (; r < r_end; r += kColRowLanes) row_step(r, *reinterpret_cast<const uint4*>(dO + r * cols + col));
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) part[rl][cg * 8 + j] = s[j];
  __syncthreads();
  const float tot = cluster_colsum(part, psum);
  if (blockIdx.y == 0 && threadIdx.x < kColsPerCta) {
    const int c = blockIdx.x * kColsPerCta + threadIdx.x;
    if (c < cols) db[c] = accumulate ? db[c] + tot : tot;
  }
}

// out[c] (+)= sum over rows of x[r * ld + c], c < cols.  Same grid and clusters.
__global__ void __launch_bounds__(kColThreads)
    k_colsum_bf16(const uint16_t* __restrict__ x, int64_t ld, float* __restrict__ out, int64_t rows, int cols,
                  int accumulate) {
  __shared__ float part[kColRowLanes][kColsPerCta + 1];
  __shared__ float psum[kColsPerCta];
  grid_dependency_wait();
  grid_launch_dependents();
  const int cg = threadIdx.x & 7;
  const int rl = threadIdx.x >> 3;
  const int col = blockIdx.x * kColsPerCta + cg * 8;
  const int64_t r_begin = rows * (int64_t)blockIdx.y / gridDim.y;
  const int64_t r_end = rows * (int64_t)(blockIdx.y + 1) / gridDim.y;
  float s[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  auto add_row = [&](const uint4& q) {
    s[0] += bf16lo(q.x); s[1] += bf16hi(q.x);
    s[2] += bf16lo(q.y); s[3] += bf16hi(q.y);
    s[4] += bf16lo(q.z); s[5] += bf16hi(q.z);
    s[6] += bf16lo(q.w); s[7] += bf16hi(q.w);
  };
  if (col < cols) {
    // rows in increasing order, the loads of four rows issued together
    int64_t r = r_begin + rl;
    for (; r + 3 * kColRowLanes < r_end; r += 4 * kColRowLanes) {
      uint4 q[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) q[u] = *reinterpret_cast<const uint4*>(x + (r + u * kColRowLanes) * ld + col);
#pragma unroll
      for (int u = 0; u < 4; ++u) add_row(q[u]);
    }
    for (; r < r_end; r += kColRowLanes) add_row(*reinterpret_cast<const uint4*>(x + r * ld + col));
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) part[rl][cg * 8 + j] = s[j];
  __syncthreads();
  const float tot = cluster_colsum(part, psum);
  if (blockIdx.y == 0 && threadIdx.x < kColsPerCta) {
    const int c = blockIdx.x * kColsPerCta + threadIdx.x;
    if (c < cols) out[c] = accumulate ? out[c] + tot : tot;
  }
}

// p[0 .. n) = 0 with 16-byte stores; n % 4 == 0 and p 16-byte aligned.
__global__ void k_zero_f32(float* __restrict__ p, int64_t n) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t n4 = n / 4;
  float4* p4 = reinterpret_cast<float4*>(p);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x)
    p4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Transposed copies: out[c * rows + r] = in[r * cols + c] for one or two bf16
// matrices of [rows, cols] (blockIdx.z picks the job).  A CTA moves a 64 x 64 tile
// through shared memory, with 16-byte loads along the input's rows and 16-byte
// stores along the output's.  rows % 8 == 0 and cols % 8 == 0, so that every
// vector lies wholly inside or wholly outside the matrix.
// Grid (ceil(cols / 64), ceil(rows / 64), jobs).
constexpr int kTrTile = 64;
constexpr int kTrThreads = 256;
struct TransposeJob {
  const uint16_t* in;
  uint16_t* out;
};
__global__ void __launch_bounds__(kTrThreads)
    k_transpose_bf16(TransposeJob j0, TransposeJob j1, int64_t rows, int cols) {
  __shared__ uint16_t tile[kTrTile][kTrTile + 2];   // 132-byte rows: conflict-free 2-byte stores
  grid_dependency_wait();
  grid_launch_dependents();
  const TransposeJob j = blockIdx.z == 0 ? j0 : j1;
  const int64_t r0 = (int64_t)blockIdx.y * kTrTile;
  const int c0 = blockIdx.x * kTrTile;
  const int v = threadIdx.x & 7;                    // which 8-element vector of a 64-element segment
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int rr = (threadIdx.x >> 3) + 32 * u;     // input row within the tile
    const int64_t r = r0 + rr;
    const int c = c0 + 8 * v;
    uint4 q = make_uint4(0, 0, 0, 0);
    if (r < rows && c < cols) q = *reinterpret_cast<const uint4*>(j.in + r * cols + c);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      tile[rr][8 * v + 2 * k] = (uint16_t)(w[k] & 0xffffu);
      tile[rr][8 * v + 2 * k + 1] = (uint16_t)(w[k] >> 16);
    }
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int cc = (threadIdx.x >> 3) + 32 * u;     // output row (input column) within the tile
    const int c = c0 + cc;
    const int64_t r = r0 + 8 * v;
    if (c < cols && r < rows) {
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        w[k] = (uint32_t)tile[8 * v + 2 * k][cc] | ((uint32_t)tile[8 * v + 2 * k + 1][cc] << 16);
      *reinterpret_cast<uint4*>(j.out + (int64_t)c * rows + r) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// m[r * cols + c] = keep(r, c) ? 1 : 0, eight columns per thread with the same
// routine the block's kernels use (cols % 8 == 0), else one element per thread.
__global__ void k_dropout_mask(uint8_t* __restrict__ m, int64_t rows, int cols, DropoutParams drop) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  if (cols % 8 == 0) {
    const int64_t n8 = rows * (int64_t)(cols / 8);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += stride) {
      const int64_t r = i / (cols / 8);
      const int64_t c0 = (i - r * (cols / 8)) * 8;
      const uint32_t bits = dropout_keep8(drop, r, c0);
      for (int j = 0; j < 8; ++j) m[r * cols + c0 + j] = (bits >> j) & 1u;
    }
    return;
  }
  const int64_t n = rows * (int64_t)cols;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += stride) {
    const int64_t r = i / cols;
    const int64_t c = i - r * cols;
    m[i] = dropout_keep(drop, r, c) ? 1 : 0;
  }
}

// y = GeLU(x), dy = GeLU'(x) with the epilogues' device functions.
__global__ void k_gelu_probe(const float* __restrict__ x, int64_t n, float* __restrict__ y, float* __restrict__ dy) {
  grid_dependency_wait();
  grid_launch_dependents();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    y[i] = gelu_f(x[i]);
    dy[i] = gelu_prime_f(x[i]);
  }
}

// Waits on an mbarrier that nothing arrives on, with the given limit, and records
// a timeout in the status word: exercises the bounded-wait error path.
__global__ void k_wait_timeout_probe(int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  grid_dependency_wait();
  grid_launch_dependents();
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait(&bar, 0, limit_ns)) {
      if (atomicCAS(status, 0, kStatusTimeout) == 0) status[1] = 99;
    }
  }
}

}  // namespace gbmlp
