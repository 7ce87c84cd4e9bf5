// Element-wise math of the MLP block, evaluated in fp32 on the device.
//
// GeLU is the tanh form 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), applied
// after the column-split first GEMM Y_i = GeLU(X A_i) of the Megatron MLP
// ("STRONGHOLD: Fast and Affordable Billion-scale Deep Learning Model Training",
// slides, item 7).  Dropout follows the row-split second GEMM (item 8); its mask is
// counter-hashed so any kernel can recompute any element's decision:
//   e = (token_offset + token) * h + column
//   r = SplitMix64 finaliser of (seed + (e + 1) * 0x9E3779B97F4A7C15)   (Steele,
//       Lea & Flood, OOPSLA 2014: output number e of a stream seeded with `seed`)
//   keep  <=>  (r >> 32) >= thr,  thr = round(p * 2^32)
// and kept values are scaled by 1/(1-p) (inverted dropout).
#pragma once
#include <cstdint>

namespace gbmlp {

constexpr float kSqrt2OverPi = 0.7978845608028654f;
constexpr float kGeluCubic = 0.044715f;

// 1 / y with the hardware reciprocal approximation (about 1 ulp); 1/inf = 0.
__device__ __forceinline__ float rcp_approx(float y) {
  float r;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(y));
  return r;
}

// The tanh form rewritten without cancellation: 0.5 x (1 + tanh(s)) = x * sigmoid(2 s)
// = x / (1 + exp(-2 s)), s = sqrt(2/pi) (x + 0.044715 x^3).  Beyond x = +-30 the
// sigmoid factor is 0 or 1 in fp32, so s is evaluated at the clamped x and the
// exponent is capped at 80 (the result there is below 1e-33 in magnitude).
__device__ __forceinline__ float gelu_f(float x) {
  const float xn = fmaxf(x, -30.0f);
  const float xc = fminf(xn, 30.0f);
  const float s = kSqrt2OverPi * fmaf(kGeluCubic * xc, xc * xc, xc);
  const float e = __expf(fminf(-2.0f * s, 80.0f));
  return xn * rcp_approx(1.0f + e);
}

// d/dx [x * sig(2 s)] = sig(2 s) + 2 x s'(x) sig(2 s) (1 - sig(2 s)), with
// sig(2 s) = r = 1 / (1 + e), 1 - sig(2 s) = e r, e = exp(-2 s), and
// s'(x) = sqrt(2/pi) (1 + 3 * 0.044715 x^2).  Same clamps as gelu_f.
__device__ __forceinline__ float gelu_prime_f(float x) {
  x = fminf(fmaxf(x, -30.0f), 30.0f);
  const float x2 = x * x;
  const float s = kSqrt2OverPi * fmaf(kGeluCubic * x, x2, x);
  const float ds = kSqrt2OverPi * fmaf(3.0f * kGeluCubic, x2, 1.0f);
  const float e = __expf(fminf(-2.0f * s, 80.0f));
  const float r = rcp_approx(1.0f + e);
  return fmaf(2.0f * x * ds, (e * r) * r, r);
}

__device__ __forceinline__ uint64_t splitmix64_at(uint64_t seed, uint64_t e) {
  uint64_t z = seed + (e + 1ull) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

struct DropoutParams {
  uint64_t seed;
  uint64_t token_offset;
  uint64_t row_width;  // h: elements per token row of the masked [tokens, h] tensor
  uint64_t thr;        // keep iff (hash >> 32) >= thr
  float scale;         // 1 / (1 - p)
};

__device__ __forceinline__ bool dropout_keep(const DropoutParams& d, int64_t token, int64_t col) {
  const uint64_t e = (d.token_offset + (uint64_t)token) * d.row_width + (uint64_t)col;
  return (splitmix64_at(d.seed, e) >> 32) >= d.thr;
}

// Keep bits (bit j for column col0 + j) of 8 consecutive elements of one row.
// The same decisions as dropout_keep, computed with less integer work: the stream
// state of element e + 1 is that of e plus the increment, and only the high 32
// bits of the final mix are formed: hi(z ^ (z >> 31)) = hi(z) ^ (hi(z) >> 31).
// thr < 2^32 because p < 1.
__device__ __forceinline__ uint32_t dropout_keep8(const DropoutParams& d, int64_t token, int64_t col0) {
  const uint64_t e0 = (d.token_offset + (uint64_t)token) * d.row_width + (uint64_t)col0;
  uint64_t x = d.seed + (e0 + 1ull) * 0x9E3779B97F4A7C15ull;
  const uint32_t thr = (uint32_t)d.thr;
  uint32_t bits = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint64_t z = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    uint32_t hi = (uint32_t)(z >> 32);
    hi ^= hi >> 31;
    bits |= (hi >= thr ? 1u : 0u) << j;
    x += 0x9E3779B97F4A7C15ull;
  }
  return bits;
}

}  // namespace gbmlp
