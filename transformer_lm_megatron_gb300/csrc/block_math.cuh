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

__device__ __forceinline__ float gelu_f(float x) {
  const float s = kSqrt2OverPi * (x + kGeluCubic * x * x * x);
  return 0.5f * x * (1.0f + tanhf(s));
}

// For |x| >= 30 the fp32 result is already exactly 1 (x > 0) or 0 (x < 0); the
// clamp keeps x*x finite so that (1 - th*th) * ds never becomes 0 * inf.
__device__ __forceinline__ float gelu_prime_f(float x) {
  x = fminf(fmaxf(x, -30.0f), 30.0f);
  const float s = kSqrt2OverPi * (x + kGeluCubic * x * x * x);
  const float th = tanhf(s);
  const float ds = kSqrt2OverPi * (1.0f + 3.0f * kGeluCubic * x * x);
  return 0.5f * (1.0f + th) + 0.5f * x * (1.0f - th * th) * ds;
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

}  // namespace gbmlp
