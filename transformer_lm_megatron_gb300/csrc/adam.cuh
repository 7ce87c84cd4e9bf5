// Mixed-precision Adam step over the fp32 gradient accumulators (HBM-bound).
//
// Per parameter (Kingma & Ba 2015, with decoupled weight decay, Loshchilov &
// Hutter 2019):  g = grad * scale;  m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;
// w = w (1 - lr wd) - step_size * m / (sqrt(v) * inv_sqrt_bc2 + eps);  weight = bf16(w)
// with step_size = lr / (1 - b1^t) and inv_sqrt_bc2 = 1 / sqrt(1 - b2^t) from the host.
// Traffic: read grad, w, m, v (16 B), write w, m, v (12 B) and the bf16 weight
// (2 B) = 30 B per parameter; four parameters per thread step with 16-byte loads.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace gbmlp {

struct AdamParams {
  float grad_scale;
  float beta1, one_minus_beta1;
  float beta2, one_minus_beta2;
  float step_size;     // lr / (1 - beta1^t)
  float inv_sqrt_bc2;  // 1 / sqrt(1 - beta2^t)
  float eps;
  float decay;         // 1 - lr * weight_decay
};

__device__ __forceinline__ void adam_one(const AdamParams& p, float g, float& w, float& m, float& v) {
  g *= p.grad_scale;
  m = fmaf(p.beta1, m, p.one_minus_beta1 * g);
  v = fmaf(p.beta2, v, p.one_minus_beta2 * g * g);
  const float denom = fmaf(sqrtf(v), p.inv_sqrt_bc2, p.eps);
  w = fmaf(-p.step_size, m / denom, w * p.decay);
}

__global__ void __launch_bounds__(256) k_adam_step(int64_t n, const float* __restrict__ grad, float* __restrict__ w,
                                                   float* __restrict__ m, float* __restrict__ v,
                                                   uint16_t* __restrict__ w16, AdamParams p) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t n4 = n >> 2;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 g4 = reinterpret_cast<const float4*>(grad)[i];
    float4 w4 = reinterpret_cast<float4*>(w)[i];
    float4 m4 = reinterpret_cast<float4*>(m)[i];
    float4 v4 = reinterpret_cast<float4*>(v)[i];
    adam_one(p, g4.x, w4.x, m4.x, v4.x);
    adam_one(p, g4.y, w4.y, m4.y, v4.y);
    adam_one(p, g4.z, w4.z, m4.z, v4.z);
    adam_one(p, g4.w, w4.w, m4.w, v4.w);
    reinterpret_cast<float4*>(w)[i] = w4;
    reinterpret_cast<float4*>(m)[i] = m4;
    reinterpret_cast<float4*>(v)[i] = v4;
    reinterpret_cast<uint2*>(w16)[i] = make_uint2(pack_bf16x2(w4.x, w4.y), pack_bf16x2(w4.z, w4.w));
  }
  // the last n % 4 parameters
  if (blockIdx.x == 0 && threadIdx.x < (n & 3)) {
    const int64_t i = (n4 << 2) + threadIdx.x;
    float wi = w[i], mi = m[i], vi = v[i];
    adam_one(p, grad[i], wi, mi, vi);
    w[i] = wi;
    m[i] = mi;
    v[i] = vi;
    const uint32_t packed = pack_bf16x2(wi, 0.0f);
    w16[i] = (uint16_t)(packed & 0xFFFFu);
  }
}

}  // namespace gbmlp
