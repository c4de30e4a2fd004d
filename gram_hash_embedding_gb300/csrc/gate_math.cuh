// The Engram gate's arithmetic ("DeepSeek V4.1" pages, blocks/stack-hashes page, `Engram.forward`),
// written once for every kernel that applies it (gate_kernel and gate_finish_kernel in gate.cu), so
// that they produce the same bits from the same sums. fp32, IEEE division and square roots (no
// fast-math).
#pragma once

#include <cstdint>

namespace engram {

// The gate of one residual copy from its three sums over the copy's dim values:
//   sh = sum h^2, sk = sum key^2, sd = sum h * q_weight * k_weight * key
//   rstd = rsqrt(sh / dim + eps) * rsqrt(sk / dim + eps), dot = sd * rstd * dim^-0.5
//   gate = sigmoid(copysign(sqrt(max(|dot|, 1e-6)), dot)); 0 where the token is masked (open false)
// rd = 1 / dim and inv_sqrt_dim = dim^-0.5 as fp32 values.
__device__ __forceinline__ float gate_of_sums(float sh, float sk, float sd, float rd, float eps, float inv_sqrt_dim,
                                              bool open) {
  const float rstd = (1.0f / sqrtf(sh * rd + eps)) * (1.0f / sqrtf(sk * rd + eps));
  const float dot = sd * rstd * inv_sqrt_dim;
  const float z = copysignf(sqrtf(fmaxf(fabsf(dot), 1e-6f)), dot);
  const float g = 1.0f / (1.0f + expf(-z));
  return open ? g : 0.f;
}

__device__ __forceinline__ uint32_t gate_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// 8 outputs bf16_rne(h + g * v) of one copy (v: the shared value row, already rounded to bf16)
__device__ __forceinline__ uint4 gate_mix8(const float* h, const float* v, float g) {
  uint4 o;
  o.x = gate_bf16x2(h[0] + g * v[0], h[1] + g * v[1]);
  o.y = gate_bf16x2(h[2] + g * v[2], h[3] + g * v[3]);
  o.z = gate_bf16x2(h[4] + g * v[4], h[5] + g * v[5]);
  o.w = gate_bf16x2(h[6] + g * v[6], h[7] + g * v[7]);
  return o;
}

}  // namespace engram
