// fp8 E4M3 -> bf16 dequantisation shared by the lookup kernels (kernels.cu) and the lookup warps of
// the projection (proj.cu), so that every path produces the same bits: the code widened exactly to
// fp32 (through f16), one fp32 round-to-nearest multiply by the row's block scale, round-to-nearest-
// even to bf16 ("DeepSeek V4.1" pages, engram-first/lookup page, `ParallelEngramEmbedding.forward`:
// the fp8 rows times their scales, cast to bf16). No flush of subnormals anywhere.
#pragma once

#include <cstdint>

#include "../../include/engram.h"

namespace engram {

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  uint32_t r;
  const uint16_t v = (uint16_t)two_codes;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}

__device__ __forceinline__ void f16x2_to_f32(uint32_t h2, float& lo, float& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h2));
}

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// two codes (low 16 bits of w, first code in the low byte) -> two bf16 (first in the low half)
__device__ __forceinline__ uint32_t dequant2(uint32_t w, float s) {
  float a, b;
  f16x2_to_f32(e4m3x2_to_f16x2(w), a, b);
  return bf16x2_rn(__fmul_rn(a, s), __fmul_rn(b, s));
}

// 8 codes (bytes of w.x then w.y) -> 8 bf16 (16 bytes)
__device__ __forceinline__ uint4 dequant8(uint2 w, float s) {
  uint4 o;
  o.x = dequant2(w.x, s);
  o.y = dequant2(w.x >> 16, s);
  o.z = dequant2(w.y, s);
  o.w = dequant2(w.y >> 16, s);
  return o;
}

__device__ __forceinline__ uint4 ld_rows_v4(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Raw bits of scale i of a scale tensor stored as SDT (ENGRAM_SCALE_*), zero-extended. The load
// only parks the bits in a register; `widen_scale` runs later, once the whole batch of row loads is
// in flight (widening right after the load would stall the thread on every scale).
template <int SDT>
__device__ __forceinline__ uint32_t ld_scale_bits(const void* S, int64_t i) {
  uint32_t v;
  if (SDT == ENGRAM_SCALE_F32) {
    asm volatile("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(v) : "l"(static_cast<const uint32_t*>(S) + i));
  } else if (SDT == ENGRAM_SCALE_BF16) {
    uint16_t h;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(h) : "l"(static_cast<const uint16_t*>(S) + i));
    v = h;
  } else {
    asm volatile("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=r"(v) : "l"(static_cast<const uint8_t*>(S) + i));
  }
  return v;
}

// The scale's value, widened to fp32 exactly.
template <int SDT>
__device__ __forceinline__ float widen_scale(uint32_t bits) {
  if (SDT == ENGRAM_SCALE_F32) return __uint_as_float(bits);
  if (SDT == ENGRAM_SCALE_BF16) return __uint_as_float(bits << 16);  // the upper half of a binary32
  if (SDT == ENGRAM_SCALE_E8M0) {  // 2^(e-127): the exponent field of a binary32; 0 is the subnormal 2^-127
    if (bits == 0xFFu) return __uint_as_float(0x7FC00000u);
    return __uint_as_float(bits == 0u ? 0x00400000u : (bits << 23));
  }
  float lo, hi;  // E4M3, as the table codes
  f16x2_to_f32(e4m3x2_to_f16x2(bits), lo, hi);
  return lo;
}

}  // namespace engram
