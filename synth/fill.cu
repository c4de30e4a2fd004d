// Device fill of the synthetic fp8 table and its fp32 scales.
//
// Input generator only: the same counter-based stream as synth/__init__.py
// (splitmix64 output function over base + (ctr + 1) * golden), so the host can
// regenerate any row bit for bit. It computes nothing of the Engram method.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  z ^= z >> 31;
  return z;
}

__device__ __forceinline__ uint64_t word_at(uint64_t base, uint64_t ctr) {
  return mix64(base + (ctr + 1ull) * 0x9E3779B97F4A7C15ull);
}

__device__ __forceinline__ uint32_t four_codes(uint64_t w, const uint8_t* __restrict__ lut) {
  uint32_t b0 = lut[(uint32_t)(w & 0xFFFFu)];
  uint32_t b1 = lut[(uint32_t)((w >> 16) & 0xFFFFu)];
  uint32_t b2 = lut[(uint32_t)((w >> 32) & 0xFFFFu)];
  uint32_t b3 = lut[(uint32_t)((w >> 48) & 0xFFFFu)];
  return b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
}

// one thread -> 16 bytes (4 words) per iteration
__global__ void fill_fp8_kernel(uint4* __restrict__ W, int64_t n16, uint64_t base, const uint8_t* __restrict__ lut) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16; i += stride) {
    const uint64_t g = (uint64_t)i * 4ull;
    uint4 v;
    v.x = four_codes(word_at(base, g + 0), lut);
    v.y = four_codes(word_at(base, g + 1), lut);
    v.z = four_codes(word_at(base, g + 2), lut);
    v.w = four_codes(word_at(base, g + 3), lut);
    W[i] = v;
  }
}

__global__ void fill_scales_kernel(float* __restrict__ S, int64_t n, uint64_t base) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += stride) {
    const uint64_t w = word_at(base, (uint64_t)i);
    const float t = __fmul_rn(__ull2float_rn(w >> 40), 5.9604644775390625e-08f);  // exact: < 2^24 times 2^-24
    S[i] = __fadd_rn(0.01f, __fmul_rn(0.99f, t));
  }
}

// scale bit patterns of the other storage types, from one generator word each (integer operations
// only; the host restatement is synth.scale_codes): kind 1 bf16, 2 UE8M0, 3 E4M3
__global__ void fill_scale_codes_kernel(void* __restrict__ S, int64_t n, uint64_t base, int kind) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += stride) {
    const uint64_t w = word_at(base, (uint64_t)i);
    if (kind == 1) {
      reinterpret_cast<uint16_t*>(S)[i] = (uint16_t)(((120u + (uint32_t)(w & 7u)) << 7) | (uint32_t)((w >> 8) & 0x7Fu));
    } else if (kind == 2) {
      reinterpret_cast<uint8_t*>(S)[i] = (uint8_t)(120u + (uint32_t)(w & 7u));
    } else {
      reinterpret_cast<uint8_t*>(S)[i] = (uint8_t)(((4u + (uint32_t)(w & 3u)) << 3) | (uint32_t)((w >> 8) & 7u));
    }
  }
}

int grid_for(int64_t n) {
  int64_t g = (n + 255) / 256;
  const int64_t cap = 152 * 16;
  return (int)(g < 1 ? 1 : (g > cap ? cap : g));
}

}  // namespace

extern "C" {

// W: device, nbytes bytes (multiple of 16, 16-byte aligned); lut: device uint8[65536].
int synth_fill_fp8(void* W, int64_t nbytes, uint64_t base, const void* lut, void* stream) {
  if (nbytes < 0 || (nbytes % 16) != 0 || (reinterpret_cast<uintptr_t>(W) % 16) != 0 || lut == nullptr) return -1;
  if (nbytes == 0) return 0;
  const int64_t n16 = nbytes / 16;
  fill_fp8_kernel<<<grid_for(n16), 256, 0, (cudaStream_t)stream>>>(reinterpret_cast<uint4*>(W), n16, base,
                                                                    reinterpret_cast<const uint8_t*>(lut));
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

// S: device float[n], 4-byte aligned.
int synth_fill_scales(void* S, int64_t n, uint64_t base, void* stream) {
  if (n < 0 || (reinterpret_cast<uintptr_t>(S) % 4) != 0) return -1;
  if (n == 0) return 0;
  fill_scales_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(reinterpret_cast<float*>(S), n, base);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

// S: device storage of n scales of kind 1 (bf16, 2-byte aligned), 2 (UE8M0) or 3 (E4M3).
int synth_fill_scale_codes(void* S, int64_t n, uint64_t base, int kind, void* stream) {
  if (n < 0 || kind < 1 || kind > 3 || (kind == 1 && (reinterpret_cast<uintptr_t>(S) % 2) != 0)) return -1;
  if (n == 0) return 0;
  fill_scale_codes_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(S, n, base, kind);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // extern "C"
