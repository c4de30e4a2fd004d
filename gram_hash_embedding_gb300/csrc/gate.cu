// The Engram gate (sm_103a): "DeepSeek V4.1" pages, blocks/stack-hashes page, `Engram.forward`,
// the part after the `wkv` projection. For every token and residual copy i:
//   rstd  = rsqrt(mean(h_i^2) + eps) * rsqrt(mean(key_i^2) + eps)
//   dot   = sum(h_i * q_weight_i * k_weight_i * key_i) * rstd * dim^-0.5
//   gate  = sigmoid(copysign(sqrt(max(|dot|, 1e-6)), dot)), 0 where the token is masked
//   out_i = bf16(h_i + gate * value)          (value is shared by the copies)
// in fp32, as the page computes it.
//
// Design: memory-bound (per token: read hc*dim residual values and (hc+1)*dim projections, write
// hc*dim), so one CTA per token reads each input once with 16-byte loads, keeps the 3*hc partial
// sums of every copy in registers, reduces them across the block, and then writes the outputs.
// The second pass re-reads h, so the first pass loads h with an L2 evict-last policy and every
// read-once stream (keys, the value, h on its last use) with evict-first: without the hints the
// keys pushed a third of h out of L2 before its second read (1.73 GB of DRAM reads instead of
// 1.51 GB at 16,384 tokens; 1.62 ms instead of 1.43 ms at 65,536). The page's PyTorch code instead
// makes ~15 full passes over fp32 temporaries.
#include <algorithm>
#include <cstdint>

#include "engram_internal.cuh"
#include "gate_math.cuh"
#include "proj.cuh"

namespace engram {
namespace {

#ifndef ENGRAM_GATE_THREADS
#define ENGRAM_GATE_THREADS 128
#endif
#ifndef ENGRAM_GATE_MIN_BLOCKS
#define ENGRAM_GATE_MIN_BLOCKS 8
#endif

constexpr int kGateMaxCopies = ENGRAM_GATE_MAX_COPIES;  // largest hc the reduction buffers hold
constexpr int kGateThreads = ENGRAM_GATE_THREADS;       // threads per CTA (one CTA per token)
// 128 threads at 8 CTAs per SM (<= 64 registers) measured best at dim 5120, 4 copies: 1.62 ms per
// 65,536 tokens vs 2.89 ms for 256 threads at 4 CTAs per SM; more resident tokens per SM overlap one
// token's reduction barrier with the loads of the others.

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// L2 eviction policies for the loads below (createpolicy: the whole access gets the priority)
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t p;
  asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint4 ld16(const uint16_t* p) { return *reinterpret_cast<const uint4*>(p); }

// 16 bytes (8 bf16) with an L2 eviction policy
__device__ __forceinline__ uint4 ld16(const uint16_t* p, uint64_t policy) {
  uint4 v;
  asm("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p), "l"(policy));
  return v;
}

// grid = T CTAs; HC residual copies known at compile time (the partial sums live in registers)
template <int HC>
// x and out may be the same buffer: each thread reads a vector of x before it writes the same
// vector of out, and no other thread touches it, so neither pointer is marked __restrict__.
__global__ void __launch_bounds__(kGateThreads, ENGRAM_GATE_MIN_BLOCKS) gate_kernel(const uint16_t* x, const uint16_t* __restrict__ kv,
                                                   const uint16_t* __restrict__ qw, const uint16_t* __restrict__ kw,
                                                   const uint8_t* __restrict__ mask, const int dim, const float eps,
                                                   const float inv_sqrt_dim, uint16_t* out) {
  pdl_wait();
  pdl_trigger();
  const int64_t t = blockIdx.x;
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int nvec = dim >> 3;  // 8 bf16 per 16-byte vector
  const uint16_t* xt = x + t * (int64_t)HC * dim;
  const uint16_t* kvt = kv + t * (int64_t)(HC + 1) * dim;
  __shared__ float red[3 * kGateMaxCopies][kGateThreads / 32];
  __shared__ float gate_s[kGateMaxCopies];

  const uint64_t keep = l2_evict_last(), stream = l2_evict_first();
  float sh[HC], sk[HC], sd[HC];
#pragma unroll
  for (int i = 0; i < HC; ++i) sh[i] = sk[i] = sd[i] = 0.f;
  for (int v = tid; v < nvec; v += nthr) {
#pragma unroll
    for (int i = 0; i < HC; ++i) {
      float h[8], k[8], q[8], w[8];
      bf16x8_to_f32(ld16(xt + (int64_t)i * dim + 8 * v, keep), h);      // read again below
      bf16x8_to_f32(ld16(kvt + (int64_t)i * dim + 8 * v, stream), k);   // read once
      bf16x8_to_f32(ld16(qw + (int64_t)i * dim + 8 * v), q);  // shared by every token (L1)
      bf16x8_to_f32(ld16(kw + (int64_t)i * dim + 8 * v), w);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        sh[i] = fmaf(h[e], h[e], sh[i]);
        sk[i] = fmaf(k[e], k[e], sk[i]);
        sd[i] = fmaf(h[e] * (q[e] * w[e]), k[e], sd[i]);
      }
    }
  }
  // block reduction of the 3*HC sums: warp shuffles, then one value per warp in shared memory
  const int lane = tid & 31, warp = tid >> 5, nwarp = (nthr + 31) >> 5;
#pragma unroll
  for (int i = 0; i < HC; ++i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sh[i] += __shfl_xor_sync(0xffffffffu, sh[i], o);
      sk[i] += __shfl_xor_sync(0xffffffffu, sk[i], o);
      sd[i] += __shfl_xor_sync(0xffffffffu, sd[i], o);
    }
    if (lane == 0) {
      red[3 * i][warp] = sh[i];
      red[3 * i + 1][warp] = sk[i];
      red[3 * i + 2][warp] = sd[i];
    }
  }
  __syncthreads();
  if (tid < HC) {
    float a = 0.f, b = 0.f, c = 0.f;
    for (int w = 0; w < nwarp; ++w) {
      a += red[3 * tid][w];
      b += red[3 * tid + 1][w];
      c += red[3 * tid + 2][w];
    }
    gate_s[tid] = gate_of_sums(a, b, c, 1.0f / (float)dim, eps, inv_sqrt_dim, mask == nullptr || mask[t] != 0);
  }
  __syncthreads();
  // out = h + gate * value (the value row is shared by the HC copies)
  const uint16_t* vt = kvt + (int64_t)HC * dim;
  uint16_t* ot = out + t * (int64_t)HC * dim;
  for (int v = tid; v < nvec; v += nthr) {
    float val[8];
    bf16x8_to_f32(ld16(vt + 8 * v, stream), val);
#pragma unroll
    for (int i = 0; i < HC; ++i) {
      float h[8];
      bf16x8_to_f32(ld16(xt + (int64_t)i * dim + 8 * v, stream), h);  // last use
      *reinterpret_cast<uint4*>(ot + (int64_t)i * dim + 8 * v) = gate_mix8(h, val, gate_s[i]);
    }
  }
}

template <int HC>
cudaError_t launch_gate_hc(const uint16_t* x, const uint16_t* kv, const uint16_t* qw, const uint16_t* kw,
                           const uint8_t* mask, int64_t T, int dim, float eps, uint16_t* out, cudaStream_t s) {
  int threads = dim / 8;
  threads = threads < 32 ? 32 : (threads > kGateThreads ? kGateThreads : ((threads + 31) / 32) * 32);
  const float inv_sqrt_dim = (float)(1.0 / sqrt((double)dim));
  return launch_pdl(gate_kernel<HC>, dim3((unsigned)T), dim3(threads), 0, s, x, kv, qw, kw, mask, dim, eps,
                    inv_sqrt_dim, out);
}

// The gate's second half after engram_project_gate's projection: the projection epilogue left, for
// every row block of 128 tokens and every key tile u (project_tile_cols(T) columns of copy u / tpc), the
// per-token sums of h^2, key^2 and h*q_weight*k_weight*key over the tile at part[block][u][0..2][token %
// 128]. A CTA per token (and, for calls of few tokens, per chunk of nvec_chunk 8-value columns) adds
// them up per copy, forms the hc gates exactly as gate_kernel does, and writes out = bf16(h + gate *
// value) for its columns from the value rows the projection stored. The sums are staged in shared
// memory by all threads, kFinishStage tiles at a time, and then added by thread (copy i, quantity q)
// in tile order: one round trip of loads per kFinishStage tiles instead of one per few tiles.
constexpr int kFinishStage = 32;

template <int HC>
__global__ void __launch_bounds__(kGateThreads, ENGRAM_GATE_MIN_BLOCKS)
    gate_finish_kernel(const uint16_t* x, const uint16_t* __restrict__ value, const float* __restrict__ part,
                       const uint8_t* __restrict__ mask, const int dim, const int tpc, const float eps,
                       const float inv_sqrt_dim, const int nvec_chunk, uint16_t* out) {
  pdl_wait();
  pdl_trigger();
  const int64_t t = blockIdx.x;
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int nvec = dim >> 3;
  __shared__ float ps[3 * kGateMaxCopies * kFinishStage];
  __shared__ float red[3 * kGateMaxCopies];
  __shared__ float gate_s[kGateMaxCopies];
  const float* pt = part + (t >> 7) * (int64_t)(HC * tpc) * 3 * 128 + (t & 127);
  float a = 0.f;
  for (int j0 = 0; j0 < tpc; j0 += kFinishStage) {
    const int nj = min(kFinishStage, tpc - j0);
    for (int e = tid; e < 3 * HC * nj; e += nthr) {  // e = (copy i, quantity q) * nj + tile j
      const int iq = e / nj, j = e - iq * nj;
      const int i = iq / 3, q = iq - 3 * i;
      ps[e] = pt[((int64_t)(i * tpc + j0 + j) * 3 + q) * 128];
    }
    __syncthreads();
    if (tid < 3 * HC)
      for (int j = 0; j < nj; ++j) a += ps[tid * nj + j];
    __syncthreads();
  }
  if (tid < 3 * HC) red[tid] = a;
  __syncthreads();
  if (tid < HC) {
    gate_s[tid] = gate_of_sums(red[3 * tid], red[3 * tid + 1], red[3 * tid + 2], 1.0f / (float)dim, eps,
                               inv_sqrt_dim, mask == nullptr || mask[t] != 0);
  }
  __syncthreads();
  const uint64_t stream = l2_evict_first();
  const uint16_t* xt = x + t * (int64_t)HC * dim;
  const uint16_t* vt = value + t * (int64_t)dim;
  uint16_t* ot = out + t * (int64_t)HC * dim;
  const int v1 = min(nvec, (int)(blockIdx.y + 1) * nvec_chunk);
  for (int v = (int)blockIdx.y * nvec_chunk + tid; v < v1; v += nthr) {
    float val[8];
    bf16x8_to_f32(ld16(vt + 8 * v, stream), val);
#pragma unroll
    for (int i = 0; i < HC; ++i) {
      float h[8];
      bf16x8_to_f32(ld16(xt + (int64_t)i * dim + 8 * v, stream), h);
      *reinterpret_cast<uint4*>(ot + (int64_t)i * dim + 8 * v) = gate_mix8(h, val, gate_s[i]);
    }
  }
}

#ifndef ENGRAM_FINISH_TARGET_CTAS
#define ENGRAM_FINISH_TARGET_CTAS 1216  // 8 CTAs on each of the 152 SMs
#endif

template <int HC>
cudaError_t launch_gate_finish_hc(const uint16_t* x, const uint16_t* value, const float* part, const uint8_t* mask,
                                  int64_t T, int dim, float eps, uint16_t* out, cudaStream_t s) {
  int threads = dim / 8;
  threads = threads < 32 ? 32 : (threads > kGateThreads ? kGateThreads : ((threads + 31) / 32) * 32);
  const float inv_sqrt_dim = (float)(1.0 / sqrt((double)dim));
  // calls of few tokens split each token's columns over several CTAs (at least `threads` vectors each)
  const int nvec = dim / 8;
  const int64_t want = (ENGRAM_FINISH_TARGET_CTAS + T - 1) / T;
  const int chunks = (int)std::max<int64_t>(1, std::min<int64_t>(want, nvec / threads));
  const int nvec_chunk = (nvec + chunks - 1) / chunks;
  return launch_pdl(gate_finish_kernel<HC>, dim3((unsigned)T, (unsigned)chunks), dim3(threads), 0, s, x, value, part,
                    mask, dim, (int)(dim / project_tile_cols(T)), eps, inv_sqrt_dim, nvec_chunk, out);
}

}  // namespace

cudaError_t launch_gate_finish(const uint16_t* x, const uint16_t* value, const float* part, const uint8_t* mask,
                               int64_t T, int hc, int dim, float eps, uint16_t* out, cudaStream_t s) {
  switch (hc) {
    case 1: return launch_gate_finish_hc<1>(x, value, part, mask, T, dim, eps, out, s);
    case 2: return launch_gate_finish_hc<2>(x, value, part, mask, T, dim, eps, out, s);
    case 4: return launch_gate_finish_hc<4>(x, value, part, mask, T, dim, eps, out, s);
    case 8: return launch_gate_finish_hc<8>(x, value, part, mask, T, dim, eps, out, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gate(const uint16_t* x, const uint16_t* kv, const uint16_t* qw, const uint16_t* kw,
                        const uint8_t* mask, int64_t T, int hc, int dim, float eps, uint16_t* out, cudaStream_t s) {
  switch (hc) {
    case 1: return launch_gate_hc<1>(x, kv, qw, kw, mask, T, dim, eps, out, s);
    case 2: return launch_gate_hc<2>(x, kv, qw, kw, mask, T, dim, eps, out, s);
    case 4: return launch_gate_hc<4>(x, kv, qw, kw, mask, T, dim, eps, out, s);
    case 8: return launch_gate_hc<8>(x, kv, qw, kw, mask, T, dim, eps, out, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace engram
