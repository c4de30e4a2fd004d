// Kernels of libengram (sm_103a): the n-gram hash, the fp8 row lookup, and both fused.
//
// Method ("DeepSeek V4.1" pages):
//   blocks/stack-hashes page, n-gram hash `forward`: compress, mask, cache, lookback with
//     cumulative blocking, multiply, rolling XOR, floored mod by primes, + offsets.
//   engram-first/lookup page, `ParallelEngramEmbedding.forward`: fp8 row + fp32 scale gather,
//     one fp32 multiply, round-to-nearest-even to bf16, +0 for out-of-range rows.
//
// Design (GB300): the path is HBM-bound (random 128-B row reads, streaming bf16 writes, ~99.9%
// of its bytes); there is no dense contraction, so no tensor cores. A CTA owns a tile of
// consecutive tokens of one sequence: it stages the tile's compressed tokens plus the
// (max_ngram-1)-token halo in shared memory, computes every hash id of the tile there, and then
// all its threads stream the tile's rows. For one layer the tile's output rows are contiguous,
// so each warp store covers whole 32-byte sectors: lane q of a row's D/16-lane group converts
// codes [8q, 8q+8) and [D/2+8q, D/2+8q+8) and writes 16 bytes into each half of the output row.
#include <cstdint>

#include "engram_internal.cuh"

namespace engram {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;          // independent rows in flight per thread
constexpr int kFusedTile = 16;      // tokens per CTA, fused kernel
constexpr int kHashTile = 64;       // tokens per CTA, hash-only kernel

// ------------------------------------------------------------------------------------------------
// integer helpers

// Floored modulo of the int64 whose two's-complement bits are r, by the column's prime.
// q = umulhi(r, floor((2^64-1)/P)) is floor(r/P) or one less (the magic number is at most one
// unit of 2^64/P low), so one conditional subtraction gives r mod P for r read as unsigned.
// For a negative x = r - 2^64 the floored residue is (r mod P) - (2^64 mod P), taken mod P.
__device__ __forceinline__ int64_t floored_mod(uint64_t r, const ColParam& c) {
  const uint64_t q = __umul64hi(r, c.magic);
  uint64_t m = r - q * c.prime;
  if (m >= c.prime) m -= c.prime;
  if ((int64_t)r < 0) m = (m >= c.wrap) ? (m - c.wrap) : (m + c.prime - c.wrap);
  return (int64_t)m;
}

// ------------------------------------------------------------------------------------------------
// fp8 -> bf16 dequant helpers (inline PTX; exact widening, one RN multiply, RNE narrowing)

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

__device__ __forceinline__ uint2 ld_rows_v2(const uint8_t* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ float ld_scale(const float* p) {
  float v;
  asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ void st_out_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// One lane's share of one output row: codes [8q, 8q+8) and [D/2+8q, D/2+8q+8) of table row `row`.
struct RowPiece {
  uint2 v0, v1;
  float s0, s1;
  bool valid;
};

__device__ __forceinline__ void piece_load(RowPiece& pc, const uint8_t* W, const float* S, int64_t rows, int64_t row,
                                           int q, int D, int block, int nsc) {
  pc.valid = (row >= 0) && (row < rows);
  if (pc.valid) {
    const uint8_t* base = W + row * (int64_t)D;
    const int k0 = 8 * q, k1 = (D >> 1) + 8 * q;
    pc.v0 = ld_rows_v2(base + k0);
    pc.v1 = ld_rows_v2(base + k1);
    const float* srow = S + row * (int64_t)nsc;
    pc.s0 = ld_scale(srow + k0 / block);
    pc.s1 = ld_scale(srow + k1 / block);
  }
}

// out_row: bf16 row of D values (2*D bytes)
__device__ __forceinline__ void piece_store(const RowPiece& pc, uint16_t* out_row, int q, int D) {
  uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a;  // masked rows are +0
  if (pc.valid) {
    a = dequant8(pc.v0, pc.s0);
    b = dequant8(pc.v1, pc.s1);
  }
  st_out_v4(out_row + 8 * q, a);
  st_out_v4(out_row + (D >> 1) + 8 * q, b);
}

// ------------------------------------------------------------------------------------------------
// shared-memory plan of the hash / fused kernels

struct SmemPlan {
  int cols_off, mult_off, roll_off, rowidx_off, tok_off, bytes;
};

__host__ __device__ inline int align16(int x) { return (x + 15) & ~15; }

__host__ __device__ inline SmemPlan smem_plan(int n_layers, int max_ngram, int n_cols, int tile, bool gather) {
  SmemPlan p;
  int o = 0;
  p.cols_off = o;   o = align16(o + n_layers * n_cols * (int)sizeof(ColParam));
  p.mult_off = o;   o = align16(o + n_layers * max_ngram * 8);
  p.roll_off = o;   o = align16(o + tile * n_layers * (max_ngram - 1) * 8);
  p.rowidx_off = o; o = align16(o + (gather ? n_layers * tile * n_cols * 8 : 0));
  p.tok_off = o;    o = align16(o + (tile + max_ngram - 1) * 4);
  p.bytes = o;
  return p;
}

// ------------------------------------------------------------------------------------------------
// hash (+ gather) kernel. grid = (ceil(L / tile), B); one CTA = `tile` consecutive tokens of row b.
//
// G = head_dim / 16 lanes per output row (power of two); unused when GATHER is false.
template <bool GATHER, int G>
__global__ void __launch_bounds__(kThreads) hash_kernel(const StateView sv, const CallArgs a, const int tile) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int N = sv.max_ngram, NL = sv.n_layers, C = sv.n_cols, H = sv.n_heads;
  const int NC = NL * C;
  const SmemPlan plan = smem_plan(NL, N, C, tile, GATHER);
  ColParam* cols_s = reinterpret_cast<ColParam*>(smem + plan.cols_off);
  uint64_t* mult_s = reinterpret_cast<uint64_t*>(smem + plan.mult_off);
  uint64_t* roll_s = reinterpret_cast<uint64_t*>(smem + plan.roll_off);
  int64_t* rowidx_s = reinterpret_cast<int64_t*>(smem + plan.rowidx_off);
  int32_t* tok_s = reinterpret_cast<int32_t*>(smem + plan.tok_off);
  __shared__ unsigned int flags_s;

  const int tid = threadIdx.x;
  const int b = blockIdx.y;
  const int64_t L = a.L;
  const int64_t t0 = (int64_t)blockIdx.x * tile;
  const int ntok = (int)min((int64_t)tile, L - t0);
  const int64_t s_b = (int64_t)a.start_pos[b];
  const bool row_ok = (s_b >= 0) && (s_b <= sv.max_seq_len - L);
  const int32_t dead = sv.dead;
  int32_t* cache_row = sv.cache + (int64_t)b * sv.max_seq_len;

  if (tid == 0) flags_s = row_ok ? 0u : ENGRAM_STATUS_BAD_START;
  for (int i = tid; i < NC; i += kThreads) cols_s[i] = sv.cols[i];
  for (int i = tid; i < NL * N; i += kThreads) mult_s[i] = sv.mult[i];
  __syncthreads();

  // 1. compressed tokens of the tile and its halo: tok_s[j] holds position t0 - (N-1) + j.
  //    In-chunk tokens come from ids (token_map, mask); earlier positions come from the cache,
  //    which this launch never writes below start_pos, so reads and writes are disjoint.
  if (row_ok) {
    for (int j = tid; j < ntok + N - 1; j += kThreads) {
      const int64_t t = t0 - (N - 1) + j;
      int32_t c;
      if (t >= 0) {
        const int64_t id = a.ids[(int64_t)b * L + t];
        if (id < 0 || id >= sv.raw_vocab) {
          c = dead;
          atomicOr(&flags_s, ENGRAM_STATUS_BAD_ID);
        } else {
          c = sv.token_map[id];
        }
        if (a.mask != nullptr && a.mask[(int64_t)b * L + t] == 0) c = dead;
      } else {
        const int64_t p = s_b + t;
        c = (p >= 0) ? cache_row[p] : dead;
      }
      tok_s[j] = c;
    }
  }
  __syncthreads();

  // 2. cache write, lookback with cumulative blocking, products and rolling XOR per layer
  if (row_ok) {
    for (int t = tid; t < ntok; t += kThreads) {
      const int32_t cur = tok_s[t + N - 1];
      const int64_t pos = s_b + t0 + t;
      cache_row[pos] = cur;
      int64_t tok[ENGRAM_MAX_NGRAM];
      bool blocked = false;
#pragma unroll
      for (int s = 0; s < ENGRAM_MAX_NGRAM; ++s) {
        if (s < N) {
          const int32_t src = tok_s[t + N - 1 - s];
          blocked = blocked || (pos < s) || (src == dead);
          tok[s] = blocked ? sv.pad_id : (int64_t)src;
        }
      }
      for (int l = 0; l < NL; ++l) {
        uint64_t r = (uint64_t)tok[0] * mult_s[l * N];
#pragma unroll
        for (int i = 1; i < ENGRAM_MAX_NGRAM; ++i) {
          if (i < N) {
            r ^= (uint64_t)tok[i] * mult_s[l * N + i];
            roll_s[(t * NL + l) * (N - 1) + (i - 1)] = r;
          }
        }
      }
    }
  }
  __syncthreads();

  // 3. hash ids: floored mod by the column's prime plus its offset; (t, layer, column) order
  //    so the optional int64 write is contiguous
  for (int e = tid; e < ntok * NC; e += kThreads) {
    const int t = e / NC;
    const int j = e - t * NC;
    const int l = j / C;
    const int col = j - l * C;
    int64_t h = -1;
    if (row_ok) {
      const ColParam cp = cols_s[j];
      h = floored_mod(roll_s[(t * NL + l) * (N - 1) + col / H], cp) + cp.offset;
    }
    if (a.hashes != nullptr) a.hashes[((int64_t)b * L + t0 + t) * NC + j] = h;
    if (GATHER) rowidx_s[(l * tile + t) * C + col] = h;
  }

  if (GATHER) {
    __syncthreads();
    // 4. gather + dequant: for each layer the tile's ntok*C output rows are contiguous
    const int D = a.head_dim, blk = a.block, nsc = D / blk;
    const int rows_per_layer = ntok * C;
    const int units = NL * rows_per_layer * G;
    const int64_t out_base_row = ((int64_t)b * L + t0) * C;
    for (int base = tid; base < units; base += kThreads * kUnroll) {
      RowPiece pc[kUnroll];
      int ls[kUnroll], rems[kUnroll];
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        const int u = base + k * kThreads;
        ls[k] = -1;
        if (u < units) {
          const int v = u / G;
          const int q = u % G;
          const int l = v / rows_per_layer;
          const int rem = v - l * rows_per_layer;
          const int t = rem / C;
          const int col = rem - t * C;
          ls[k] = l;
          rems[k] = rem;
          piece_load(pc[k], a.W[l], a.S[l], a.rows[l], rowidx_s[(l * tile + t) * C + col], q, D, blk, nsc);
        }
      }
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        if (ls[k] >= 0) {
          const int u = base + k * kThreads;
          const int q = u % G;
          uint16_t* orow = a.out[ls[k]] + (out_base_row + rems[k]) * (int64_t)D;
          piece_store(pc[k], orow, q, D);
        }
      }
    }
  }

  __syncthreads();
  if (tid == 0 && flags_s != 0u) atomicOr(sv.status, flags_s);
}

// ------------------------------------------------------------------------------------------------
// standalone lookup: grid-stride over (index, lane) units

template <int G>
__global__ void __launch_bounds__(kThreads) lookup_kernel(const int64_t* __restrict__ idx, const int64_t n_idx,
                                                          const uint8_t* __restrict__ W,
                                                          const float* __restrict__ S, const int64_t rows,
                                                          const int D, const int blk, uint16_t* __restrict__ out) {
  const int nsc = D / blk;
  const int64_t units = n_idx * G;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  for (int64_t base = (int64_t)blockIdx.x * kThreads + threadIdx.x; base < units; base += stride * kUnroll) {
    RowPiece pc[kUnroll];
    int64_t rowid[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const int64_t u = base + k * stride;
      rowid[k] = -1;
      if (u < units) {
        rowid[k] = u / G;
        piece_load(pc[k], W, S, rows, __ldg(idx + rowid[k]), (int)(u % G), D, blk, nsc);
      }
    }
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      if (rowid[k] >= 0) {
        const int64_t u = base + k * stride;
        piece_store(pc[k], out + rowid[k] * (int64_t)D, (int)(u % G), D);
      }
    }
  }
}

__global__ void fill_i32_kernel(int32_t* p, int64_t n, int32_t v) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) p[i] = v;
}

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 152;
  }
  return n;
}

template <bool GATHER, int G>
cudaError_t launch_hash_g(const StateView& sv, const CallArgs& a, int tile, cudaStream_t s) {
  const SmemPlan plan = smem_plan(sv.n_layers, sv.max_ngram, sv.n_cols, tile, GATHER);
  auto kern = hash_kernel<GATHER, G>;
  if (plan.bytes > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, plan.bytes);
    if (e != cudaSuccess) return e;
  }
  dim3 grid((unsigned)((a.L + tile - 1) / tile), (unsigned)a.B);
  kern<<<grid, kThreads, plan.bytes, s>>>(sv, a, tile);
  return cudaGetLastError();
}

template <int G>
cudaError_t launch_lookup_g(const int64_t* idx, int64_t n_idx, const uint8_t* W, const float* S, int64_t rows, int D,
                            int blk, uint16_t* out, cudaStream_t s) {
  const int64_t units = n_idx * G;
  int64_t blocks = (units + (int64_t)kThreads * kUnroll - 1) / ((int64_t)kThreads * kUnroll);
  const int64_t cap = (int64_t)sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  lookup_kernel<G><<<(unsigned)blocks, kThreads, 0, s>>>(idx, n_idx, W, S, rows, D, blk, out);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fill_i32(int32_t* p, int64_t n, int32_t value, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  fill_i32_kernel<<<(unsigned)blocks, 256, 0, s>>>(p, n, value);
  return cudaGetLastError();
}

cudaError_t launch_hash(const StateView& sv, const CallArgs& a, cudaStream_t s) {
  return launch_hash_g<false, 1>(sv, a, kHashTile, s);
}

cudaError_t launch_hash_lookup(const StateView& sv, const CallArgs& a, cudaStream_t s) {
  switch (a.head_dim / 16) {
    case 1: return launch_hash_g<true, 1>(sv, a, kFusedTile, s);
    case 2: return launch_hash_g<true, 2>(sv, a, kFusedTile, s);
    case 4: return launch_hash_g<true, 4>(sv, a, kFusedTile, s);
    case 8: return launch_hash_g<true, 8>(sv, a, kFusedTile, s);
    case 16: return launch_hash_g<true, 16>(sv, a, kFusedTile, s);
    case 32: return launch_hash_g<true, 32>(sv, a, kFusedTile, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_lookup(const int64_t* idx, int64_t n_idx, const uint8_t* W, const float* S, int64_t rows,
                          int32_t head_dim, int32_t block, uint16_t* out, cudaStream_t s) {
  switch (head_dim / 16) {
    case 1: return launch_lookup_g<1>(idx, n_idx, W, S, rows, head_dim, block, out, s);
    case 2: return launch_lookup_g<2>(idx, n_idx, W, S, rows, head_dim, block, out, s);
    case 4: return launch_lookup_g<4>(idx, n_idx, W, S, rows, head_dim, block, out, s);
    case 8: return launch_lookup_g<8>(idx, n_idx, W, S, rows, head_dim, block, out, s);
    case 16: return launch_lookup_g<16>(idx, n_idx, W, S, rows, head_dim, block, out, s);
    case 32: return launch_lookup_g<32>(idx, n_idx, W, S, rows, head_dim, block, out, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace engram
