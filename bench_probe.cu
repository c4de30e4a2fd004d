// Measurement probes behind the fused kernel's roofline: what random row reads cost the DRAM on
// this GPU, how fast the fused kernel's byte pattern can move at all, and whether placing a row's
// fp32 scale next to its fp8 codes would change that. Timing and counting only: the regions are
// uninitialised device memory, the outputs are meaningless, and nothing here is on the product
// path. Built and run by `python bench.py --probe access|gather|layout|depth`.
//
//   access  3,145,728 random reads of 4, 16, 32, 64 and 128 bytes (one kernel per size, named
//           probe_read_<size>) into a 48 GB region; then 4-byte reads with other load flavours
//           (probe_read_flavour<.cg / .cs / relaxed>) and with the context's L2 fetch granularity
//           limit set to 32 bytes (a per-context setting: it ends with the process). Run it under ncu
//           with dram__bytes_read.sum to see the DRAM bytes each access costs.
//   gather  the fused kernel's bytes without the hash: per row a random 128-B code row and a random
//           4-B scale read, 256 B written in order; 3,145,728 rows (one full-scale launch) out of
//           768,022,850 (both full-scale tables), several launch shapes; read-only and write-only
//           splits; then the main patterns again with the L2 fetch granularity limit at 32 bytes.
//   layout  the same gather with the scale stored separately, not read, right after the codes
//           (144-B and 256-B records) or in a block after every 32 rows.
//   depth   the gather (read + write, separate scales) with 2 to 8 rows in flight per 8-lane group in
//           registers, and 4 to 16 rows landed in shared memory by cp.async, at the 32-B fetch limit.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstring>

#define CK(x)                                                                            \
  do {                                                                                   \
    cudaError_t e_ = (x);                                                                \
    if (e_ != cudaSuccess) {                                                             \
      std::printf("%s failed: %s\n", #x, cudaGetErrorString(e_));                        \
      return 1;                                                                          \
    }                                                                                    \
  } while (0)

namespace {

constexpr int64_t kRowsFull = 768022850;  // 384,006,168 + 384,016,682 rows
constexpr int64_t kN = 3145728;           // rows of one full-scale launch (65,536 tokens x 48)

// splitmix64 finaliser: the row picked by access i of index set `seed`
__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void make_idx(int64_t* idx, int64_t n, int64_t rows, uint64_t seed) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i < n) idx[i] = (int64_t)(mix64(seed * 0x100000001ull + (uint64_t)i) % (uint64_t)rows);
}

// ---------------------------------------------------------------------------------------- access
// One access of BYTES bytes at the start of a random 128-B slot: BYTES <= 16 is one lane's load,
// larger sizes are BYTES/16 adjacent lanes loading 16 B each.
template <int BYTES>
__global__ void probe_read(const unsigned char* __restrict__ region, const int64_t* __restrict__ idx, int64_t n,
                           uint32_t* __restrict__ sink) {
  constexpr int LANES = BYTES >= 16 ? BYTES / 16 : 1;
  const int64_t g = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) / LANES;
  const int lane = threadIdx.x % LANES;
  if (g >= n) return;
  const unsigned char* p = region + idx[g] * 128;
  uint32_t v;
  if (BYTES == 4) {
    v = __ldg(reinterpret_cast<const uint32_t*>(p));
  } else {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(p) + lane);
    v = w.x ^ w.y ^ w.z ^ w.w;
  }
  if (v == 0x9E3779B9u) sink[0] = v;  // keeps the load; practically never taken
}

// 4-byte reads at the start of a random 128-B slot with another load flavour:
// 0 ld.global.cg (L2 only), 1 ld.global.cs (streaming), 2 ld.relaxed.gpu.global
template <int FLAVOUR>
__global__ void probe_read_flavour(const unsigned char* __restrict__ region, const int64_t* __restrict__ idx,
                                   int64_t n, uint32_t* __restrict__ sink) {
  const int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (g >= n) return;
  const uint32_t* p = reinterpret_cast<const uint32_t*>(region + idx[g] * 128);
  uint32_t v;
  if (FLAVOUR == 0) {
    asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(p));
  } else if (FLAVOUR == 1) {
    asm volatile("ld.global.cs.u32 %0, [%1];" : "=r"(v) : "l"(p));
  } else {
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p));
  }
  if (v == 0x9E3779B9u) sink[0] = v;  // keeps the load; practically never taken
}

// ---------------------------------------------------------------------------------------- gather
// LAYOUT 0: codes at base + 128 k, scale at sbase + 4 k (the pages' separate tensors)
//        1: codes only (no scale read)
//        2: records of STRIDE bytes: codes at STRIDE k, scale at STRIDE k + 128
//        3: blocks of 32 rows: [32 x 128 B codes][32 x 4 B scales] (4,224 B)
// MODE 0: read + write; 1: read only (a practically never taken store keeps the loads); 2: write only;
//      3: read + write, the writes with an L2 evict-first policy (as the fused kernel writes its rows);
//      4: read + write in the fused kernel's layout: lane q loads codes [8q, 8q+8) and [64+8q, 64+8q+8)
//         and writes 16 bytes into each half of the 256-byte output row, so every warp store covers
//         whole 32-byte sectors
template <int U, int LAYOUT, int STRIDE, int MODE>
__global__ void __launch_bounds__(256) probe_gather(const unsigned char* __restrict__ base,
                                                    const float* __restrict__ sbase,
                                                    const int64_t* __restrict__ idx, uint4* __restrict__ out,
                                                    int64_t n_rows) {
  const int lane8 = threadIdx.x & 7;
  const int64_t groups = (int64_t)gridDim.x * (blockDim.x >> 3);
  const int64_t g0 = blockIdx.x * (int64_t)(blockDim.x >> 3) + (threadIdx.x >> 3);
  for (int64_t b0 = g0; b0 < n_rows; b0 += groups * U) {
    uint4 v[U];
    float s[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t row = b0 + (int64_t)u * groups;
      v[u] = make_uint4((uint32_t)row, 1u, 2u, 3u);
      s[u] = 1.f;
      if (MODE != 2 && row < n_rows) {
        const int64_t k = __ldg(idx + row);
        const unsigned char* c;
        const float* sp = nullptr;
        if (LAYOUT == 0) {
          c = base + k * 128;
          sp = sbase + k;
        } else if (LAYOUT == 1) {
          c = base + k * 128;
        } else if (LAYOUT == 2) {
          c = base + k * STRIDE;
          sp = reinterpret_cast<const float*>(c + 128);
        } else {
          const int64_t blk = k >> 5, j = k & 31;
          c = base + blk * 4224 + j * 128;
          sp = reinterpret_cast<const float*>(base + blk * 4224 + 4096 + j * 4);
        }
        if (MODE == 4) {
          const uint2 lo = __ldg(reinterpret_cast<const uint2*>(c) + lane8);
          const uint2 hi = __ldg(reinterpret_cast<const uint2*>(c + 64) + lane8);
          v[u] = make_uint4(lo.x, lo.y, hi.x, hi.y);
        } else {
          v[u] = __ldg(reinterpret_cast<const uint4*>(c) + lane8);
        }
        if (LAYOUT != 1) s[u] = __ldg(sp);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t row = b0 + (int64_t)u * groups;
      if (row >= n_rows) continue;
      const uint32_t sb = __float_as_uint(s[u]);
      const uint4 a = make_uint4(v[u].x ^ sb, v[u].y, v[u].z, v[u].w);
      const uint4 b = make_uint4(v[u].x, v[u].y ^ sb, v[u].z, v[u].w);
      uint4* o = out + row * 16;
      if (MODE == 1) {
        if ((a.x ^ b.y ^ a.z) == 0x12345678u) o[lane8] = a;
      } else if (MODE == 4) {
        o[lane8] = make_uint4(v[u].x ^ sb, v[u].y, v[u].x, v[u].y);
        o[8 + lane8] = make_uint4(v[u].z ^ sb, v[u].w, v[u].z, v[u].w);
      } else if (MODE == 3) {
        uint64_t pol;
        asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
        asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(o + lane8), "r"(a.x), "r"(a.y),
                     "r"(a.z), "r"(a.w), "l"(pol) : "memory");
        asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(o + 8 + lane8), "r"(b.x),
                     "r"(b.y), "r"(b.z), "r"(b.w), "l"(pol) : "memory");
      } else {
        o[lane8] = a;
        o[8 + lane8] = b;
      }
    }
  }
}

struct Gather {
  const unsigned char* base;
  const float* sbase;
  int64_t* idx[4];
  uint4* out;
  cudaEvent_t e0, e1;
};

template <int U, int LAYOUT, int STRIDE, int MODE>
int time_gather(const Gather& g, const char* what, int blocks, int64_t* const* idx) {
  const int reps = 200;
  for (int w = 0; w < 3; ++w) probe_gather<U, LAYOUT, STRIDE, MODE><<<blocks, 256>>>(g.base, g.sbase, idx[w & 3], g.out, kN);
  CK(cudaGetLastError());
  CK(cudaDeviceSynchronize());
  CK(cudaEventRecord(g.e0));
  for (int i = 0; i < reps; ++i) probe_gather<U, LAYOUT, STRIDE, MODE><<<blocks, 256>>>(g.base, g.sbase, idx[i & 3], g.out, kN);
  CK(cudaEventRecord(g.e1));
  CK(cudaEventSynchronize(g.e1));
  float ms = 0.f;
  CK(cudaEventElapsedTime(&ms, g.e0, g.e1));
  const double us = ms * 1e3 / reps;
  const char* kind = MODE == 0 ? "read+write"
                     : (MODE == 1 ? "read only"
                                  : (MODE == 2 ? "write only" : (MODE == 3 ? "rw, evict-first writes" : "rw, fused layout")));
  std::printf("%-44s %-10s grid %6d x 256, %d rows/thread-group pass: %7.1f us per launch\n", what, kind, blocks, U, us);
  return 0;
}

// The separate-scales gather (read + write) with its row loads landed in shared memory by
// cp.async instead of registers, so a thread keeps U rows in flight without holding them: lane q of a
// row's 8-lane group copies codes [16q, 16q+16) and lane 0 the row's 4-byte scale, then every lane
// waits for its own copies, the warp synchronises (the scale is another lane's copy), and the lane
// writes its two 16-byte pieces of the 256-B output row. Shared memory per CTA: U x 4,224 bytes.
template <int U>
__global__ void __launch_bounds__(256) probe_gather_async(const unsigned char* __restrict__ base,
                                                          const float* __restrict__ sbase,
                                                          const int64_t* __restrict__ idx, uint4* __restrict__ out,
                                                          int64_t n_rows) {
  extern __shared__ __align__(16) unsigned char sm[];
  uint4* codes_s = reinterpret_cast<uint4*>(sm);                   // [U][256]
  float* scales_s = reinterpret_cast<float*>(sm + U * 256 * 16);   // [U][32]
  const int lane8 = threadIdx.x & 7, grp = threadIdx.x >> 3;
  const int64_t groups = (int64_t)gridDim.x * 32;
  const int64_t g0 = blockIdx.x * 32LL + grp;
  for (int64_t b0 = g0; b0 < n_rows; b0 += groups * U) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t row = b0 + (int64_t)u * groups;
      if (row < n_rows) {
        const int64_t k = __ldg(idx + row);
        const uint32_t dst = (uint32_t)__cvta_generic_to_shared(codes_s + u * 256 + threadIdx.x);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(base + k * 128 + lane8 * 16)
                     : "memory");
        if (lane8 == 0) {
          const uint32_t sdst = (uint32_t)__cvta_generic_to_shared(scales_s + u * 32 + grp);
          asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(sdst), "l"(sbase + k) : "memory");
        }
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncwarp();
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t row = b0 + (int64_t)u * groups;
      if (row >= n_rows) continue;
      const uint4 v = codes_s[u * 256 + threadIdx.x];
      const uint32_t sb = __float_as_uint(scales_s[u * 32 + grp]);
      uint4* o = out + row * 16;
      o[lane8] = make_uint4(v.x ^ sb, v.y, v.z, v.w);
      o[8 + lane8] = make_uint4(v.x, v.y ^ sb, v.z, v.w);
    }
    __syncwarp();  // the next pass overwrites this warp's slots
  }
}

template <int U>
int time_gather_async(const Gather& g, const char* what, int blocks, int64_t* const* idx) {
  const int reps = 200;
  const int smem = U * 4224;
  CK(cudaFuncSetAttribute(probe_gather_async<U>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  for (int w = 0; w < 3; ++w) probe_gather_async<U><<<blocks, 256, smem>>>(g.base, g.sbase, idx[w & 3], g.out, kN);
  CK(cudaGetLastError());
  CK(cudaDeviceSynchronize());
  CK(cudaEventRecord(g.e0));
  for (int i = 0; i < reps; ++i) probe_gather_async<U><<<blocks, 256, smem>>>(g.base, g.sbase, idx[i & 3], g.out, kN);
  CK(cudaEventRecord(g.e1));
  CK(cudaEventSynchronize(g.e1));
  float ms = 0.f;
  CK(cudaEventElapsedTime(&ms, g.e0, g.e1));
  std::printf("%-44s %-10s grid %6d x 256, %d rows/thread-group pass: %7.1f us per launch\n", what, "read+write",
              blocks, U, ms * 1e3 / reps);
  return 0;
}

int run_access(int64_t region_bytes) {
  const int64_t slots = region_bytes / 128;
  unsigned char* region;
  int64_t* idx;
  uint32_t* sink;
  CK(cudaMalloc(&region, slots * 128));
  CK(cudaMalloc(&idx, kN * 8));
  CK(cudaMalloc(&sink, 4));
  make_idx<<<(unsigned)((kN + 255) / 256), 256>>>(idx, kN, slots, 3);
  CK(cudaDeviceSynchronize());
  cudaEvent_t e0, e1;
  CK(cudaEventCreate(&e0));
  CK(cudaEventCreate(&e1));
  std::printf("access probe: %lld random reads per launch into %.1f GB (one 128-B slot each)\n", (long long)kN,
              slots * 128 / 1e9);
  auto timed = [&](auto kernel, const char* name, int bytes, int lanes) -> int {
    const int64_t threads = kN * lanes;
    const unsigned blocks = (unsigned)((threads + 255) / 256);
    for (int r = 0; r < 3; ++r) kernel<<<blocks, 256>>>(region, idx, kN, sink);
    CK(cudaGetLastError());
    CK(cudaEventRecord(e0));
    kernel<<<blocks, 256>>>(region, idx, kN, sink);
    CK(cudaEventRecord(e1));
    CK(cudaEventSynchronize(e1));
    float ms = 0.f;
    CK(cudaEventElapsedTime(&ms, e0, e1));
    std::printf("%-28s %3d-byte accesses, %7.1f us\n", name, bytes, ms * 1e3);
    return 0;
  };
  int rc = 0;
  rc |= timed(probe_read<4>, "probe_read<4>", 4, 1);
  rc |= timed(probe_read<16>, "probe_read<16>", 16, 1);
  rc |= timed(probe_read<32>, "probe_read<32>", 32, 2);
  rc |= timed(probe_read<64>, "probe_read<64>", 64, 4);
  rc |= timed(probe_read<128>, "probe_read<128>", 128, 8);
  std::printf("4-byte reads with other load flavours:\n");
  rc |= timed(probe_read_flavour<0>, "probe_read_flavour<.cg>", 4, 1);
  rc |= timed(probe_read_flavour<1>, "probe_read_flavour<.cs>", 4, 1);
  rc |= timed(probe_read_flavour<2>, "probe_read_flavour<relaxed>", 4, 1);
  size_t gran = 0;
  CK(cudaDeviceGetLimit(&gran, cudaLimitMaxL2FetchGranularity));
  CK(cudaDeviceSetLimit(cudaLimitMaxL2FetchGranularity, 32));
  size_t now = 0;
  CK(cudaDeviceGetLimit(&now, cudaLimitMaxL2FetchGranularity));
  std::printf("L2 fetch granularity limit %zu -> %zu bytes for this context:\n", gran, now);
  rc |= timed(probe_read<4>, "probe_read<4> (32-B limit)", 4, 1);
  CK(cudaDeviceSetLimit(cudaLimitMaxL2FetchGranularity, gran));
  return rc;
}

int run_gather(int mode) {  // 0 gather, 1 layout, 2 depth
  const int64_t region = kRowsFull * 144;  // 110.6 GB: room for every layout
  Gather g;
  unsigned char* base;
  CK(cudaMalloc(&base, region));
  CK(cudaMalloc(&g.out, kN * 256));
  int64_t* half[4];
  for (int i = 0; i < 4; ++i) {
    CK(cudaMalloc(&g.idx[i], kN * 8));
    CK(cudaMalloc(&half[i], kN * 8));
    make_idx<<<(unsigned)((kN + 255) / 256), 256>>>(g.idx[i], kN, kRowsFull, 11 + i);
    make_idx<<<(unsigned)((kN + 255) / 256), 256>>>(half[i], kN, kRowsFull / 2, 21 + i);  // 256-B records
  }
  CK(cudaDeviceSynchronize());
  g.base = base;
  g.sbase = reinterpret_cast<const float*>(base + kRowsFull * 128);
  CK(cudaEventCreate(&g.e0));
  CK(cudaEventCreate(&g.e1));
  int sms = 0;
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  const int short_ctas = (int)(kN / 128);  // 128 rows per CTA, one pass of 4 rows per thread group
  int rc = 0;
  std::printf("gather probe: %lld random rows per launch out of %lld (128-B codes + 4-B scale read, 256 B written)\n",
              (long long)kN, (long long)kRowsFull);
  if (mode == 2) {  // rows in flight: registers vs shared memory, at the 32-B fetch limit
    size_t gran = 0;
    CK(cudaDeviceGetLimit(&gran, cudaLimitMaxL2FetchGranularity));
    CK(cudaDeviceSetLimit(cudaLimitMaxL2FetchGranularity, 32));
    std::printf("L2 fetch granularity limit %zu -> 32 bytes:\n", gran);
    rc |= time_gather<2, 0, 0, 0>(g, "registers, short CTAs", (int)(kN / 64), g.idx);
    rc |= time_gather<4, 0, 0, 0>(g, "registers, short CTAs", short_ctas, g.idx);
    rc |= time_gather<8, 0, 0, 0>(g, "registers, short CTAs", (int)(kN / 256), g.idx);
    rc |= time_gather_async<4>(g, "cp.async to shared memory, short CTAs", short_ctas, g.idx);
    rc |= time_gather_async<8>(g, "cp.async to shared memory, short CTAs", (int)(kN / 256), g.idx);
    rc |= time_gather_async<16>(g, "cp.async to shared memory, short CTAs", (int)(kN / 512), g.idx);
    rc |= time_gather_async<8>(g, "cp.async to shared memory, 6 CTAs/SM", sms * 6, g.idx);
    CK(cudaDeviceSetLimit(cudaLimitMaxL2FetchGranularity, gran));
  } else if (mode == 0) {
    rc |= time_gather<4, 0, 0, 0>(g, "separate scales, short CTAs", short_ctas, g.idx);
    rc |= time_gather<4, 0, 0, 3>(g, "separate scales, short CTAs", short_ctas, g.idx);
    rc |= time_gather<4, 0, 0, 4>(g, "separate scales, short CTAs", short_ctas, g.idx);
    rc |= time_gather<1, 0, 0, 0>(g, "separate scales, one row per thread group", (int)(kN / 32), g.idx);
    rc |= time_gather<4, 0, 0, 0>(g, "separate scales, persistent 4 CTAs/SM", sms * 4, g.idx);
    rc |= time_gather<8, 0, 0, 0>(g, "separate scales, persistent 8 CTAs/SM", sms * 8, g.idx);
    rc |= time_gather<4, 0, 0, 0>(g, "separate scales, 32 CTAs/SM", sms * 32, g.idx);
    rc |= time_gather<4, 0, 0, 1>(g, "separate scales, short CTAs", short_ctas, g.idx);
    rc |= time_gather<1, 0, 0, 1>(g, "separate scales, one row per thread group", (int)(kN / 32), g.idx);
    rc |= time_gather<4, 0, 0, 2>(g, "separate scales, 8 CTAs/SM", sms * 8, g.idx);
    size_t gran = 0;  // the same patterns with the context's L2 fetch granularity limit at 32 bytes
    CK(cudaDeviceGetLimit(&gran, cudaLimitMaxL2FetchGranularity));
    CK(cudaDeviceSetLimit(cudaLimitMaxL2FetchGranularity, 32));
    std::printf("L2 fetch granularity limit %zu -> 32 bytes:\n", gran);
    rc |= time_gather<4, 0, 0, 0>(g, "separate scales, short CTAs", short_ctas, g.idx);
    rc |= time_gather<4, 0, 0, 4>(g, "separate scales, short CTAs", short_ctas, g.idx);
    rc |= time_gather<4, 0, 0, 1>(g, "separate scales, short CTAs", short_ctas, g.idx);
    CK(cudaDeviceSetLimit(cudaLimitMaxL2FetchGranularity, gran));
  } else {
    for (int m = 0; m < 2; ++m) {
      if (m == 0) {
        rc |= time_gather<4, 0, 0, 0>(g, "separate scales", short_ctas, g.idx);
        rc |= time_gather<4, 1, 0, 0>(g, "codes only (no scale read)", short_ctas, g.idx);
        rc |= time_gather<4, 2, 144, 0>(g, "144-B records (scale after the codes)", short_ctas, g.idx);
        rc |= time_gather<4, 2, 256, 0>(g, "256-B records (384M rows)", short_ctas, half);
        rc |= time_gather<4, 3, 0, 0>(g, "blocks of 32 rows + their 32 scales", short_ctas, g.idx);
      } else {
        rc |= time_gather<4, 0, 0, 1>(g, "separate scales", short_ctas, g.idx);
        rc |= time_gather<4, 1, 0, 1>(g, "codes only (no scale read)", short_ctas, g.idx);
        rc |= time_gather<4, 2, 144, 1>(g, "144-B records (scale after the codes)", short_ctas, g.idx);
        rc |= time_gather<4, 2, 256, 1>(g, "256-B records (384M rows)", short_ctas, half);
        rc |= time_gather<4, 3, 0, 1>(g, "blocks of 32 rows + their 32 scales", short_ctas, g.idx);
      }
    }
  }
  return rc;
}

}  // namespace

int main(int argc, char** argv) {
  if (argc != 2 || (std::strcmp(argv[1], "access") && std::strcmp(argv[1], "gather") && std::strcmp(argv[1], "layout") &&
                    std::strcmp(argv[1], "depth"))) {
    std::printf("usage: %s access|gather|layout|depth\n", argv[0]);
    return 2;
  }
  size_t free_b = 0, total_b = 0;
  CK(cudaMemGetInfo(&free_b, &total_b));
  const bool access = !std::strcmp(argv[1], "access");
  const int64_t need = access ? (int64_t)48e9 + kN * 8 : kRowsFull * 144 + kN * (256 + 64);
  if ((int64_t)free_b < need + ((int64_t)2 << 30)) {
    std::printf("probe needs %.1f GB of free device memory, %.1f GB free\n", need / 1e9, free_b / 1e9);
    return 3;
  }
  if (access) return run_access((int64_t)48e9);
  return run_gather(!std::strcmp(argv[1], "layout") ? 1 : (!std::strcmp(argv[1], "depth") ? 2 : 0));
}
