// Row-sharded lookup over several ranks ("DeepSeek V4.1" pages, engram-first/lookup page,
// `ParallelEngramEmbedding`): rank r holds rows [r * part, (r + 1) * part) of each table, with
// part = ceil(rows / world). The pages look up every index on every rank, zero the rows a rank does
// not own and sum the mostly-zero [.., D] results over all ranks with an all-reduce. Here a rank
// instead sends each of its requests only to the rank that owns the row and receives that one row
// back: these kernels are the two ends of that exchange.
//
//   shard_pack   groups the indices of one lookup by owning rank (bucket `world` = indices outside
//                [0, rows), which no rank owns), stable within a bucket, and emits for each the
//                owner-local row id and its position in the request list; the bucket sizes are the
//                split sizes of the all-to-all exchanges.
//   shard_unpack scatters the rows received back (in the packed order) to their positions and writes
//                +0 rows at the positions of the unowned indices, as the pages' masked rows.
//
// Design: pack is two passes over the indices (8 B read per index per pass, 16 B written) around a
// one-CTA scan: a per-segment count, the scan that turns the counts into each segment's start in
// each bucket, then a scatter that ranks the elements of a segment with warp ballots, so the order is
// deterministic. Unpack moves
// 2 * head_dim bytes per row with 16-byte accesses.
#include <cstdint>
#include <mutex>

#include "engram_internal.cuh"
#include "proj.cuh"

namespace engram {
namespace {

constexpr int kPackThreads = 256;
constexpr int kPackPerThread = 16;
constexpr int kSeg = kPackThreads * kPackPerThread;  // indices per segment (one CTA)
constexpr int kMaxBuckets = ENGRAM_MAX_SHARDS + 1;

__device__ __forceinline__ int bucket_of(int64_t v, int64_t rows, int64_t part, int world) {
  if (v < 0 || v >= rows) return world;
  return (int)(v / part);
}

// seg_counts[s][b]: indices of segment s in bucket b
__global__ void __launch_bounds__(kPackThreads) shard_count_kernel(const int64_t* __restrict__ idx, int64_t n,
                                                                   int64_t rows, int64_t part, int world,
                                                                   int32_t* __restrict__ seg_counts) {
  pdl_wait();
  pdl_trigger();
  __shared__ int cnt[kMaxBuckets];
  const int nb = world + 1;
  for (int b = threadIdx.x; b < nb; b += blockDim.x) cnt[b] = 0;
  __syncthreads();
  const int64_t s0 = (int64_t)blockIdx.x * kSeg;
  int64_t v[kPackPerThread];  // all of this thread's indices in flight at once
#pragma unroll
  for (int j = 0; j < kPackPerThread; ++j) {
    const int64_t i = s0 + (int64_t)j * kPackThreads + threadIdx.x;
    v[j] = i < n ? idx[i] : -1;
  }
#pragma unroll
  for (int j = 0; j < kPackPerThread; ++j) {
    const int64_t i = s0 + (int64_t)j * kPackThreads + threadIdx.x;
    if (i < n) atomicAdd(&cnt[bucket_of(v[j], rows, part, world)], 1);
  }
  __syncthreads();
  for (int b = threadIdx.x; b < nb; b += blockDim.x) seg_counts[(int64_t)blockIdx.x * nb + b] = cnt[b];
}

// One CTA: turns seg_counts[s][b] (the count of segment s in bucket b) into the position where segment
// s's entries of bucket b start in the packed arrays (buckets one after the other, segments in order
// inside a bucket), in place, and writes the bucket totals to counts. Offsets fit int32: n < 2^31.
constexpr int kScanThreads = 1024;
__global__ void __launch_bounds__(kScanThreads) shard_scan_kernel(int32_t* __restrict__ seg_counts, int64_t n_seg,
                                                                  int world, int64_t* __restrict__ counts) {
  pdl_wait();
  pdl_trigger();
  __shared__ int32_t warp_sums[kScanThreads / 32];
  __shared__ int32_t carry_s;
  const int nb = world + 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t bucket_start = 0;  // entries of the buckets before b
  for (int b = 0; b < nb; ++b) {
    if (tid == 0) carry_s = bucket_start;
    __syncthreads();
    for (int64_t s0 = 0; s0 < n_seg; s0 += kScanThreads) {
      const int64_t s = s0 + tid;
      const int32_t c = s < n_seg ? seg_counts[s * nb + b] : 0;
      // inclusive scan of c over the CTA: within the warp, then over the warps' sums
      int32_t x = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) warp_sums[warp] = x;
      __syncthreads();
      if (warp == 0) {
        int32_t w = lane < kScanThreads / 32 ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
          if (lane >= o) w += y;
        }
        if (lane < kScanThreads / 32) warp_sums[lane] = w;  // inclusive over the warps
      }
      __syncthreads();
      const int32_t before = carry_s + (warp > 0 ? warp_sums[warp - 1] : 0) + x - c;
      if (s < n_seg) seg_counts[s * nb + b] = before;
      __syncthreads();
      if (tid == 0) carry_s += warp_sums[kScanThreads / 32 - 1];
      __syncthreads();
    }
    const int32_t total = carry_s - bucket_start;
    if (tid == 0) counts[b] = total;
    bucket_start = carry_s;
    __syncthreads();
  }
}

// Writes every index of segment s to its bucket, in index order within the bucket, from the start
// positions shard_scan_kernel left in seg_base.
__global__ void __launch_bounds__(kPackThreads) shard_scatter_kernel(const int64_t* __restrict__ idx, int64_t n,
                                                                     int64_t rows, int64_t part, int world,
                                                                     const int32_t* __restrict__ seg_base,
                                                                     int64_t* __restrict__ local_rows,
                                                                     int64_t* __restrict__ positions) {
  pdl_wait();
  pdl_trigger();
  __shared__ int32_t base[kMaxBuckets];                      // where this segment's part of bucket b goes next
  __shared__ int warp_cnt[kPackThreads / 32][kMaxBuckets];   // this pass's elements per (warp, bucket)
  const int nb = world + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int b = threadIdx.x; b < nb; b += blockDim.x) base[b] = seg_base[(int64_t)blockIdx.x * nb + b];
  const int64_t s0 = (int64_t)blockIdx.x * kSeg;
  const unsigned lt = (1u << lane) - 1u;
  int64_t vals[kPackPerThread];  // all of this thread's indices in flight at once
#pragma unroll
  for (int j = 0; j < kPackPerThread; ++j) {
    const int64_t i = s0 + (int64_t)j * kPackThreads + threadIdx.x;
    vals[j] = i < n ? idx[i] : 0;
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kPackPerThread; ++j) {
    const int64_t i = s0 + (int64_t)j * kPackThreads + threadIdx.x;
    const bool in = i < n;
    const int64_t v = vals[j];
    const int b = in ? bucket_of(v, rows, part, world) : -1;
    // rank of this element among the warp's elements of the same bucket
    int my_rank = 0;
    for (int bb = 0; bb < nb; ++bb) {
      const unsigned m = __ballot_sync(0xffffffffu, b == bb);
      if (b == bb) my_rank = __popc(m & lt);
      if (lane == 0) warp_cnt[warp][bb] = __popc(m);
    }
    __syncthreads();
    if (in) {
      int64_t off = (int64_t)base[b] + my_rank;
      for (int w = 0; w < warp; ++w) off += warp_cnt[w][b];
      local_rows[off] = b < world ? v - (int64_t)b * part : v;
      positions[off] = i;
    }
    __syncthreads();
    if (threadIdx.x < nb) {
      int add = 0;
      for (int w = 0; w < kPackThreads / 32; ++w) add += warp_cnt[w][threadIdx.x];
      base[threadIdx.x] += add;
    }
    __syncthreads();
  }
}

// unit u = (entry u / G, 16-byte piece u % G) with G = 2 * D / 16 pieces per row
__global__ void __launch_bounds__(256) shard_unpack_kernel(const uint4* __restrict__ recv,
                                                           const int64_t* __restrict__ positions, int64_t m,
                                                           int64_t n, int G, uint4* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int64_t units = n * G;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units; u += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = u / G;
    const int q = (int)(u - e * G);
    const int64_t pos = positions[e];
    if (pos < 0 || pos >= n) continue;  // not a position of this lookup: nothing to write
    out[pos * G + q] = e < m ? recv[e * G + q] : make_uint4(0u, 0u, 0u, 0u);
  }
}

}  // namespace

int64_t shard_pack_segments(int64_t n) { return (n + kSeg - 1) / kSeg; }

cudaError_t launch_shard_pack(const int64_t* idx, int64_t n, int64_t rows, int32_t world, int64_t* counts,
                              int64_t* local_rows, int64_t* positions, int32_t* seg_counts, cudaStream_t s) {
  const int64_t part = (rows + world - 1) / world;
  const int64_t n_seg = shard_pack_segments(n);
  cudaError_t e = launch_pdl(shard_count_kernel, dim3((unsigned)n_seg), dim3(kPackThreads), 0, s, idx, n, rows,
                             part < 1 ? (int64_t)1 : part, (int)world, seg_counts);
  if (e != cudaSuccess) return e;
  e = launch_pdl(shard_scan_kernel, dim3(1), dim3(kScanThreads), 0, s, seg_counts, n_seg, (int)world, counts);
  if (e != cudaSuccess) return e;
  return launch_pdl(shard_scatter_kernel, dim3((unsigned)n_seg), dim3(kPackThreads), 0, s, idx, n, rows,
                    part < 1 ? (int64_t)1 : part, (int)world, (const int32_t*)seg_counts, local_rows, positions);
}

cudaError_t launch_shard_unpack(const uint16_t* recv, const int64_t* positions, int64_t m, int64_t n,
                                int32_t head_dim, uint16_t* out, cudaStream_t s) {
  const int G = head_dim * 2 / 16;
  const int64_t units = n * G;
  int64_t blocks = (units + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  return launch_pdl(shard_unpack_kernel, dim3((unsigned)blocks), dim3(256), 0, s,
                    reinterpret_cast<const uint4*>(recv), positions, m, n, G, reinterpret_cast<uint4*>(out));
}

}  // namespace engram

// ------------------------------------------------------------------------------------------------
// engram_shard_pack_static: the same pack for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc (or any routine that allocates) at the point where they pack:
// a serving loop whose device memory is all handed out up front by its own pool, code that runs
// while a stream is being captured into a CUDA graph (where a plain cudaMalloc is not allowed), or a
// runtime that forbids the latency and synchronisation of an allocation on its hot path. They still
// own the inputs and outputs; only the pack's scratch (one int32 count per segment of 4096 indices
// and bucket) comes from this fixed array instead of a caller's workspace. Every device that loads
// the library holds the array until the process exits.
namespace engram {

constexpr int64_t kStaticPackCounts = 16384;  // 64 KB: n <= 16384 / (world + 1) segments of 4096 indices
__device__ __align__(256) static int32_t g_pack_scratch[kStaticPackCounts];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_pack_scratch_mutex;
int32_t* g_pack_scratch_ptr[kMaxDevices] = {};  // device address of g_pack_scratch, per device
}  // namespace

int64_t static_pack_max_n(int32_t world) { return (kStaticPackCounts / (world + 1)) * (int64_t)kSeg; }

// The array's device address on the current device, looked up once per device. In host code the
// name g_pack_scratch is only a host-side stand-in, never a device address.
cudaError_t static_pack_scratch(int32_t** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_pack_scratch_mutex);
  if (g_pack_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_pack_scratch);
    if (e != cudaSuccess) return e;
    g_pack_scratch_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_pack_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace engram
