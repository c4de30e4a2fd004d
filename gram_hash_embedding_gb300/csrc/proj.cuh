// Internal declarations of the tensor-core projection (proj.cu), the gate's finishing pass (gate.cu)
// and the two ends of the sharded lookup's exchange (shard.cu), used by the C-ABI layer.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace engram {

// out[T][N] = bf16(emb[T][K] @ w[N][K]^T); withhold >= 0: the test hook of engram_project_withhold
cudaError_t launch_project(const uint16_t* emb, const uint16_t* w, int64_t T, int32_t K, int32_t N, uint16_t* out,
                           cudaStream_t s, int32_t withhold = -1);

// columns of the projection's output tiles for a call of T tokens (128 or 256); the gate's partial
// sums come one set per tile
int64_t project_tile_cols(int64_t T);

// fp32 values of the partial-sum array of the fused gate projection for T tokens
int64_t project_gate_partials(int64_t T, int32_t hc, int32_t dim);

// projection with the gate epilogue: value [T][dim] bf16 and the key tiles' partial sums
cudaError_t launch_project_gate_sums(const uint16_t* x, const uint16_t* emb, const uint16_t* wkv, const uint16_t* qw,
                                     const uint16_t* kw, int64_t T, int32_t K, int32_t hc, int32_t dim,
                                     uint16_t* value, float* part, cudaStream_t s);

// The projection with its A looked up inside the same kernel, one tile group ahead of the loads
// (engram_lookup_project*): token t's row ids at idx[t * idx_stride + c], c < n_cols; A = emb
// [T][n_cols * head_dim] bf16, a workspace written by the kernel; counters: lookup_ahead_counters(T)
// words of workspace, zeroed by the launcher on the stream.
struct LookupArgs {
  const int64_t* idx;
  int64_t idx_stride;
  int32_t n_cols;
  const uint8_t* W;
  const void* S;
  int64_t rows;
  int32_t head_dim, block, scale_dtype;
  uint16_t* emb;
  unsigned int* counters;
};
int64_t lookup_ahead_counters(int64_t T);
cudaError_t launch_lookup_project(const LookupArgs& la, const uint16_t* wkv, int64_t T, int32_t N, uint16_t* out,
                                  cudaStream_t s);
cudaError_t launch_lookup_project_gate_sums(const uint16_t* x, const LookupArgs& la, const uint16_t* wkv,
                                            const uint16_t* qw, const uint16_t* kw, int64_t T, int32_t hc,
                                            int32_t dim, uint16_t* value, float* part, cudaStream_t s);

// the gate from the partial sums, out = bf16(h + gate * value)
cudaError_t launch_gate_finish(const uint16_t* x, const uint16_t* value, const float* part, const uint8_t* mask,
                               int64_t T, int hc, int dim, float eps, uint16_t* out, cudaStream_t s);

cudaError_t device_status_take(unsigned int* flags, int clear, cudaStream_t s);

// sharded lookup: segments of the pack's count pass (one int32 count per segment and bucket)
int64_t shard_pack_segments(int64_t n);
cudaError_t launch_shard_pack(const int64_t* idx, int64_t n, int64_t rows, int32_t world, int64_t* counts,
                              int64_t* local_rows, int64_t* positions, int32_t* seg_counts, cudaStream_t s);
// engram_shard_pack_static: largest n for `world` ranks, and the fixed scratch array's device address
int64_t static_pack_max_n(int32_t world);
cudaError_t static_pack_scratch(int32_t** out);
cudaError_t launch_shard_unpack(const uint16_t* recv, const int64_t* positions, int64_t m, int64_t n,
                                int32_t head_dim, uint16_t* out, cudaStream_t s);

}  // namespace engram
