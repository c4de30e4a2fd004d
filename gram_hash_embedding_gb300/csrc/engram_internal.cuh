// Internal declarations shared by the kernels and the C-ABI layer of libengram.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/engram.h"

namespace engram {

// One hash column (layer l, n-gram size n, head h) as the kernels use it.
struct ColParam {
  uint64_t prime;   // P, 1 <= P < 2^62
  uint64_t magic;   // floor((2^64 - 1) / P): quotient estimate that is exact or one short
  uint64_t wrap;    // 2^64 mod P: corrects the unsigned residue of a negative int64
  int64_t offset;   // the column's first row in the layer's table
};

// Device-resident view of a state, passed by value to the kernels.
struct StateView {
  const int32_t* token_map;  // [raw_vocab]
  const uint64_t* mult;      // [n_layers][max_ngram]
  const ColParam* cols;      // [n_layers][C]
  int32_t* cache;            // [max_batch][max_seq_len]
  unsigned int* status;      // ENGRAM_STATUS_* bits
  int64_t raw_vocab;
  int64_t max_seq_len;
  int64_t pad_id;
  int32_t dead;
  int32_t max_batch;
  int32_t n_layers, max_ngram, n_heads, n_cols;
};

// Per-call arguments of the hash / fused kernels.
struct CallArgs {
  const int64_t* ids;
  const uint8_t* mask;        // may be null
  const int32_t* start_pos;
  const int32_t* cache_rows;  // [B] cache row of each call row; null: row b uses cache row b
  int64_t* hashes;            // may be null (fused)
  const int32_t* cu_seqlens;  // packed calls: [B+1] sequence extents in ids; null for dense [B, L] calls
  int64_t L;                  // dense: tokens per row; packed: max_len (a longer sequence is skipped)
  int64_t total;              // packed: tokens in ids (T); dense: B * L
  int32_t B;
  int32_t early;              // fused dense calls: 1 when the host found that none of this call's inputs (ids,
                              // mask, start_pos, cache_rows, tables) is written by the previous kernel of this
                              // library on the stream, so they may be read before pdl_wait()
  int32_t head_dim, block;
  int32_t scale_dtype;        // ENGRAM_SCALE_*: storage type of S
  const uint8_t* W[ENGRAM_MAX_LAYERS];
  const void* S[ENGRAM_MAX_LAYERS];
  int64_t rows[ENGRAM_MAX_LAYERS];
  uint16_t* out[ENGRAM_MAX_LAYERS];
};

// Programmatic dependent launch. Every kernel of this library starts with pdl_wait(): it returns
// once the kernel before it on the stream has completed and its writes are visible (at once when
// there is none or the launch was not programmatic), so stream order holds for every global read
// and write. Then pdl_trigger() lets the next launch be scheduled while this grid drains: its CTAs
// take SM slots as this grid's last wave leaves instead of after a full launch gap.
#ifndef ENGRAM_PDL
#define ENGRAM_PDL 1
#endif

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KernelArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KernelArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = ENGRAM_PDL;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Launchers (kernels.cu). Return cudaGetLastError() of the launch.
cudaError_t launch_fill_i32(int32_t* p, int64_t n, int32_t value, cudaStream_t s);
cudaError_t launch_hash(const StateView& sv, const CallArgs& a, cudaStream_t s);
cudaError_t launch_hash_lookup(const StateView& sv, const CallArgs& a, cudaStream_t s);
cudaError_t launch_gate(const uint16_t* x, const uint16_t* kv, const uint16_t* qw, const uint16_t* kw,
                        const uint8_t* mask, int64_t T, int hc, int dim, float eps, uint16_t* out, cudaStream_t s);
cudaError_t launch_lookup(const int64_t* idx, int64_t n_idx, const uint8_t* W, const void* S, int64_t rows,
                          int32_t head_dim, int32_t block, int32_t scale_dtype, uint16_t* out, cudaStream_t s);

}  // namespace engram
