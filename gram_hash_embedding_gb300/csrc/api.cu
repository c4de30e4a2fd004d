// C ABI of libengram: state management, host-side argument checks, launches.
// Declarations and the contract of every entry point are in include/engram.h.
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "engram_internal.cuh"
#include "proj.cuh"

struct engram_state {
  engram_layout lay;
  int device;
  int32_t* d_token_map;
  uint64_t* d_mult;
  engram::ColParam* d_cols;
  int32_t* d_cache;
  unsigned int* d_status;
  unsigned int* d_status_taken;  // engram_state_status: the word as read by the atomic exchange
};

namespace {

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Return code of a launch path. A failed launch leaves its error in the runtime's last-error slot,
// where the caller's next unrelated launch check would find it; take it out here.
inline int launch_rc(cudaError_t e) {
  if (e == cudaSuccess) return ENGRAM_OK;
  cudaGetLastError();
  return ENGRAM_ERR_CUDA;
}

// ------------------------------------------------------------------------------------------------
// What this library's last launch on each stream writes. Every kernel of the library is a
// programmatic dependent launch: it may be scheduled while the kernel before it on the stream drains,
// and only that kernel can still be running when it starts (a kernel launched otherwise, a copy or an
// event wait in between is waited for in full, and each of our kernels triggers its successor only
// after its own wait). So a fused hash + lookup may read its inputs before waiting when none of them
// overlaps what our last launch on the same stream writes; a stale record (a stream handle reused)
// can only be more cautious than needed, never less, because the kernel before it is then not ours.
struct Span {
  uintptr_t lo, hi;  // [lo, hi)
};

std::mutex g_writes_mutex;
std::unordered_map<uintptr_t, std::vector<Span>> g_last_writes;

inline Span span(const void* p, uint64_t bytes) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return Span{lo, lo + (uintptr_t)bytes};
}

// The per-thread default stream is a different stream in every host thread, so its record is the
// thread's own; cudaStreamLegacy and the null handle name the same (legacy) stream.
thread_local std::vector<Span> t_per_thread_writes;
thread_local bool t_per_thread_recorded = false;

uintptr_t stream_key(cudaStream_t s) { return s == cudaStreamLegacy ? 0 : reinterpret_cast<uintptr_t>(s); }

void record_writes(cudaStream_t s, std::vector<Span> writes) {
  if (s == cudaStreamPerThread) {
    t_per_thread_writes = std::move(writes);
    t_per_thread_recorded = true;
    return;
  }
  std::lock_guard<std::mutex> lock(g_writes_mutex);
  g_last_writes[stream_key(s)] = std::move(writes);
}

bool overlaps(const std::vector<Span>& writes, const std::vector<Span>& inputs) {
  for (const Span& w : writes)
    for (const Span& r : inputs)
      if (r.lo < w.hi && w.lo < r.hi) return true;
  return false;
}

bool untouched_by_last_launch(cudaStream_t s, const std::vector<Span>& inputs) {
  if (s == cudaStreamPerThread) return !t_per_thread_recorded || !overlaps(t_per_thread_writes, inputs);
  std::lock_guard<std::mutex> lock(g_writes_mutex);
  auto it = g_last_writes.find(stream_key(s));
  return it == g_last_writes.end() || !overlaps(it->second, inputs);
}

// After a launch path: record what it wrote on success; after a failure what ran is unknown, so the
// next fused call on the stream reads nothing early.
int launched(int rc, cudaStream_t s, std::vector<Span> writes) {
  if (rc != ENGRAM_OK) writes = {Span{0, ~(uintptr_t)0}};
  record_writes(s, std::move(writes));
  return rc;
}

// Reads the status word and, when asked, clears it in the same atomic step, so that a flag raised
// by a kernel on another stream between the read and the clear is not lost.
__global__ void status_take_kernel(unsigned int* status, unsigned int* taken, int clear) {
  *taken = clear ? atomicExch(status, 0u) : atomicOr(status, 0u);
}

inline bool head_dim_ok(int32_t D, int32_t block) {
  const bool pow2 = D == 16 || D == 32 || D == 64 || D == 128 || D == 256 || D == 512;
  return pow2 && block >= 8 && block % 8 == 0 && D % block == 0;
}

int cols_total(const engram_layout& l) { return l.n_layers * (l.max_ngram - 1) * l.n_heads; }

inline bool scale_dtype_ok(int32_t t) { return t >= ENGRAM_SCALE_F32 && t <= ENGRAM_SCALE_E4M3; }

// bytes of one stored scale (also the alignment S needs)
inline uintptr_t scale_bytes(int32_t t) {
  return t == ENGRAM_SCALE_F32 ? 4 : (t == ENGRAM_SCALE_BF16 ? 2 : 1);
}

int check_layout(const engram_layout* l) {
  if (l == nullptr) return ENGRAM_ERR_INVALID;
  if (l->n_layers < 1 || l->max_ngram < 2 || l->n_heads < 1 || l->max_batch < 1 || l->max_seq_len < 1 ||
      l->raw_vocab < 1)
    return ENGRAM_ERR_INVALID;
  if (l->n_layers > ENGRAM_MAX_LAYERS || l->max_ngram > ENGRAM_MAX_NGRAM) return ENGRAM_ERR_UNSUPPORTED;
  if ((int64_t)l->n_layers * (l->max_ngram - 1) * l->n_heads > ENGRAM_MAX_COLS_TOTAL) return ENGRAM_ERR_UNSUPPORTED;
  if (l->max_batch > 65535 || l->max_seq_len > ((int64_t)1 << 40)) return ENGRAM_ERR_UNSUPPORTED;
  if (l->dead < INT32_MIN || l->dead > INT32_MAX) return ENGRAM_ERR_INVALID;
  if (!head_dim_ok(l->head_dim, l->block) || !scale_dtype_ok(l->scale_dtype)) return ENGRAM_ERR_UNSUPPORTED;
  return ENGRAM_OK;
}

engram::StateView view(const engram_state* st) {
  engram::StateView v;
  v.token_map = st->d_token_map;
  v.mult = st->d_mult;
  v.cols = st->d_cols;
  v.cache = st->d_cache;
  v.status = st->d_status;
  v.raw_vocab = st->lay.raw_vocab;
  v.max_seq_len = st->lay.max_seq_len;
  v.pad_id = st->lay.pad_id;
  v.dead = (int32_t)st->lay.dead;
  v.max_batch = st->lay.max_batch;
  v.n_layers = st->lay.n_layers;
  v.max_ngram = st->lay.max_ngram;
  v.n_heads = st->lay.n_heads;
  v.n_cols = (st->lay.max_ngram - 1) * st->lay.n_heads;
  return v;
}

bool on_state_device(const engram_state* st) {
  int dev = -1;
  return cudaGetDevice(&dev) == cudaSuccess && dev == st->device;
}

void free_state(engram_state* st) {
  if (st == nullptr) return;
  cudaFree(st->d_token_map);
  cudaFree(st->d_mult);
  cudaFree(st->d_cols);
  cudaFree(st->d_cache);
  cudaFree(st->d_status);
  cudaFree(st->d_status_taken);
  delete st;
}

// common checks of engram_hash / engram_hash_lookup
int check_call(const engram_state* st, const int64_t* ids, const uint8_t* mask, const int32_t* start_pos,
               const int32_t* cache_rows, int32_t B, int64_t L) {
  (void)mask;
  if (st == nullptr || B < 0 || L < 0) return ENGRAM_ERR_INVALID;
  if (B == 0 || L == 0) return ENGRAM_OK;
  if (ids == nullptr || start_pos == nullptr || !aligned(ids, 8) || !aligned(start_pos, 4)) return ENGRAM_ERR_INVALID;
  if (cache_rows != nullptr && !aligned(cache_rows, 4)) return ENGRAM_ERR_INVALID;
  if (B > st->lay.max_batch || L > st->lay.max_seq_len) return ENGRAM_ERR_RANGE;
  // tiles of >= 4 tokens keep the grid's x extent, ceil(L / tile), inside CUDA's 2^31 - 1
  if ((int64_t)B * L > ((int64_t)1 << 40) || L > ((int64_t)1 << 32)) return ENGRAM_ERR_UNSUPPORTED;
  if (!on_state_device(st)) return ENGRAM_ERR_INVALID;
  return ENGRAM_OK;
}

engram::CallArgs call_args(const engram_state* st, const int64_t* ids, const uint8_t* mask,
                           const int32_t* start_pos, const int32_t* cache_rows, int32_t B, int64_t L,
                           int64_t* hashes) {
  engram::CallArgs a;
  std::memset(&a, 0, sizeof a);
  a.ids = ids;
  a.mask = mask;
  a.start_pos = start_pos;
  a.cache_rows = cache_rows;
  a.hashes = hashes;
  a.cu_seqlens = nullptr;
  a.L = L;
  a.total = (int64_t)B * L;
  a.B = B;
  a.head_dim = st->lay.head_dim;
  a.block = st->lay.block;
  a.scale_dtype = st->lay.scale_dtype;
  return a;
}

// per-layer tables and outputs of a fused call (host arrays of n_layers device pointers)
int fill_tables(const engram_state* st, const uint8_t* const* W, const void* const* S, const int64_t* rows,
                uint16_t* const* out, engram::CallArgs* a) {
  if (W == nullptr || S == nullptr || rows == nullptr || out == nullptr) return ENGRAM_ERR_INVALID;
  const uintptr_t sb = scale_bytes(st->lay.scale_dtype);
  for (int l = 0; l < st->lay.n_layers; ++l) {
    if (rows[l] < 0 || out[l] == nullptr || !aligned(out[l], 16)) return ENGRAM_ERR_INVALID;
    if (rows[l] > 0 && (W[l] == nullptr || S[l] == nullptr || !aligned(W[l], 16) || !aligned(S[l], sb)))
      return ENGRAM_ERR_INVALID;
    a->W[l] = W[l];
    a->S[l] = S[l];
    a->rows[l] = rows[l];
    a->out[l] = out[l];
  }
  return ENGRAM_OK;
}

}  // namespace

extern "C" {

int engram_state_create(const engram_layout* layout, const int64_t* token_map, const int64_t* multipliers,
                        const int64_t* primes, const int64_t* offsets, engram_stream_t stream, engram_state** out) {
  if (out == nullptr) return ENGRAM_ERR_INVALID;
  *out = nullptr;
  int rc = check_layout(layout);
  if (rc != ENGRAM_OK) return rc;
  if (token_map == nullptr || multipliers == nullptr || primes == nullptr || offsets == nullptr)
    return ENGRAM_ERR_INVALID;
  const engram_layout& l = *layout;
  const int C = (l.max_ngram - 1) * l.n_heads;
  const int NC = cols_total(l);

  std::vector<int32_t> tm(l.raw_vocab);
  for (int64_t i = 0; i < l.raw_vocab; ++i) {
    if (token_map[i] < INT32_MIN || token_map[i] > INT32_MAX) return ENGRAM_ERR_INVALID;
    tm[i] = (int32_t)token_map[i];
  }
  std::vector<uint64_t> mult(l.n_layers * l.max_ngram);
  for (size_t i = 0; i < mult.size(); ++i) mult[i] = (uint64_t)multipliers[i];
  // column j = (n-2)*n_heads + h of layer ll uses primes[ll][n-2][h]: the same flat order
  std::vector<engram::ColParam> cols(NC);
  for (int ll = 0; ll < l.n_layers; ++ll) {
    for (int j = 0; j < C; ++j) {
      const int64_t p = primes[ll * C + j];
      const int64_t o = offsets[ll * C + j];
      if (p < 1 || p >= ((int64_t)1 << 62)) return ENGRAM_ERR_INVALID;
      if (o > INT64_MAX - (p - 1) || o < INT64_MIN + 1) return ENGRAM_ERR_INVALID;
      engram::ColParam& cp = cols[ll * C + j];
      cp.prime = (uint64_t)p;
      cp.magic = UINT64_MAX / (uint64_t)p;
      cp.wrap = (UINT64_MAX % (uint64_t)p + 1u) % (uint64_t)p;
      cp.offset = o;
    }
  }

  engram_state* st = new engram_state;
  std::memset(st, 0, sizeof *st);
  st->lay = l;
  if (cudaGetDevice(&st->device) != cudaSuccess) {
    delete st;
    return ENGRAM_ERR_CUDA;
  }
  cudaStream_t s = (cudaStream_t)stream;
  const int64_t cache_n = (int64_t)l.max_batch * l.max_seq_len;
  if (cudaMalloc(&st->d_token_map, tm.size() * sizeof(int32_t)) != cudaSuccess ||
      cudaMalloc(&st->d_mult, mult.size() * sizeof(uint64_t)) != cudaSuccess ||
      cudaMalloc(&st->d_cols, cols.size() * sizeof(engram::ColParam)) != cudaSuccess ||
      cudaMalloc(&st->d_cache, cache_n * sizeof(int32_t)) != cudaSuccess ||
      cudaMalloc(&st->d_status, sizeof(unsigned int)) != cudaSuccess ||
      cudaMalloc(&st->d_status_taken, sizeof(unsigned int)) != cudaSuccess) {
    cudaGetLastError();
    free_state(st);
    return ENGRAM_ERR_NOMEM;
  }
  cudaError_t e = cudaMemcpyAsync(st->d_token_map, tm.data(), tm.size() * sizeof(int32_t), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(st->d_mult, mult.data(), mult.size() * sizeof(uint64_t), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(st->d_cols, cols.data(), cols.size() * sizeof(engram::ColParam), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(st->d_status, 0, sizeof(unsigned int), s);
  if (e == cudaSuccess) e = engram::launch_fill_i32(st->d_cache, cache_n, (int32_t)l.dead, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);  // host staging vectors go out of scope
  if (e != cudaSuccess) {
    cudaGetLastError();
    free_state(st);
    return ENGRAM_ERR_CUDA;
  }
  *out = st;
  return ENGRAM_OK;
}

int engram_state_destroy(engram_state* state) {
  if (state == nullptr) return ENGRAM_OK;
  int prev = -1;
  cudaGetDevice(&prev);
  if (prev != state->device) cudaSetDevice(state->device);
  cudaDeviceSynchronize();
  free_state(state);
  if (prev >= 0 && prev != state->device) cudaSetDevice(prev);
  return ENGRAM_OK;
}

int engram_cache_reset(engram_state* state, engram_stream_t stream) {
  if (state == nullptr || !on_state_device(state)) return ENGRAM_ERR_INVALID;
  return launched(launch_rc(engram::launch_fill_i32(state->d_cache,
                                                    (int64_t)state->lay.max_batch * state->lay.max_seq_len,
                                                    (int32_t)state->lay.dead, (cudaStream_t)stream)),
                  (cudaStream_t)stream, {});
}

int engram_state_status(engram_state* state, engram_stream_t stream, uint32_t* flags, int clear) {
  if (state == nullptr || flags == nullptr || !on_state_device(state)) return ENGRAM_ERR_INVALID;
  cudaStream_t s = (cudaStream_t)stream;
  unsigned int v = 0;
  status_take_kernel<<<1, 1, 0, s>>>(state->d_status, state->d_status_taken, clear ? 1 : 0);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaMemcpyAsync(&v, state->d_status_taken, sizeof v, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return launched(launch_rc(e), s, {});
  *flags = v;
  return launched(ENGRAM_OK, s, {});
}

int engram_hash(engram_state* state, const int64_t* ids, const uint8_t* mask, const int32_t* start_pos,
                const int32_t* cache_rows, int32_t B, int64_t L, int64_t* hashes, engram_stream_t stream) {
  int rc = check_call(state, ids, mask, start_pos, cache_rows, B, L);
  if (rc != ENGRAM_OK || B == 0 || L == 0) return rc;
  if (hashes == nullptr || !aligned(hashes, 8)) return ENGRAM_ERR_INVALID;
  engram::CallArgs a = call_args(state, ids, mask, start_pos, cache_rows, B, L, hashes);
  const int NC = cols_total(state->lay);
  return launched(launch_rc(engram::launch_hash(view(state), a, (cudaStream_t)stream)), (cudaStream_t)stream,
                  {span(hashes, (uint64_t)B * L * NC * 8)});
}

int engram_lookup(const int64_t* idx, int64_t n_idx, const uint8_t* W, const void* S, int64_t rows,
                  int32_t head_dim, int32_t block, int32_t scale_dtype, uint16_t* out, engram_stream_t stream) {
  if (n_idx < 0 || rows < 0) return ENGRAM_ERR_INVALID;
  if (!head_dim_ok(head_dim, block) || !scale_dtype_ok(scale_dtype)) return ENGRAM_ERR_UNSUPPORTED;
  if (n_idx == 0) return ENGRAM_OK;
  if (idx == nullptr || out == nullptr || !aligned(idx, 8) || !aligned(out, 16)) return ENGRAM_ERR_INVALID;
  if (rows > 0 && (W == nullptr || S == nullptr || !aligned(W, 16) || !aligned(S, scale_bytes(scale_dtype))))
    return ENGRAM_ERR_INVALID;
  if (n_idx > ((int64_t)1 << 40)) return ENGRAM_ERR_UNSUPPORTED;
  return launched(
      launch_rc(engram::launch_lookup(idx, n_idx, W, S, rows, head_dim, block, scale_dtype, out, (cudaStream_t)stream)),
      (cudaStream_t)stream, {span(out, (uint64_t)n_idx * head_dim * 2)});
}

int engram_hash_lookup(engram_state* state, const int64_t* ids, const uint8_t* mask, const int32_t* start_pos,
                       const int32_t* cache_rows, int32_t B, int64_t L, const uint8_t* const* W,
                       const void* const* S, const int64_t* rows, uint16_t* const* out, int64_t* hashes,
                       engram_stream_t stream) {
  int rc = check_call(state, ids, mask, start_pos, cache_rows, B, L);
  if (rc != ENGRAM_OK || B == 0 || L == 0) return rc;
  if (hashes != nullptr && !aligned(hashes, 8)) return ENGRAM_ERR_INVALID;
  engram::CallArgs a = call_args(state, ids, mask, start_pos, cache_rows, B, L, hashes);
  rc = fill_tables(state, W, S, rows, out, &a);
  if (rc != ENGRAM_OK) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  const engram_layout& lay = state->lay;
  const int C = (lay.max_ngram - 1) * lay.n_heads;
  const uint64_t n_tok = (uint64_t)B * L;
  std::vector<Span> reads = {span(ids, n_tok * 8), span(start_pos, (uint64_t)B * 4)};
  if (mask != nullptr) reads.push_back(span(mask, n_tok));
  if (cache_rows != nullptr) reads.push_back(span(cache_rows, (uint64_t)B * 4));
  std::vector<Span> writes;
  if (hashes != nullptr) writes.push_back(span(hashes, n_tok * cols_total(lay) * 8));
  for (int l = 0; l < lay.n_layers; ++l) {
    reads.push_back(span(W[l], (uint64_t)rows[l] * lay.head_dim));
    reads.push_back(span(S[l], (uint64_t)rows[l] * (lay.head_dim / lay.block) * scale_bytes(lay.scale_dtype)));
    writes.push_back(span(out[l], n_tok * C * lay.head_dim * 2));
  }
  a.early = untouched_by_last_launch(s, reads) ? 1 : 0;
  return launched(launch_rc(engram::launch_hash_lookup(view(state), a, s)), s, std::move(writes));
}

namespace {

// common checks of the packed calls; on success fills *a (without tables)
int packed_call(const engram_state* st, const int64_t* ids, const uint8_t* mask, const int32_t* cu_seqlens,
                const int32_t* start_pos, const int32_t* cache_rows, int32_t B, int64_t T, int64_t max_len,
                int64_t* hashes, engram::CallArgs* a) {
  if (st == nullptr || B < 0 || T < 0 || max_len < 0) return ENGRAM_ERR_INVALID;
  if (B == 0 || T == 0 || max_len == 0) return ENGRAM_OK;
  if (ids == nullptr || cu_seqlens == nullptr || start_pos == nullptr || !aligned(ids, 8) ||
      !aligned(cu_seqlens, 4) || !aligned(start_pos, 4))
    return ENGRAM_ERR_INVALID;
  if (hashes != nullptr && !aligned(hashes, 8)) return ENGRAM_ERR_INVALID;
  if (cache_rows != nullptr && !aligned(cache_rows, 4)) return ENGRAM_ERR_INVALID;
  if (B > st->lay.max_batch || max_len > st->lay.max_seq_len) return ENGRAM_ERR_RANGE;
  // int32 extents; the packed grid then has floor(T / tile) + B < 2^29 + 2^16 CTAs (tiles of >= 4
  // tokens, B <= max_batch <= 65,535), inside CUDA's 2^31 - 1
  if (T > ((int64_t)1 << 31) - 1) return ENGRAM_ERR_UNSUPPORTED;
  if (!on_state_device(st)) return ENGRAM_ERR_INVALID;
  *a = call_args(st, ids, mask, start_pos, cache_rows, B, max_len, hashes);
  a->cu_seqlens = cu_seqlens;
  a->total = T;
  return ENGRAM_OK;
}

}  // namespace

int engram_hash_varlen(engram_state* state, const int64_t* ids, const uint8_t* mask, const int32_t* cu_seqlens,
                       const int32_t* start_pos, const int32_t* cache_rows, int32_t B, int64_t T, int64_t max_len,
                       int64_t* hashes, engram_stream_t stream) {
  if (hashes == nullptr && state != nullptr && B > 0 && T > 0 && max_len > 0) return ENGRAM_ERR_INVALID;
  engram::CallArgs a;
  int rc = packed_call(state, ids, mask, cu_seqlens, start_pos, cache_rows, B, T, max_len, hashes, &a);
  if (rc != ENGRAM_OK || B == 0 || T == 0 || max_len == 0) return rc;
  return launched(launch_rc(engram::launch_hash(view(state), a, (cudaStream_t)stream)), (cudaStream_t)stream,
                  {span(hashes, (uint64_t)T * cols_total(state->lay) * 8)});
}

int engram_hash_lookup_varlen(engram_state* state, const int64_t* ids, const uint8_t* mask,
                              const int32_t* cu_seqlens, const int32_t* start_pos, const int32_t* cache_rows,
                              int32_t B, int64_t T, int64_t max_len, const uint8_t* const* W, const void* const* S,
                              const int64_t* rows, uint16_t* const* out, int64_t* hashes, engram_stream_t stream) {
  engram::CallArgs a;
  int rc = packed_call(state, ids, mask, cu_seqlens, start_pos, cache_rows, B, T, max_len, hashes, &a);
  if (rc != ENGRAM_OK || B == 0 || T == 0 || max_len == 0) return rc;
  rc = fill_tables(state, W, S, rows, out, &a);
  if (rc != ENGRAM_OK) return rc;
  std::vector<Span> writes;
  const engram_layout& lay = state->lay;
  const int C = (lay.max_ngram - 1) * lay.n_heads;
  if (hashes != nullptr) writes.push_back(span(hashes, (uint64_t)T * cols_total(lay) * 8));
  for (int l = 0; l < lay.n_layers; ++l) writes.push_back(span(out[l], (uint64_t)T * C * lay.head_dim * 2));
  return launched(launch_rc(engram::launch_hash_lookup(view(state), a, (cudaStream_t)stream)), (cudaStream_t)stream,
                  std::move(writes));
}

int engram_gate(const uint16_t* x, const uint16_t* kv, const uint16_t* q_weight, const uint16_t* k_weight,
                const uint8_t* mask, int64_t T, int32_t hc, int32_t dim, float eps, uint16_t* out,
                engram_stream_t stream) {
  if (T < 0) return ENGRAM_ERR_INVALID;
  if (!(hc == 1 || hc == 2 || hc == 4 || hc == 8) || dim < 8 || dim % 8 != 0) return ENGRAM_ERR_UNSUPPORTED;
  if (T == 0) return ENGRAM_OK;
  if (T > ((int64_t)1 << 31) - 1) return ENGRAM_ERR_UNSUPPORTED;
  if (x == nullptr || kv == nullptr || q_weight == nullptr || k_weight == nullptr || out == nullptr)
    return ENGRAM_ERR_INVALID;
  if (!aligned(x, 16) || !aligned(kv, 16) || !aligned(q_weight, 16) || !aligned(k_weight, 16) || !aligned(out, 16))
    return ENGRAM_ERR_INVALID;
  return launched(
      launch_rc(engram::launch_gate(x, kv, q_weight, k_weight, mask, T, hc, dim, eps, out, (cudaStream_t)stream)),
      (cudaStream_t)stream, {span(out, (uint64_t)T * hc * dim * 2)});
}

int engram_project(const uint16_t* emb, const uint16_t* w, int64_t T, int32_t K, int32_t N, uint16_t* out,
                   engram_stream_t stream) {
  if (T < 0) return ENGRAM_ERR_INVALID;
  if (K < 8 || K % 8 != 0 || N < 8 || N % 8 != 0 || N > INT32_MAX - 256 || T > INT32_MAX)
    return ENGRAM_ERR_UNSUPPORTED;
  if (T == 0) return ENGRAM_OK;
  if (emb == nullptr || w == nullptr || out == nullptr || !aligned(emb, 16) || !aligned(w, 16) || !aligned(out, 16))
    return ENGRAM_ERR_INVALID;
  return launched(launch_rc(engram::launch_project(emb, w, T, K, N, out, (cudaStream_t)stream)), (cudaStream_t)stream,
                  {span(out, (uint64_t)T * N * 2)});
}

int engram_project_withhold(const uint16_t* emb, const uint16_t* w, int64_t T, int32_t K, int32_t N, uint16_t* out,
                            int32_t tile, engram_stream_t stream) {
  if (T < 0 || tile < 0) return ENGRAM_ERR_INVALID;
  if (K < 8 || K % 8 != 0 || N < 8 || N % 8 != 0 || N > INT32_MAX - 256 || T > INT32_MAX)
    return ENGRAM_ERR_UNSUPPORTED;
  if (T == 0) return ENGRAM_OK;
  if (emb == nullptr || w == nullptr || out == nullptr || !aligned(emb, 16) || !aligned(w, 16) || !aligned(out, 16))
    return ENGRAM_ERR_INVALID;
  return launched(launch_rc(engram::launch_project(emb, w, T, K, N, out, (cudaStream_t)stream, tile)),
                  (cudaStream_t)stream, {span(out, (uint64_t)T * N * 2)});
}

namespace {
inline bool gate_shape_ok(int32_t hc, int32_t dim) {
  return (hc == 1 || hc == 2 || hc == 4 || hc == 8) && dim >= 256 && dim % 256 == 0 &&
         (int64_t)(hc + 1) * dim <= INT32_MAX - 256;
}

uint64_t round256(uint64_t b) { return (b + 255u) & ~(uint64_t)255u; }
}  // namespace

uint64_t engram_project_gate_workspace(int64_t T, int32_t hc, int32_t dim) {
  if (T <= 0 || !gate_shape_ok(hc, dim)) return 0;
  return round256((uint64_t)T * (uint64_t)dim * 2u) +
         round256((uint64_t)engram::project_gate_partials(T, hc, dim) * sizeof(float));
}

int engram_project_gate(const uint16_t* x, const uint16_t* emb, const uint16_t* wkv, const uint16_t* q_weight,
                        const uint16_t* k_weight, const uint8_t* mask, int64_t T, int32_t K, int32_t hc, int32_t dim,
                        float eps, void* workspace, uint64_t workspace_bytes, uint16_t* out, engram_stream_t stream) {
  if (T < 0) return ENGRAM_ERR_INVALID;
  if (!gate_shape_ok(hc, dim) || K < 8 || K % 8 != 0 || T > INT32_MAX) return ENGRAM_ERR_UNSUPPORTED;
  if (T == 0) return ENGRAM_OK;
  if (x == nullptr || emb == nullptr || wkv == nullptr || q_weight == nullptr || k_weight == nullptr ||
      out == nullptr || workspace == nullptr)
    return ENGRAM_ERR_INVALID;
  if (!aligned(x, 16) || !aligned(emb, 16) || !aligned(wkv, 16) || !aligned(q_weight, 16) ||
      !aligned(k_weight, 16) || !aligned(out, 16) || !aligned(workspace, 256))
    return ENGRAM_ERR_INVALID;
  if (workspace_bytes < engram_project_gate_workspace(T, hc, dim)) return ENGRAM_ERR_INVALID;
  uint16_t* value = static_cast<uint16_t*>(workspace);
  float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + round256((uint64_t)T * dim * 2u));
  cudaStream_t s = (cudaStream_t)stream;
  int rc = launch_rc(engram::launch_project_gate_sums(x, emb, wkv, q_weight, k_weight, T, K, hc, dim, value, part, s));
  if (rc != ENGRAM_OK) return launched(rc, s, {});
  return launched(launch_rc(engram::launch_gate_finish(x, value, part, mask, T, hc, dim, eps, out, s)), s,
                  {span(out, (uint64_t)T * hc * dim * 2), span(workspace, workspace_bytes)});
}

namespace {
// workspace of the lookup-ahead projections: the looked-up rows, then the counters
uint64_t lookup_rows_bytes(int64_t T, int32_t n_cols, int32_t head_dim) {
  return round256((uint64_t)T * (uint64_t)n_cols * (uint64_t)head_dim * 2u);
}
uint64_t lookup_counter_bytes(int64_t T) { return round256((uint64_t)engram::lookup_ahead_counters(T) * 4u); }

// common checks of engram_lookup_project(_gate) past T == 0; fills the lookup arguments
int lookup_ahead_args(const int64_t* idx, int64_t idx_stride, int32_t n_cols, const engram_table* tb,
                      void* workspace, engram::LookupArgs* la) {
  if (idx == nullptr || !aligned(idx, 8) || idx_stride < n_cols || workspace == nullptr || !aligned(workspace, 256))
    return ENGRAM_ERR_INVALID;
  if (tb->rows > 0 && (tb->W == nullptr || tb->S == nullptr || !aligned(tb->W, 16) ||
                       !aligned(tb->S, scale_bytes(tb->scale_dtype))))
    return ENGRAM_ERR_INVALID;
  la->idx = idx;
  la->idx_stride = idx_stride;
  la->n_cols = n_cols;
  la->W = static_cast<const uint8_t*>(tb->W);
  la->S = tb->S;
  la->rows = tb->rows;
  la->head_dim = tb->head_dim;
  la->block = tb->block;
  la->scale_dtype = tb->scale_dtype;
  la->emb = static_cast<uint16_t*>(workspace);
  return ENGRAM_OK;
}

// the shape checks that do not depend on pointers (T >= 0 checked by the caller)
int lookup_ahead_shape(int64_t T, int32_t n_cols, const engram_table* tb) {
  if (tb == nullptr || n_cols < 1 || tb->rows < 0) return ENGRAM_ERR_INVALID;
  if (!head_dim_ok(tb->head_dim, tb->block) || !scale_dtype_ok(tb->scale_dtype) || T > INT32_MAX ||
      (int64_t)n_cols * tb->head_dim > INT32_MAX - 256)
    return ENGRAM_ERR_UNSUPPORTED;
  return ENGRAM_OK;
}
}  // namespace

uint64_t engram_lookup_project_workspace(int64_t T, int32_t n_cols, int32_t head_dim) {
  if (T <= 0 || n_cols <= 0 || head_dim <= 0) return 0;
  return lookup_rows_bytes(T, n_cols, head_dim) + lookup_counter_bytes(T);
}

int engram_lookup_project(const int64_t* idx, int64_t idx_stride, int64_t T, int32_t n_cols,
                          const engram_table* table, const uint16_t* wkv, int32_t N, void* workspace,
                          uint64_t workspace_bytes, uint16_t* out, engram_stream_t stream) {
  if (T < 0) return ENGRAM_ERR_INVALID;
  int rc = lookup_ahead_shape(T, n_cols, table);
  if (rc != ENGRAM_OK) return rc;
  if (N < 8 || N % 8 != 0 || N > INT32_MAX - 256) return ENGRAM_ERR_UNSUPPORTED;
  if (T == 0) return ENGRAM_OK;
  engram::LookupArgs la;
  rc = lookup_ahead_args(idx, idx_stride, n_cols, table, workspace, &la);
  if (rc != ENGRAM_OK) return rc;
  if (wkv == nullptr || out == nullptr || !aligned(wkv, 16) || !aligned(out, 16)) return ENGRAM_ERR_INVALID;
  if (workspace_bytes < engram_lookup_project_workspace(T, n_cols, table->head_dim)) return ENGRAM_ERR_INVALID;
  la.counters = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(workspace) +
                                                lookup_rows_bytes(T, n_cols, table->head_dim));
  return launched(launch_rc(engram::launch_lookup_project(la, wkv, T, N, out, (cudaStream_t)stream)),
                  (cudaStream_t)stream, {span(out, (uint64_t)T * N * 2), span(workspace, workspace_bytes)});
}

uint64_t engram_lookup_project_gate_workspace(int64_t T, int32_t n_cols, int32_t head_dim, int32_t hc, int32_t dim) {
  const uint64_t rows = engram_lookup_project_workspace(T, n_cols, head_dim);
  const uint64_t gate = engram_project_gate_workspace(T, hc, dim);
  return rows == 0 || gate == 0 ? 0 : rows + gate;
}

int engram_lookup_project_gate(const uint16_t* x, const int64_t* idx, int64_t idx_stride, int64_t T, int32_t n_cols,
                               const engram_table* table, const uint16_t* wkv, const uint16_t* q_weight,
                               const uint16_t* k_weight, const uint8_t* mask, int32_t hc, int32_t dim, float eps,
                               void* workspace, uint64_t workspace_bytes, uint16_t* out, engram_stream_t stream) {
  if (T < 0) return ENGRAM_ERR_INVALID;
  int rc = lookup_ahead_shape(T, n_cols, table);
  if (rc != ENGRAM_OK) return rc;
  if (!gate_shape_ok(hc, dim)) return ENGRAM_ERR_UNSUPPORTED;
  if (T == 0) return ENGRAM_OK;
  engram::LookupArgs la;
  rc = lookup_ahead_args(idx, idx_stride, n_cols, table, workspace, &la);
  if (rc != ENGRAM_OK) return rc;
  if (x == nullptr || wkv == nullptr || q_weight == nullptr || k_weight == nullptr || out == nullptr)
    return ENGRAM_ERR_INVALID;
  if (!aligned(x, 16) || !aligned(wkv, 16) || !aligned(q_weight, 16) || !aligned(k_weight, 16) || !aligned(out, 16))
    return ENGRAM_ERR_INVALID;
  if (workspace_bytes < engram_lookup_project_gate_workspace(T, n_cols, table->head_dim, hc, dim))
    return ENGRAM_ERR_INVALID;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const uint64_t rows_bytes = lookup_rows_bytes(T, n_cols, table->head_dim);
  la.counters = reinterpret_cast<unsigned int*>(ws + rows_bytes);
  uint8_t* gate_ws = ws + rows_bytes + lookup_counter_bytes(T);
  uint16_t* value = reinterpret_cast<uint16_t*>(gate_ws);
  float* part = reinterpret_cast<float*>(gate_ws + round256((uint64_t)T * dim * 2u));
  cudaStream_t s = (cudaStream_t)stream;
  rc = launch_rc(engram::launch_lookup_project_gate_sums(x, la, wkv, q_weight, k_weight, T, hc, dim, value, part, s));
  if (rc != ENGRAM_OK) return launched(rc, s, {});
  return launched(launch_rc(engram::launch_gate_finish(x, value, part, mask, T, hc, dim, eps, out, s)), s,
                  {span(out, (uint64_t)T * hc * dim * 2), span(workspace, workspace_bytes)});
}

int engram_device_status(engram_stream_t stream, uint32_t* flags, int clear) {
  if (flags == nullptr) return ENGRAM_ERR_INVALID;
  unsigned int v = 0;
  int rc = launched(launch_rc(engram::device_status_take(&v, clear ? 1 : 0, (cudaStream_t)stream)),
                    (cudaStream_t)stream, {});
  if (rc != ENGRAM_OK) return rc;
  *flags = v;
  return ENGRAM_OK;
}

uint64_t engram_shard_pack_workspace(int64_t n, int32_t world) {
  if (n <= 0 || world < 1 || world > ENGRAM_MAX_SHARDS) return 0;
  return round256((uint64_t)engram::shard_pack_segments(n) * (uint64_t)(world + 1) * sizeof(int32_t));
}

int engram_shard_pack(const int64_t* idx, int64_t n, int64_t rows, int32_t world, int64_t* counts,
                      int64_t* local_rows, int64_t* positions, void* workspace, uint64_t workspace_bytes,
                      engram_stream_t stream) {
  if (n < 0 || rows < 0) return ENGRAM_ERR_INVALID;
  if (world < 1 || world > ENGRAM_MAX_SHARDS) return ENGRAM_ERR_UNSUPPORTED;
  if (n == 0) return ENGRAM_OK;
  if (n > INT32_MAX) return ENGRAM_ERR_UNSUPPORTED;  // bucket offsets are int32
  if (idx == nullptr || counts == nullptr || local_rows == nullptr || positions == nullptr || workspace == nullptr)
    return ENGRAM_ERR_INVALID;
  if (!aligned(idx, 8) || !aligned(counts, 8) || !aligned(local_rows, 8) || !aligned(positions, 8) ||
      !aligned(workspace, 16))
    return ENGRAM_ERR_INVALID;
  if (workspace_bytes < engram_shard_pack_workspace(n, world)) return ENGRAM_ERR_INVALID;
  return launched(launch_rc(engram::launch_shard_pack(idx, n, rows, world, counts, local_rows, positions,
                                                      static_cast<int32_t*>(workspace), (cudaStream_t)stream)),
                  (cudaStream_t)stream,
                  {span(counts, (uint64_t)(world + 1) * 8), span(local_rows, (uint64_t)n * 8),
                   span(positions, (uint64_t)n * 8), span(workspace, workspace_bytes)});
}

int engram_shard_pack_static(const int64_t* idx, int64_t n, int64_t rows, int32_t world, int64_t* counts,
                             int64_t* local_rows, int64_t* positions, engram_stream_t stream) {
  if (n < 0 || rows < 0) return ENGRAM_ERR_INVALID;
  if (world < 1 || world > ENGRAM_MAX_SHARDS) return ENGRAM_ERR_UNSUPPORTED;
  if (n == 0) return ENGRAM_OK;
  if (n > engram::static_pack_max_n(world)) return ENGRAM_ERR_UNSUPPORTED;  // beyond the fixed scratch
  if (idx == nullptr || counts == nullptr || local_rows == nullptr || positions == nullptr) return ENGRAM_ERR_INVALID;
  if (!aligned(idx, 8) || !aligned(counts, 8) || !aligned(local_rows, 8) || !aligned(positions, 8))
    return ENGRAM_ERR_INVALID;
  int32_t* scratch = nullptr;
  int rc = launch_rc(engram::static_pack_scratch(&scratch));
  if (rc != ENGRAM_OK) return rc;
  return launched(
      launch_rc(engram::launch_shard_pack(idx, n, rows, world, counts, local_rows, positions, scratch,
                                          (cudaStream_t)stream)),
      (cudaStream_t)stream,
      {span(counts, (uint64_t)(world + 1) * 8), span(local_rows, (uint64_t)n * 8), span(positions, (uint64_t)n * 8)});
}

int engram_shard_unpack(const uint16_t* rows, const int64_t* positions, int64_t m, int64_t n, int32_t head_dim,
                        uint16_t* out, engram_stream_t stream) {
  if (n < 0 || m < 0 || m > n) return ENGRAM_ERR_INVALID;
  if (head_dim < 8 || head_dim % 8 != 0 || head_dim > 65536) return ENGRAM_ERR_UNSUPPORTED;
  if (n == 0) return ENGRAM_OK;
  if (positions == nullptr || out == nullptr || (m > 0 && rows == nullptr)) return ENGRAM_ERR_INVALID;
  if (!aligned(positions, 8) || !aligned(out, 16) || (m > 0 && !aligned(rows, 16))) return ENGRAM_ERR_INVALID;
  if (n > ((int64_t)1 << 40)) return ENGRAM_ERR_UNSUPPORTED;
  return launched(launch_rc(engram::launch_shard_unpack(rows, positions, m, n, head_dim, out, (cudaStream_t)stream)),
                  (cudaStream_t)stream, {span(out, (uint64_t)n * head_dim * 2)});
}

int engram_set_l2_fetch_granularity(int32_t bytes, int32_t* previous) {
  if (bytes != 0 && bytes != 32 && bytes != 64 && bytes != 128) return ENGRAM_ERR_INVALID;
  size_t old = 0;
  if (cudaDeviceGetLimit(&old, cudaLimitMaxL2FetchGranularity) != cudaSuccess ||
      cudaDeviceSetLimit(cudaLimitMaxL2FetchGranularity, (size_t)bytes) != cudaSuccess) {
    cudaGetLastError();
    return ENGRAM_ERR_CUDA;
  }
  if (previous != nullptr) *previous = (int32_t)old;
  return ENGRAM_OK;
}

int engram_state_layout(const engram_state* state, engram_layout* layout) {
  if (state == nullptr || layout == nullptr) return ENGRAM_ERR_INVALID;
  *layout = state->lay;
  return ENGRAM_OK;
}

const char* engram_strerror(int code) {
  switch (code) {
    case ENGRAM_OK: return "ok";
    case ENGRAM_ERR_INVALID: return "invalid argument (null or misaligned pointer, negative size, bad layout value)";
    case ENGRAM_ERR_RANGE: return "out of range (B > max_batch or L > max_seq_len)";
    case ENGRAM_ERR_CUDA: return "CUDA runtime or launch error";
    case ENGRAM_ERR_NOMEM: return "device allocation failed";
    case ENGRAM_ERR_UNSUPPORTED:
      return "beyond the library limits (head_dim, block, scale type, layers, n-gram size)";
    default: return "unknown error code";
  }
}

}  // extern "C"
