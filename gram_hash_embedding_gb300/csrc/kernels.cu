// Kernels of libengram (sm_103a): the n-gram hash, the fp8 row lookup, and both fused.
//
// Method ("DeepSeek V4.1" pages):
//   blocks/stack-hashes page, n-gram hash `forward`: compress, mask, cache, lookback with
//     cumulative blocking, multiply, rolling XOR, floored mod by primes, + offsets.
//   engram-first/lookup page, `ParallelEngramEmbedding.forward`: fp8 row + block-scale gather
//     (the scale, stored as fp32, bf16, UE8M0 or E4M3, widened to fp32), one fp32 multiply,
//     round-to-nearest-even to bf16, +0 for out-of-range rows.
//
// Design (GB300): the path is HBM-bound (random 128-B row reads, streaming bf16 writes, ~99.9%
// of its bytes); there is no dense contraction, so no tensor cores. A CTA owns a tile of
// consecutive tokens of one sequence: it stages the tile's compressed tokens plus the
// (max_ngram-1)-token halo in shared memory, computes every hash id of the tile there, and then
// all its threads stream the tile's rows through registers, several rows in flight per thread.
// For one layer the tile's output rows are contiguous: lane q of a row's D/16-lane group loads codes
// [16q, 16q+16) with one 16-byte load and writes their 32 bf16 bytes, one whole sector, with one
// 256-bit store, so a warp moves 4 rows per load and per store instruction.
//
// DRAM per row: 128 B of codes, the sector holding its scale (32 B with the context's L2 fetch
// limit at 32 B, engram_set_l2_fetch_granularity; a 128-B line at the 64-B default) and the 256-B
// bf16 write: 416 (512) DRAM bytes for 388 algorithmic bytes. A variant that landed rows and scales
// in shared memory with bulk copies (TMA engine) and per-warp mbarrier pipelines was measured slower
// at every shape tried (its shared-memory slots cap the SM at ~1000 rows in flight and leave 8-16
// warps to convert), so the register path is the one kept.
#include <cstdint>

#include "dequant.cuh"
#include "engram_internal.cuh"

namespace engram {
namespace {

// Launch shapes (compile-time; each default is the value measured fastest on a GB300).
#ifndef ENGRAM_THREADS
#define ENGRAM_THREADS 256
#endif
#ifndef ENGRAM_UNROLL
#define ENGRAM_UNROLL 4
#endif
#ifndef ENGRAM_MIN_BLOCKS
#define ENGRAM_MIN_BLOCKS 4
#endif
#ifndef ENGRAM_FUSED_TILE
#define ENGRAM_FUSED_TILE 8
#endif
#ifndef ENGRAM_TARGET_CTAS
#define ENGRAM_TARGET_CTAS 608
#endif
#ifndef ENGRAM_HASH_TILE
#define ENGRAM_HASH_TILE 32
#endif
#ifndef ENGRAM_HASH_THREADS
#define ENGRAM_HASH_THREADS 96
#endif

constexpr int kThreads = ENGRAM_THREADS;           // threads per CTA, fused and lookup kernels
constexpr int kUnroll = ENGRAM_UNROLL;             // independent row pieces in flight per thread
constexpr int kMinBlocks = ENGRAM_MIN_BLOCKS;      // fused kernel: 4 CTAs per SM, i.e. <= 64 registers
constexpr int kFusedTile = ENGRAM_FUSED_TILE;      // largest tile (tokens per CTA) of the fused kernel: 8-token
                                                   // tiles beat 16 at full scale (more, shorter CTAs keep more
                                                   // row loads in flight; the hash phase is the same per token)
constexpr int kMinFusedTile = 4;                   // below 4 tokens the halo and hash phase dominate
constexpr int kTargetCtas = ENGRAM_TARGET_CTAS;    // fused grid size the tile choice aims for (one wave at 4 CTAs
                                                   // per SM; consecutive launches overlap, so fewer, fuller CTAs
                                                   // win: an 8K-token chunk takes 33.6 us at 8-token tiles against
                                                   // 36.8 us at 4-token tiles aiming for 1216 CTAs, same box)
constexpr int kHashTile = ENGRAM_HASH_TILE;        // tokens per CTA, hash-only kernel
constexpr int kHashThreads = ENGRAM_HASH_THREADS;  // threads per CTA, hash-only kernel (<= kThreads); 96 keeps
                                                   // every thread busy in step 3 at 48 columns (2 tokens a pass)

// Checked builds (-DENGRAM_CHECKED=1, a debugging aid in place of a memory checker): the hash and
// fused kernels test every global access against the call's sizes before making it; an access
// outside them is skipped and raises ENGRAM_STATUS_CHECK. Release builds compile the tests away.
#ifndef ENGRAM_CHECKED
#define ENGRAM_CHECKED 0
#endif

__device__ __forceinline__ bool in_bounds(bool ok, unsigned int* flags_s) {
  if (!ENGRAM_CHECKED || ok) return true;
  atomicOr(flags_s, ENGRAM_STATUS_CHECK);
  return false;
}

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

// bf16 output rows are written once and not read again by this kernel: an L2 evict-first policy
// lets them leave L2 ahead of lines still in use (254.7 vs 257.0 us per full-scale launch). A lane
// writes its 32 bytes with one 256-bit store (a whole sector) when the output is 32-byte aligned,
// else with two 16-byte stores.
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t policy;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
  return policy;
}

__device__ __forceinline__ void st_out_v4(void* p, uint4 v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w), "l"(policy)
               : "memory");
}

__device__ __forceinline__ void st_out_v8(void* p, uint4 a, uint4 b, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8}, %9;" ::"l"(p), "r"(a.x),
               "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w), "l"(policy)
               : "memory");
}

__host__ __device__ constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x >> 1); }

// One lane's share of one output row: codes [16q, 16q+8) and [16q+8, 16q+16) of table row `row`.
struct RowPiece {
  uint2 v0, v1;
  uint32_t s0, s1;  // raw scale bits (widened when the piece is stored)
  bool valid;
};

// D (head_dim) is a compile-time power of two, so row offsets are shifts; the scale block is a
// power of two too (it divides D), passed as its log2. ONE: the row has a single scale (block >= D),
// so both halves share one scale load. SDT: the scales' storage type (ENGRAM_SCALE_*).
template <int D, bool ONE, int SDT>
__device__ __forceinline__ void piece_load(RowPiece& pc, const uint8_t* W, const void* S, int64_t rows, int64_t row,
                                           int q, int blk_shift) {
  pc.valid = (row >= 0) && (row < rows);
  if (pc.valid) {
    const uint8_t* base = W + (row << ilog2(D));
    const int k0 = 16 * q, k1 = 16 * q + 8;
    const uint4 w = ld_rows_v4(base + k0);  // one 16-byte load: a row's D/16 lanes fetch it in one request
    pc.v0 = make_uint2(w.x, w.y);
    pc.v1 = make_uint2(w.z, w.w);
    const int64_t srow = row << (ilog2(D) - blk_shift);
    pc.s0 = ld_scale_bits<SDT>(S, srow + (k0 >> blk_shift));
    pc.s1 = ONE ? pc.s0 : ld_scale_bits<SDT>(S, srow + (k1 >> blk_shift));
  }
}

// out_row: bf16 row of D values (2*D bytes)
template <int D, int SDT>
__device__ __forceinline__ void piece_store(const RowPiece& pc, uint16_t* out_row, int q) {
  uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a;  // masked rows are +0
  if (pc.valid) {
    a = dequant8(pc.v0, widen_scale<SDT>(pc.s0));
    b = dequant8(pc.v1, widen_scale<SDT>(pc.s1));
  }
  const uint64_t policy = evict_first_policy();
  uint16_t* p = out_row + 16 * q;  // 32 bytes: a whole sector when the output is 32-byte aligned
  if ((reinterpret_cast<uintptr_t>(p) & 31) == 0) {
    st_out_v8(p, a, b, policy);
  } else {
    st_out_v4(p, a, policy);
    st_out_v4(p + 8, b, policy);
  }
}

// ------------------------------------------------------------------------------------------------
// shared-memory plan of the hash phase (all kernels that hash a token tile)

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

// The per-column constants and the multipliers into shared memory (every thread of the CTA). They
// are written once, when the state is created, so this may run before pdl_wait().
__device__ __forceinline__ void stage_constants(const StateView& sv, unsigned char* smem, const SmemPlan& plan) {
  ColParam* cols_s = reinterpret_cast<ColParam*>(smem + plan.cols_off);
  uint64_t* mult_s = reinterpret_cast<uint64_t*>(smem + plan.mult_off);
  for (int i = threadIdx.x; i < sv.n_layers * sv.n_cols; i += blockDim.x) cols_s[i] = sv.cols[i];
  for (int i = threadIdx.x; i < sv.n_layers * sv.max_ngram; i += blockDim.x) mult_s[i] = sv.mult[i];
}

// Step 3 for one column: the thread's tokens t1, t1 + tstep, ... and running indices into the rolling
// values (ri), the int64 hash output (hi) and the tile's row ids (xi). The options of the call are
// template parameters, so the loop body tests nothing per token; it is 22% faster than one loop that
// tested them and recomputed the indices per token (12.8 vs 10.0 us per 65,536-token hash launch).
struct ModWalk {
  int ri, rstep;
  int64_t hi, hstep;
  int xi, xstep;
};

template <bool HASHES, bool ROWIDX>
__device__ __forceinline__ void mod_column(const uint64_t* roll_s, const ColParam cp, ModWalk w, int64_t* hashes,
                                           int64_t* rowidx_s, const int t1, const int ntok, const int tstep,
                                           const int64_t tok0, const int64_t total, unsigned int* flags_s) {
#pragma unroll 4
  for (int t = t1; t < ntok; t += tstep) {
    const int64_t h = floored_mod(roll_s[w.ri], cp) + cp.offset;
    if (HASHES && in_bounds(tok0 + t < total, flags_s)) hashes[w.hi] = h;
    if (ROWIDX) rowidx_s[w.xi] = h;
    w.ri += w.rstep;
    w.hi += w.hstep;
    w.xi += w.xstep;
  }
}

// ------------------------------------------------------------------------------------------------
// hash phase of one tile: `ntok` consecutive tokens starting at t0 of sequence b, whose Lb tokens
// start at element seq_off of ids / mask / hashes and use cache row b (or cache_rows[b]). Called by
// every thread of the CTA (contains barriers). Fills rowidx (layer-major: [l][t][col]) when given,
// and the optional int64 hash output. Returns whether the sequence's cache row and start position
// fit the cache. With `defer` it writes no global memory (no cache write, no hash output; rowidx is
// filled): the caller writes them after pdl_wait() (write_deferred).
__device__ __forceinline__ bool hash_tile(const StateView& sv, const CallArgs& a, unsigned char* smem,
                                          const SmemPlan& plan, const int tile, const int b, const int64_t seq_off,
                                          const int64_t Lb, const int64_t t0, const int ntok, const bool want_rowidx,
                                          const bool staged, unsigned int* flags_s, const bool defer = false) {
  const int N = sv.max_ngram, NL = sv.n_layers, C = sv.n_cols, H = sv.n_heads;
  const int NC = NL * C;
  ColParam* cols_s = reinterpret_cast<ColParam*>(smem + plan.cols_off);
  uint64_t* mult_s = reinterpret_cast<uint64_t*>(smem + plan.mult_off);
  uint64_t* roll_s = reinterpret_cast<uint64_t*>(smem + plan.roll_off);
  int64_t* rowidx_s = reinterpret_cast<int64_t*>(smem + plan.rowidx_off);
  int32_t* tok_s = reinterpret_cast<int32_t*>(smem + plan.tok_off);
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int64_t s_b = (int64_t)a.start_pos[b];
  const int64_t r_b = a.cache_rows != nullptr ? (int64_t)a.cache_rows[b] : (int64_t)b;
  const bool slot_ok = (r_b >= 0) && (r_b < sv.max_batch);
  const bool row_ok = slot_ok && (s_b >= 0) && (s_b <= sv.max_seq_len - Lb);
  const int32_t dead = sv.dead;
  int32_t* cache_row = sv.cache + (slot_ok ? r_b : 0) * sv.max_seq_len;  // dereferenced only when row_ok

  if (tid == 0 && !row_ok) atomicOr(flags_s, slot_ok ? ENGRAM_STATUS_BAD_START : ENGRAM_STATUS_BAD_ROW);
  if (!staged) stage_constants(sv, smem, plan);

  // 1. compressed tokens of the tile and its halo: tok_s[j] holds position t0 - (N-1) + j.
  //    In-chunk tokens come from ids (token_map, mask) and do not wait for the start position;
  //    earlier positions come from the cache, which this launch never writes below start_pos, so
  //    reads and writes are disjoint.
  for (int j = tid; j < ntok + N - 1; j += nthr) {
    const int64_t t = t0 - (N - 1) + j;
    int32_t c = dead;
    if (t >= 0) {
      if (in_bounds(seq_off + t >= 0 && seq_off + t < a.total, flags_s)) {
        const int64_t id = a.ids[seq_off + t];
        if (id < 0 || id >= sv.raw_vocab) {
          if (row_ok) atomicOr(flags_s, ENGRAM_STATUS_BAD_ID);
        } else {
          c = sv.token_map[id];
        }
        if (a.mask != nullptr && a.mask[seq_off + t] == 0) c = dead;
      }
    } else if (row_ok) {
      const int64_t p = s_b + t;
      if (p >= 0 && in_bounds(p < sv.max_seq_len && r_b >= 0 && r_b < sv.max_batch, flags_s)) c = cache_row[p];
    }
    tok_s[j] = c;
  }
  __syncthreads();

  // 2. cache write, lookback with cumulative blocking, products and rolling XOR per layer
  if (row_ok) {
    for (int t = tid; t < ntok; t += nthr) {
      const int32_t cur = tok_s[t + N - 1];
      const int64_t pos = s_b + t0 + t;
      if (!defer && in_bounds(pos >= 0 && pos < sv.max_seq_len, flags_s)) cache_row[pos] = cur;
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

  // 3. hash ids: floored mod by the column's prime plus its offset. Thread -> (column j, token t)
  //    with j fixed per thread, so consecutive threads write consecutive int64 of the optional
  //    [B, L, layer, column] output; rowidx is compact and layer-major ([l][t][col]), i.e. in the
  //    order of each layer's contiguous output rows.
  if (NC <= nthr) {
    const int j = tid % NC;
    const int tstep = nthr / NC;
    if (tid < tstep * NC) {
      const int l = j / C;
      const int col = j - l * C;
      const int t1 = tid / NC;
      const ModWalk w{(t1 * NL + l) * (N - 1) + col / H, tstep * NL * (N - 1), (seq_off + t0 + t1) * NC + j,
                      (int64_t)tstep * NC, (l * ntok + t1) * C + col, tstep * C};
      const bool out_h = a.hashes != nullptr && !defer;
      if (!row_ok) {  // the row wrote nothing: its hash ids are -1
        ModWalk v = w;
        for (int t = t1; t < ntok; t += tstep, v.hi += v.hstep, v.xi += v.xstep) {
          if (out_h && in_bounds(seq_off + t0 + t < a.total, flags_s)) a.hashes[v.hi] = -1;
          if (want_rowidx) rowidx_s[v.xi] = -1;
        }
      } else if (!want_rowidx) {
        mod_column<true, false>(roll_s, cols_s[j], w, a.hashes, rowidx_s, t1, ntok, tstep, seq_off + t0, a.total, flags_s);
      } else if (!out_h) {
        mod_column<false, true>(roll_s, cols_s[j], w, a.hashes, rowidx_s, t1, ntok, tstep, seq_off + t0, a.total, flags_s);
      } else {
        mod_column<true, true>(roll_s, cols_s[j], w, a.hashes, rowidx_s, t1, ntok, tstep, seq_off + t0, a.total, flags_s);
      }
    }
  } else {
    for (int e = tid; e < ntok * NC; e += nthr) {
      const int t = e / NC;
      const int j = e - t * NC;
      const int l = j / C;
      const int col = j - l * C;
      int64_t h = -1;
      if (row_ok) {
        const ColParam cp = cols_s[j];
        h = floored_mod(roll_s[(t * NL + l) * (N - 1) + col / H], cp) + cp.offset;
      }
      if (a.hashes != nullptr && !defer && in_bounds(seq_off + t0 + t < a.total, flags_s))
        a.hashes[(seq_off + t0 + t) * NC + j] = h;
      if (want_rowidx) rowidx_s[(l * ntok + t) * C + col] = h;
    }
  }
  return row_ok;
}

// ------------------------------------------------------------------------------------------------
// packed calls: which tile of which sequence a CTA takes

__device__ __forceinline__ int64_t floor_div(int64_t x, int64_t d) {
  const int64_t q = x / d;
  return (x % d != 0 && x < 0) ? q - 1 : q;
}

// An extent the kernels can run: inside [0, T] and at most max_len (a.L) tokens long.
__device__ __forceinline__ bool extent_ok(const CallArgs& a, int64_t start, int64_t end) {
  return start >= 0 && end <= a.total && end >= start && end - start <= a.L;
}

// CTA k of a packed launch (a 1-D grid of floor(T / tile) + B CTAs) takes tile j = k - Q(b) of the
// last sequence b with Q(b) <= k, where Q(b) = floor(cu_seqlens[b] / tile) + b. For non-decreasing
// cu_seqlens, Q increases strictly and Q(b+1) - Q(b) >= floor(L_b / tile) + 1 >= ceil(L_b / tile), so
// every tile of every sequence gets its own CTA and at most one CTA per sequence finds no tokens (a
// grid sized by the longest sequence left most CTAs of a decode-heavy batch empty). The search samples
// Q at up to blockDim.x points per round: one round up to blockDim.x sequences, two up to its square.
// CTA k < B also checks the extent of sequence k and raises ENGRAM_STATUS_BAD_LENGTH if it is
// inconsistent, so every such sequence is flagged whether or not a CTA lands on it. Called by all
// threads of the CTA; the result is the same in every thread. False: nothing to do.
__device__ bool packed_tile(const StateView& sv, const CallArgs& a, const int tile, int& b, int64_t& seq_off,
                            int64_t& Lb, int64_t& t0) {
  __shared__ int32_t cu_s[kThreads];  // the last round's samples: the extents of the candidates
  const int64_t k = blockIdx.x;
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int32_t* cu = a.cu_seqlens;
  if (tid == 0 && k < a.B && !extent_ok(a, cu[k], cu[k + 1])) atomicOr(sv.status, ENGRAM_STATUS_BAD_LENGTH);
  int64_t lo = 0, n = a.B, end;  // candidates lo .. lo + n - 1 (lo + n <= B throughout)
  for (;;) {
    const int64_t step = (n + nthr - 1) / nthr;
    bool le = false;
    if (tid * step < n) {
      const int64_t i = lo + tid * step;
      const int32_t v = cu[i];
      le = floor_div(v, tile) + i <= k;
      if (step == 1) cu_s[tid] = v;
    } else if (step == 1 && tid == n) {
      cu_s[tid] = cu[lo + n];  // the end of the last candidate
    }
    const int c = __syncthreads_count(le);  // the samples with Q <= k are a prefix when Q increases
    if (c == 0) return false;
    if (step == 1) {  // every candidate was sampled: b is the last one with Q <= k
      b = (int)(lo + c - 1);
      seq_off = cu_s[c - 1];
      end = c < nthr ? cu_s[c] : cu[b + 1];
      break;
    }
    lo += (int64_t)(c - 1) * step;
    n = min(step, n - (int64_t)(c - 1) * step);
  }
  if (!extent_ok(a, seq_off, end)) return false;  // flagged by CTA b
  Lb = end - seq_off;
  const int64_t j = k - (floor_div(seq_off, tile) + b);
  t0 = j * tile;
  return j >= 0 && t0 < Lb;
}

// ------------------------------------------------------------------------------------------------
// fused kernel: hash a tile, then (GATHER) stream its rows through registers.
// Dense calls: grid = (ceil(L / tile), B), one CTA = `tile` consecutive tokens of sequence b. Packed
// calls: a 1-D grid of floor(T / tile) + B CTAs mapped to (sequence, tile) pairs by packed_tile.
// D = head_dim (compile time); G = D / 16 lanes per output row. Unused when GATHER is false.
// The cache writes and hash-id stores of a tile whose hash phase ran with `defer` (before pdl_wait()):
// the tokens are still in tok_s and the hash ids in rowidx_s.
__device__ __forceinline__ void write_deferred(const StateView& sv, const CallArgs& a, const unsigned char* smem,
                                               const SmemPlan& plan, const int b, const int64_t seq_off,
                                               const int64_t t0, const int ntok, const bool row_ok,
                                               unsigned int* flags_s) {
  const int N = sv.max_ngram, C = sv.n_cols, NC = sv.n_layers * sv.n_cols;
  const int32_t* tok_s = reinterpret_cast<const int32_t*>(smem + plan.tok_off);
  const int64_t* rowidx_s = reinterpret_cast<const int64_t*>(smem + plan.rowidx_off);
  if (row_ok) {
    const int64_t s_b = (int64_t)a.start_pos[b];
    const int64_t r_b = a.cache_rows != nullptr ? (int64_t)a.cache_rows[b] : (int64_t)b;
    int32_t* cache_row = sv.cache + r_b * sv.max_seq_len;
    for (int t = threadIdx.x; t < ntok; t += blockDim.x) {
      const int64_t pos = s_b + t0 + t;
      if (in_bounds(pos >= 0 && pos < sv.max_seq_len, flags_s)) cache_row[pos] = tok_s[t + N - 1];
    }
  }
  if (a.hashes != nullptr) {  // rowidx holds the hash ids (-1 for a rejected row) layer-major
    for (int e = threadIdx.x; e < ntok * NC; e += blockDim.x) {
      const int t = e / NC;
      const int j = e - t * NC;
      const int l = j / C;
      if (in_bounds(seq_off + t0 + t < a.total, flags_s))
        a.hashes[(seq_off + t0 + t) * NC + j] = rowidx_s[(l * ntok + t) * C + (j - l * C)];
    }
  }
}

// ------------------------------------------------------------------------------------------------
// fused kernel: hash a tile, then (GATHER) stream its rows through registers.
// Dense calls: grid = (ceil(L / tile), B), one CTA = `tile` consecutive tokens of sequence b. Packed
// calls: a 1-D grid of floor(T / tile) + B CTAs mapped to (sequence, tile) pairs by packed_tile.
// D = head_dim (compile time); G = D / 16 lanes per output row. Unused when GATHER is false.
//
// Early reads (dense fused calls with a.early set): a launch overlaps the drain of the kernel before
// it only as far as it reads nothing that kernel writes. The host sets a.early when this library's
// previous launch on the stream writes none of the call's inputs (any other kind of producer is waited
// for in full by the launch itself), so a CTA may then read ids, mask, start positions and the tables
// before pdl_wait(): it hashes its tile and issues its first batch of row loads, and waits only before
// its first store. A tile whose lookback reaches below the chunk (t0 < max_ngram - 1) reads the cache,
// which the previous kernel may write, so it waits before hashing. Cache writes and hash-id stores are
// deferred until after the wait. Every CTA waits before it exits and triggers the next launch only
// after its wait, so a later kernel can never run ahead of a kernel two launches back.
template <bool GATHER, int D, bool ONE, int SDT>
__global__ void __launch_bounds__(kThreads, kMinBlocks) hash_kernel(const StateView sv, const CallArgs a, const int tile) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ unsigned int flags_s;
  const int NL = sv.n_layers, C = sv.n_cols;
  const SmemPlan plan = smem_plan(NL, sv.max_ngram, C, tile, GATHER);
  // dense calls: every CTA has tokens, so it stages the state's constants while the previous kernel
  // drains; packed calls learn their extents first (CTAs without tokens exit at once)
  const bool dense = a.cu_seqlens == nullptr;
  if (dense) stage_constants(sv, smem, plan);
  const bool early = GATHER && dense && a.early != 0;
  bool waited = false;
  auto wait_once = [&]() {
    if (!waited) {
      pdl_wait();
      pdl_trigger();
      waited = true;
    }
  };
  if (!early) wait_once();
  const int64_t* rowidx_s = reinterpret_cast<const int64_t*>(smem + plan.rowidx_off);
  const int tid = threadIdx.x;
  int b;
  int64_t seq_off, Lb, t0;
  if (a.cu_seqlens != nullptr) {
    if (!packed_tile(sv, a, tile, b, seq_off, Lb, t0)) return;
  } else {
    b = blockIdx.y;
    seq_off = (int64_t)b * a.L;
    Lb = a.L;
    t0 = (int64_t)blockIdx.x * tile;
  }
  if (t0 >= Lb) {
    wait_once();
    return;
  }
  const int ntok = (int)min((int64_t)tile, Lb - t0);
  if (tid == 0) flags_s = 0u;
  if (early && t0 < sv.max_ngram - 1) wait_once();  // the lookback reads the cache below this chunk
  const bool defer = !waited;
  __syncthreads();
  const bool row_ok = hash_tile(sv, a, smem, plan, tile, b, seq_off, Lb, t0, ntok, GATHER, dense, &flags_s, defer);

  if (GATHER) {
    __syncthreads();
    // 4. gather + dequant. Units run over all layers at once (so a short tile, e.g. one decode
    //    token, issues every layer's row loads in one batch); within a layer the tile's ntok*C rows
    //    are contiguous in its output and in rowidx, so unit u = (row u/G, piece u%G) needs only
    //    shifts, and its layer is found by comparison.
    constexpr int G = D / 16;
    const int blk_shift = __ffs(a.block) - 1;
    const int rpl = ntok * C;
    const int upl = rpl * G;  // units per layer
    const int units = NL * upl;
    const int64_t out_base_row = (seq_off + t0) * C;
    for (int base = tid; base < units; base += kThreads * kUnroll) {
      RowPiece pc[kUnroll];
      uint16_t* orow[kUnroll];
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        int u = base + k * kThreads;
        orow[k] = nullptr;
        if (u < units) {
          int l = 0;
          while (u >= upl) {
            u -= upl;
            ++l;
          }
          const int r = u / G;
          if (!in_bounds(out_base_row + r < a.total * C, &flags_s)) continue;
          orow[k] = a.out[l] + (out_base_row + r) * D;
          piece_load<D, ONE, SDT>(pc[k], a.W[l], a.S[l], a.rows[l], rowidx_s[l * rpl + r], u % G, blk_shift);
        }
      }
      wait_once();  // the outputs may be the previous kernel's: no store before it has completed
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        const int u = base + k * kThreads;
        if (orow[k] != nullptr) piece_store<D, SDT>(pc[k], orow[k], u % G);
      }
    }
  }
  wait_once();
  if (defer) write_deferred(sv, a, smem, plan, b, seq_off, t0, ntok, row_ok, &flags_s);

  __syncthreads();
  if (tid == 0 && flags_s != 0u) atomicOr(sv.status, flags_s);
}

// ------------------------------------------------------------------------------------------------
// standalone lookup: grid-stride over (index, lane) units

template <int D, bool ONE, int SDT>
__global__ void __launch_bounds__(kThreads) lookup_kernel(const int64_t* __restrict__ idx, const int64_t n_idx,
                                                          const uint8_t* __restrict__ W,
                                                          const void* __restrict__ S, const int64_t rows,
                                                          const int blk_shift, uint16_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  constexpr int G = D / 16;
  const int64_t units = n_idx * G;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  const int64_t first = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  // the row ids of a batch are loaded before any of its rows (and the next batch's while this one's
  // rows are in flight): loading each id next to its row made every row wait for its own id
  // (144.2 vs 132.1 us per 1.57M-row launch with the grid below)
  int64_t next_row[kUnroll];
#pragma unroll
  for (int k = 0; k < kUnroll; ++k) {
    const int64_t u = first + k * stride;
    next_row[k] = u < units ? __ldg(idx + u / G) : -1;
  }
  for (int64_t base = first; base < units; base += stride * kUnroll) {
    RowPiece pc[kUnroll];
    int64_t row[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      row[k] = next_row[k];
      const int64_t u = base + (kUnroll + k) * stride;
      next_row[k] = u < units ? __ldg(idx + u / G) : -1;
    }
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const int64_t u = base + k * stride;
      if (u < units) piece_load<D, ONE, SDT>(pc[k], W, S, rows, row[k], (int)(u % G), blk_shift);
    }
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const int64_t u = base + k * stride;
      if (u < units) piece_store<D, SDT>(pc[k], out + (u / G) * D, (int)(u % G));
    }
  }
}

__global__ void fill_i32_kernel(int32_t* p, int64_t n, int32_t v) {
  pdl_wait();
  pdl_trigger();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) p[i] = v;
}

template <bool GATHER, int D, bool ONE, int SDT>
cudaError_t launch_hash_k(const StateView& sv, const CallArgs& a, int tile, cudaStream_t s) {
  const SmemPlan plan = smem_plan(sv.n_layers, sv.max_ngram, sv.n_cols, tile, GATHER);
  auto kern = hash_kernel<GATHER, D, ONE, SDT>;
  if (plan.bytes > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, plan.bytes);
    if (e != cudaSuccess) return e;
  }
  const dim3 grid = a.cu_seqlens != nullptr ? dim3((unsigned)(a.total / tile + a.B))
                                             : dim3((unsigned)((a.L + tile - 1) / tile), (unsigned)a.B);
  return launch_pdl(kern, grid, dim3(GATHER ? kThreads : kHashThreads), plan.bytes, s, sv, a, tile);
}

// a row with a single scale block (block >= head_dim) loads its scale once
template <int D, int SDT>
cudaError_t launch_fused_s(const StateView& sv, const CallArgs& a, int tile, cudaStream_t s) {
  if (a.block >= D) return launch_hash_k<true, D, true, SDT>(sv, a, tile, s);
  return launch_hash_k<true, D, false, SDT>(sv, a, tile, s);
}

template <int D>
cudaError_t launch_fused_d(const StateView& sv, const CallArgs& a, int tile, cudaStream_t s) {
  switch (a.scale_dtype) {
    case ENGRAM_SCALE_F32: return launch_fused_s<D, ENGRAM_SCALE_F32>(sv, a, tile, s);
    case ENGRAM_SCALE_BF16: return launch_fused_s<D, ENGRAM_SCALE_BF16>(sv, a, tile, s);
    case ENGRAM_SCALE_E8M0: return launch_fused_s<D, ENGRAM_SCALE_E8M0>(sv, a, tile, s);
    case ENGRAM_SCALE_E4M3: return launch_fused_s<D, ENGRAM_SCALE_E4M3>(sv, a, tile, s);
    default: return cudaErrorInvalidValue;
  }
}

template <int D, int SDT>
cudaError_t launch_lookup_s(const int64_t* idx, int64_t n_idx, const uint8_t* W, const void* S, int64_t rows,
                            int blk, uint16_t* out, cudaStream_t s) {
  constexpr int G = D / 16;
  const int64_t units = n_idx * G;
  int64_t blocks = (units + (int64_t)kThreads * kUnroll - 1) / ((int64_t)kThreads * kUnroll);
  // one batch of kUnroll pieces per thread: many short CTAs beat a grid-stride loop over a few
  // (138.5 vs 144.2 us at 32 CTAs per SM); the cap only keeps huge calls inside the grid limit
  const int64_t cap = (int64_t)1 << 30;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const int blk_shift = ilog2(blk);
  auto kern = blk >= D ? lookup_kernel<D, true, SDT> : lookup_kernel<D, false, SDT>;
  return launch_pdl(kern, dim3((unsigned)blocks), dim3(kThreads), 0, s, idx, n_idx, W, S, rows, blk_shift, out);
}

template <int D>
cudaError_t launch_lookup_g(const int64_t* idx, int64_t n_idx, const uint8_t* W, const void* S, int64_t rows,
                            int blk, int sdt, uint16_t* out, cudaStream_t s) {
  switch (sdt) {
    case ENGRAM_SCALE_F32: return launch_lookup_s<D, ENGRAM_SCALE_F32>(idx, n_idx, W, S, rows, blk, out, s);
    case ENGRAM_SCALE_BF16: return launch_lookup_s<D, ENGRAM_SCALE_BF16>(idx, n_idx, W, S, rows, blk, out, s);
    case ENGRAM_SCALE_E8M0: return launch_lookup_s<D, ENGRAM_SCALE_E8M0>(idx, n_idx, W, S, rows, blk, out, s);
    case ENGRAM_SCALE_E4M3: return launch_lookup_s<D, ENGRAM_SCALE_E4M3>(idx, n_idx, W, S, rows, blk, out, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_fill_i32(int32_t* p, int64_t n, int32_t value, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  return launch_pdl(fill_i32_kernel, dim3((unsigned)blocks), dim3(256), 0, s, p, n, value);
}

cudaError_t launch_hash(const StateView& sv, const CallArgs& a, cudaStream_t s) {
  return launch_hash_k<false, 16, false, ENGRAM_SCALE_F32>(sv, a, kHashTile, s);
}

// Tokens per CTA of the fused kernel: the largest power of two in [kMinFusedTile, kFusedTile] that
// still gives about kTargetCtas CTAs, so small launches (one 8K-token chunk, a 16K-token prefill) fill several
// waves instead of leaving SMs idle; a smaller tile only re-reads a (max_ngram-1)-token halo more.
int fused_tile(const CallArgs& a) {
#ifdef ENGRAM_FIXED_TILE
  return ENGRAM_FIXED_TILE;
#endif
  int tile = kFusedTile;
  // CTAs that do work: every row's tiles (dense), or about total/tile + one partial tile per sequence
  auto active = [&](int t) {
    return a.cu_seqlens != nullptr ? a.total / t + a.B : (int64_t)a.B * ((a.L + t - 1) / t);
  };
  while (tile > kMinFusedTile && active(tile) < kTargetCtas) tile >>= 1;
  return tile;
}

cudaError_t launch_hash_lookup(const StateView& sv, const CallArgs& a, cudaStream_t s) {
  const int tile = fused_tile(a);
  switch (a.head_dim) {
    case 16: return launch_fused_d<16>(sv, a, tile, s);
    case 32: return launch_fused_d<32>(sv, a, tile, s);
    case 64: return launch_fused_d<64>(sv, a, tile, s);
    case 128: return launch_fused_d<128>(sv, a, tile, s);
    case 256: return launch_fused_d<256>(sv, a, tile, s);
    case 512: return launch_fused_d<512>(sv, a, tile, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_lookup(const int64_t* idx, int64_t n_idx, const uint8_t* W, const void* S, int64_t rows,
                          int32_t head_dim, int32_t block, int32_t scale_dtype, uint16_t* out, cudaStream_t s) {
  switch (head_dim) {
    case 16: return launch_lookup_g<16>(idx, n_idx, W, S, rows, block, scale_dtype, out, s);
    case 32: return launch_lookup_g<32>(idx, n_idx, W, S, rows, block, scale_dtype, out, s);
    case 64: return launch_lookup_g<64>(idx, n_idx, W, S, rows, block, scale_dtype, out, s);
    case 128: return launch_lookup_g<128>(idx, n_idx, W, S, rows, block, scale_dtype, out, s);
    case 256: return launch_lookup_g<256>(idx, n_idx, W, S, rows, block, scale_dtype, out, s);
    case 512: return launch_lookup_g<512>(idx, n_idx, W, S, rows, block, scale_dtype, out, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace engram
