// The Engram `wkv` projection on the sm_103a tensor cores: "DeepSeek V4.1" pages, blocks/stack-hashes
// page, `Engram.forward`, kv = wkv(embedding rows flattened over the hash columns):
//   kv[t][n] = bf16_rne( sum_k emb[t][k] * wkv[n][k] )     (bf16 inputs, fp32 accumulation)
// and, fused into the same kernel's epilogue, the sums that the gate after it needs, so that the
// keys are never written to memory (engram_project_gate).
//
// Design (GB300): a dense contraction (T x K x N = 65,536 x 3,072 x 25,600 per layer at the released
// width), so it runs on the 5th-generation tensor cores. A cluster of two CTAs on two SMs (a pair)
// computes 256 x 256 output tiles with M = 256 MMAs issued by its leader (tcgen05.mma.cta_group::2):
// each CTA holds its 128 rows of A and half of the B tile, and receives its 128 rows of the
// accumulator in its own tensor memory. The 76 pairs are persistent and walk the tile list. In each
// CTA the warps specialise:
//   warp 0      one thread issues TMA loads (128-byte swizzle) of its 128 x 128 A block and 128 x 128
//               B block (two 64-column boxes each) into a 3-stage ring of 64 KB stages, counted on the
//               leader's barriers;
//   warp 1      allocates 512 columns of tensor memory in both CTAs (two 128 x 256 fp32 accumulators);
//               in the leader one thread issues the MMAs (M 256, N 256, K 16; 8 per stage) and commits
//               each stage back to both loaders and each finished tile to both epilogues;
//   warps 2-5   the epilogue: each thread owns one row (one tensor-memory lane), reads its 256 fp32
//               accumulators 32 columns at a time and either rounds them to bf16 and stores them (a
//               swizzled shared-memory chunk per warp, written out by a TMA store), or (gate epilogue)
//               turns a key tile into three partial sums per row.
// The two accumulators let the epilogue of tile i run while the tensor cores compute tile i+1.
// The lookup-ahead form (engram_lookup_project*) adds warps 6-9, which look the rows of A up from the
// hash ids into a workspace one tile group ahead of the loads (see "lookup ahead" below); the loader
// waits, once per group, until that group's rows are written.
// Tiles are visited in groups of 16 tile rows, column block outer, so the tiles in flight share a few
// A and B blocks, which stay in L2. Built with ENGRAM_PROJ_CLUSTER=1 or 4 the same kernel runs one
// CTA per tile (M = 128 MMAs) or two pairs side by side that share A by TMA multicast; both measured
// no faster.
//
// Every wait is bounded (tc_ptx.cuh): a wait that runs out raises ENGRAM_STATUS_TIMEOUT in the
// library's device status word, the CTA stops issuing work, waits for its copies and MMAs in
// flight, frees its tensor memory and exits.
#include <cuda.h>

#include <cstdint>
#include <mutex>

#include "dequant.cuh"
#include "engram_internal.cuh"
#include "proj.cuh"
#include "tc_ptx.cuh"

namespace engram {

// Flags raised by kernels that have no state object (read with engram_device_status).
__device__ unsigned int g_device_status;

namespace {

constexpr int kBM = 128;           // tile rows of one CTA (tokens)
constexpr int kBN = 256;           // widest tile (output features); calls of one row tile use 128 (project_tile_cols)
#ifndef ENGRAM_PROJ_KATOMS
// 128-byte swizzle atoms (64 bf16 of K each) per stage. Two atoms (8 MMAs per stage wait and commit)
// measured as fast as one with the store epilogue and 2.4-4.0% faster with the gate epilogue (steady
// state under the power cap, 16,384 and 65,536 tokens); three atoms (two stages) were slower.
#define ENGRAM_PROJ_KATOMS 2
#endif
constexpr int kAtomK = 64;                        // K of one 128-byte swizzle row: 64 bf16
constexpr int kKAtoms = ENGRAM_PROJ_KATOMS;
constexpr int kBK = kAtomK * kKAtoms;             // K per stage
constexpr int kUmmaK = 16;         // K of one tcgen05.mma (kind::f16)
constexpr int kThreads = 192;      // 6 warps: loader, MMA, 4 epilogue
#ifndef ENGRAM_LOOKUP_WARPS
#define ENGRAM_LOOKUP_WARPS 4
#endif
#ifndef ENGRAM_LOOKUP_BATCH
#define ENGRAM_LOOKUP_BATCH 8
#endif
#ifndef ENGRAM_LOOKUP_CHUNK
#define ENGRAM_LOOKUP_CHUNK 8  // largest chunk; smaller calls take smaller chunks (lookup_chunk_tokens)
#endif
constexpr int kLookupWarps = ENGRAM_LOOKUP_WARPS;  // lookup ahead: warps 6, 7, ... look the rows of A up
constexpr int kThreadsLookup = kThreads + 32 * kLookupWarps;
constexpr int kChunkTokens = ENGRAM_LOOKUP_CHUNK;  // lookup ahead: most tokens per chunk of work (all columns)
constexpr int kLookupBatch = ENGRAM_LOOKUP_BATCH;  // lookup ahead: 16-code pieces in flight per lane
constexpr uint32_t kABytes = kBM * kBK * 2;
constexpr uint32_t kAAtomBytes = kBM * kAtomK * 2;  // one atom of the A block: 128 rows of 128 bytes
constexpr uint32_t kEpiChunkBytes = 32 * 32 * 2;  // one epilogue warp's 32 rows x 32 columns of bf16
#ifndef ENGRAM_PROJ_PAIR_STAGES
#define ENGRAM_PROJ_PAIR_STAGES 3  // stages of 64 KB (two atoms of K) in the ring of a CTA of a pair
#endif
#ifndef ENGRAM_PROJ_GROUP
#define ENGRAM_PROJ_GROUP 16  // 256-row blocks per tile group (16 measured ahead of 4, 8 and 32)
#endif

// Sizes below are per 64-column atom of K; a stage holds kKAtoms of them.
// CS = 1: one CTA computes a 128 x 256 tile with M = 128 MMAs (A + all of B, 48 KB per atom).
// CS = 2: a cluster of two CTAs (a pair) computes a 256 x 256 tile with M = 256 pair MMAs issued by
// the leader; each CTA loads its own 128 rows of A and its half (128 rows) of B, 32 KB per atom, so
// each SM reads 2/3 of the bytes per MMA from L2 that a lone CTA does.
// CS = 4: two pairs side by side along N compute a 256 x 512 tile and share A: each CTA loads 64 of
// its 128 A rows and multicasts them to the CTA at the same place in the other pair, so L2 serves
// 3/4 of the bytes per MMA of a pair. Four-CTA clusters fill 144 of the 152 SMs.
// BN: tile columns (256, or 128 for calls with few row tiles); the ring keeps the bytes of
// ENGRAM_PROJ_PAIR_STAGES stages of the 256-column form, so narrower tiles get more stages.
template <int CS, int BN = kBN>
struct Cfg {
  static constexpr bool kPairs = CS >= 2;
  static constexpr int kAccCols = BN;                          // fp32 accumulator columns per tile
  static constexpr int kTmemCols = 2 * BN;                     // two accumulators
  static constexpr int kBRows = kPairs ? BN / 2 : BN;          // rows of the B tile this CTA loads
  static constexpr int kARows = CS == 4 ? kBM / 2 : kBM;        // rows of A this CTA loads per stage
  static constexpr uint32_t kBBytes = kBRows * kBK * 2;
  static constexpr uint32_t kBAtomBytes = kBRows * kAtomK * 2;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = kPairs ? (int)(ENGRAM_PROJ_PAIR_STAGES * (kABytes + (kBM * kBK * 2)) / kStageBytes)
                                        : 4 / kKAtoms;
  static constexpr uint32_t kTxBytes = kPairs ? 2 * kStageBytes : kStageBytes;  // per stage, both CTAs of a pair
  static constexpr int kTileM = kPairs ? 2 * kBM : kBM;        // rows of one cluster tile
  static constexpr int kNBlocks = CS == 4 ? 2 : 1;             // 256-column blocks of one cluster tile
  static constexpr int kGroup = (kPairs ? 1 : 2) * ENGRAM_PROJ_GROUP;  // tile rows per group (256-row units)
  static constexpr uint32_t kIdesc = tc::idesc_bf16_f32(kTileM, BN);
  // shared memory: the stage ring (1024-byte aligned), then barriers and two words
  static constexpr uint32_t kRingBytes = kStages * kStageBytes;
  static constexpr uint32_t kEpiOff = kRingBytes;  // output staging: 2 chunks of 32 x 32 bf16 per epilogue warp
  static constexpr uint32_t kEpiBytes = 4 * 2 * kEpiChunkBytes;
  static constexpr uint32_t kBarOff = kEpiOff + kEpiBytes;  // full[S], empty[S], acc_full[2], acc_empty[2], drain
  static constexpr uint32_t kNumBars = 2 * kStages + 4 + 1;
  static constexpr uint32_t kTmemSlotOff = kBarOff + 8 * kNumBars;  // tensor-memory base written by the alloc
  static constexpr uint32_t kAbortOff = kTmemSlotOff + 4;          // set by a role whose wait ran out
  static constexpr uint32_t kGroupOff = kAbortOff + 4;             // lookup ahead: the loader's tile group
  static constexpr uint32_t kSmemBytes = kGroupOff + 4 + 1024;     // + slack to align the ring to 1024 bytes
  static_assert(kSmemBytes <= 232448, "the stage ring must fit in a CTA's shared memory");
};

enum Epilogue { EPI_STORE = 0, EPI_GATE = 1 };

struct ProjParams {
  int64_t T;        // rows of emb (tokens)
  int32_t K;        // columns of emb and wkv
  int32_t N;        // rows of wkv = output columns
  int32_t num_kb;   // ceil(K / kBK)
  int32_t n_mtile;  // ceil(T / cluster tile rows)
  int32_t bn;       // tile columns: 256, or 128 (project_tile_cols)
  int32_t n_nblk;   // ceil(N / bn)
  int32_t n_ntile;  // ceil(n_nblk / 256-column blocks per cluster tile)
  int64_t n_tiles;
  // EPI_STORE: out [T][N] bf16
  uint16_t* out;
  // EPI_GATE: N = (hc + 1) * dim, dim a multiple of 256. Key tiles (columns < hc * dim) produce the
  // partial sums sum(h^2), sum(k^2), sum(h * q_weight * k_weight * k) of every row over their 256
  // columns into part[m_blk][n_blk][3][kBM]; value tiles store bf16 rows into value [T][dim].
  const uint16_t* x;   // [T][hc][dim] residual copies (h)
  const uint16_t* qw;  // [hc][dim]
  const uint16_t* kw;  // [hc][dim]
  uint16_t* value;     // [T][dim]
  float* part;         // [ceil(T / kBM)][hc * dim / bn][3][kBM]
  int32_t hc, dim;
  // test hook (engram_project_withhold): the leader of every cluster does not signal the completion
  // of its tile number `withhold` (counted from 0 per cluster), so that tile's epilogue waits in vain
  // until its time limit; -1: every tile is signalled
  int32_t withhold;
  // Lookup ahead (engram_lookup_project*): A is the bf16 lookup of hash ids, written by this kernel's
  // lookup warps into `emb` one tile group ahead of the loads that read it.
  const int64_t* idx;       // token t's n_cols table row ids at idx[t * idx_stride + c]
  int64_t idx_stride;
  const uint8_t* W;         // fp8 E4M3 codes [rows][head_dim]
  const void* S;            // scales [rows][head_dim / block], stored as scale_dtype
  int64_t rows;
  uint16_t* emb;            // [T][K] bf16, K = n_cols * head_dim: the looked-up rows (A of the projection)
  unsigned int* counters;   // [0]: next chunk to take; [1 + g]: chunks of tile group g written
  int32_t chunk_tokens;     // tokens per chunk of lookup work: a power of two up to kChunkTokens
  int64_t n_chunks;         // ceil(T / chunk_tokens)
  int32_t group_tokens;     // tokens of one tile group
  int32_t n_cols, head_dim, block, scale_dtype;
};

// tile index -> (tile row, column block): groups of `group` tile rows, column block outer, so the
// tiles in flight at one time share a few A and B blocks, which stay in L2
__device__ __forceinline__ void tile_coords(const ProjParams& p, int group, int64_t tile, int32_t& mt, int32_t& nb) {
  const int64_t per_group = (int64_t)group * p.n_ntile;
  const int64_t g = tile / per_group;
  const int64_t r = tile - g * per_group;
  const int32_t m0 = (int32_t)(g * group);
  const int32_t gm = min(group, p.n_mtile - m0);
  mt = m0 + (int32_t)(r % gm);
  nb = (int32_t)(r / gm);
}

__device__ __forceinline__ void raise_timeout(volatile int* abort) {
  *abort = 1;
  atomicOr(&g_device_status, (unsigned)ENGRAM_STATUS_TIMEOUT);
}

// lane 0 waits, the warp follows its result (keeps the warp converged for .sync.aligned tcgen05 ops)
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) {
    ok = tc::mbar_wait(bar, parity, abort) ? 1 : 0;
    if (!ok) raise_timeout(abort);
  }
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ uint4 ld_nc_v4(const uint16_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 pack8(const float* v) {
  return make_uint4(tc::f32x2_to_bf16x2(v[0], v[1]), tc::f32x2_to_bf16x2(v[2], v[3]),
                    tc::f32x2_to_bf16x2(v[4], v[5]), tc::f32x2_to_bf16x2(v[6], v[7]));
}

// bf16 output of one accumulator tile, for this warp's 32 rows (rows y0 .. y0 + 31 of the tensor of
// `tmap`, columns x0 .. x0 + 255): 32 columns at a time, each thread converts its row to bf16 and
// writes it into a 2 KB staging chunk (64-byte rows, 16-byte pieces swizzled as the tensor map's
// 64-byte swizzle expects, so the warp's writes hit distinct banks), and lane 0 stores the chunk with
// one TMA copy. Two chunks per warp alternate; a chunk is rewritten only after the copy issued from it
// two chunks earlier has read it. Whole 128-byte lines reach L2 instead of a 16-byte piece of each of
// 32 rows per store instruction, which costs less power (the projection runs at the power limit).
template <int COLS>
__device__ __forceinline__ void store_tile_rows_tma(uint32_t taddr, const void* tmap, uint32_t stage_base, int x0,
                                                    int32_t y0) {
  const int lane = threadIdx.x & 31;
#pragma unroll 1
  for (int c = 0; c < COLS / 32; ++c) {
    float v[32];
    tc::tmem_load_32cols(taddr + 32 * c, v);
    const uint32_t chunk = stage_base + (uint32_t)(c & 1) * kEpiChunkBytes;
    if (lane == 0) tc::bulk_wait_group_read_1();
    __syncwarp();
    const uint32_t row = chunk + (uint32_t)lane * 64u;
#pragma unroll
    for (int g = 0; g < 4; ++g) tc::st_shared_v4(row + (uint32_t)((g ^ ((lane >> 1) & 3)) * 16), pack8(v + 8 * g));
    tc::fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
      tc::tma_store_2d(tmap, chunk, x0 + 32 * c, y0);
      tc::bulk_commit_group();
    }
  }
}

// Gate sums of one key tile over its 256 columns for this thread's row: the key values are the
// accumulators rounded to bf16 (the projection's output type); h, q_weight and k_weight are bf16.
// sums[0] = sum h^2, sums[1] = sum k^2, sums[2] = sum h * (q_weight * k_weight) * k, in fp32.
// h streams from memory (it was prefetched into L2 a tile earlier); two 32-column chunks of it are
// in flight in registers while a third is reduced.
__device__ __forceinline__ void load_h_chunk(uint4 (&d)[4], const uint16_t* hrow, int c) {
#pragma unroll
  for (int g = 0; g < 4; ++g) d[g] = hrow != nullptr ? ld_nc_v4(hrow + 32 * c + 8 * g) : make_uint4(0u, 0u, 0u, 0u);
}

template <int COLS>
__device__ __forceinline__ void gate_tile_row(uint32_t taddr, const uint16_t* hrow, const uint16_t* qrow,
                                              const uint16_t* wrow, float (&sums)[3]) {
  constexpr int kChunks = COLS / 32;
  float sh = 0.f, sk = 0.f, sd = 0.f;
  uint4 h0[4], h1[4], h2[4];
  load_h_chunk(h0, hrow, 0);
  load_h_chunk(h1, hrow, 1);
#pragma unroll 1
  for (int c = 0; c < kChunks; ++c) {
    if (c + 2 < kChunks) load_h_chunk(h2, hrow, c + 2);
    float v[32];
    tc::tmem_load_32cols(taddr + 32 * c, v);
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      float h[8], q[8], w[8], k[8];
      bf16x8_to_f32(h0[g], h);
      bf16x8_to_f32(ld_nc_v4(qrow + 32 * c + 8 * g), q);  // the same for every row: L1 hits
      bf16x8_to_f32(ld_nc_v4(wrow + 32 * c + 8 * g), w);
      bf16x8_to_f32(pack8(v + 8 * g), k);                    // round the keys to bf16
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        sh = fmaf(h[e], h[e], sh);
        sk = fmaf(k[e], k[e], sk);
        sd = fmaf(h[e] * (q[e] * w[e]), k[e], sd);
      }
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      h0[g] = h1[g];
      h1[g] = h2[g];
    }
  }
  sums[0] = sh;
  sums[1] = sk;
  sums[2] = sd;
}

// the row of h that this thread's row of a key tile reads (null: a value tile or a row past T)
__device__ __forceinline__ const uint16_t* h_row(const ProjParams& p, int64_t row, int col0) {
  const int key_cols = p.hc * p.dim;
  if (col0 >= key_cols || row >= p.T) return nullptr;
  const int i = col0 / p.dim;
  return p.x + (row * p.hc + i) * p.dim + (col0 - i * p.dim);
}

// ------------------------------------------------------------------------------------------------
// lookup ahead: warps 6-9 of every CTA look the rows of A up (engram-first/lookup page,
// `ParallelEngramEmbedding.forward`, through the same dequantisation as engram_lookup) into the
// workspace, one tile group ahead of the TMA loads that read them. The work is cut into chunks of
// up to kChunkTokens tokens (all their columns; fewer in calls too small to give every lookup warp a
// chunk of that size), taken in token order from a global counter by whichever warp is free, so no
// CTA waits on another one being resident. A warp takes a chunk of tile group g
// only once its own CTA's loader has reached group g - 1, which keeps the looked-up rows of at most
// two groups (8,192 tokens) ahead of the MMAs, in L2. The loader, before the first load of a tile
// of group g, waits until all chunks of group g are written.

__device__ __forceinline__ void st_v8(void* ptr, const uint4& a, const uint4& b) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(a.x), "r"(a.y), "r"(a.z),
               "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}

// The row ids of one batch of units of a chunk: unit u = u0 + 32 i + lane is token t0 + tt[i],
// column-and-piece cq[i] (column cq / pieces, piece cq % pieces); tt[i] = -1 past the chunk.
__device__ __forceinline__ void lookup_ids(const ProjParams& p, int64_t t0, int u0, int n_units, int per_token,
                                           int piece_shift, int lane, int64_t (&row)[kLookupBatch],
                                           int (&tt)[kLookupBatch], int (&cq)[kLookupBatch]) {
#pragma unroll
  for (int i = 0; i < kLookupBatch; ++i) {
    const int u = u0 + i * 32 + lane;
    tt[i] = u < n_units ? u / per_token : -1;
    cq[i] = u < n_units ? u - tt[i] * per_token : 0;
    row[i] = u < n_units ? __ldg(p.idx + (t0 + tt[i]) * p.idx_stride + (cq[i] >> piece_shift)) : -1;
  }
}

// Tokens [t0, t1), every column, into p.emb. Unit u is one 16-code piece (token t0 + u / per_token,
// then column-and-piece u % per_token), so consecutive lanes read one row's codes contiguously and
// write consecutive 32-byte pieces of the output. Each lane keeps kLookupBatch pieces in flight, and
// the ids of the next batch are loaded while the current batch's codes and scales are on their way.
// SDT (the scales' storage type) and ONE (a piece's 16 codes share one scale) are template
// parameters: no branch may sit between a load and the end of the batch, since the copy that joins
// two branches would wait for the loaded value and serialise the batch's loads.
template <int SDT, bool ONE>
__device__ __forceinline__ void lookup_chunk(const ProjParams& p, int64_t t0, int64_t t1, int lane) {
  const int pieces = p.head_dim >> 4;
  const int piece_shift = __ffs(pieces) - 1;
  const int per_token = p.n_cols * pieces;
  const int n_units = (int)(t1 - t0) * per_token;
  const int64_t K = (int64_t)p.n_cols * p.head_dim;
  const int64_t spr = p.head_dim / p.block;  // scales per table row
  int64_t row[kLookupBatch];
  int tt[kLookupBatch], cq[kLookupBatch];
  lookup_ids(p, t0, 0, n_units, per_token, piece_shift, lane, row, tt, cq);
#pragma unroll 1
  for (int u0 = 0; u0 < n_units; u0 += 32 * kLookupBatch) {
    uint4 code[kLookupBatch];
    uint32_t s0[kLookupBatch], s1[kLookupBatch];
    int tt_c[kLookupBatch], cq_c[kLookupBatch];
    bool ok[kLookupBatch];
#pragma unroll
    for (int i = 0; i < kLookupBatch; ++i) {
      code[i] = make_uint4(0u, 0u, 0u, 0u);
      s0[i] = s1[i] = 0u;
      ok[i] = row[i] >= 0 && row[i] < p.rows;
      tt_c[i] = tt[i];
      cq_c[i] = cq[i];
      if (ok[i]) {
        const int k0 = 16 * (cq[i] & (pieces - 1));
        code[i] = ld_rows_v4(p.W + row[i] * p.head_dim + k0);
        s0[i] = ld_scale_bits<SDT>(p.S, row[i] * spr + k0 / p.block);
        if (!ONE) s1[i] = ld_scale_bits<SDT>(p.S, row[i] * spr + (k0 + 8) / p.block);
      }
    }
    if (u0 + 32 * kLookupBatch < n_units)
      lookup_ids(p, t0, u0 + 32 * kLookupBatch, n_units, per_token, piece_shift, lane, row, tt, cq);
#pragma unroll
    for (int i = 0; i < kLookupBatch; ++i) {
      if (tt_c[i] < 0) continue;
      uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a;  // rows outside the table are +0
      if (ok[i]) {
        a = dequant8(make_uint2(code[i].x, code[i].y), widen_scale<SDT>(s0[i]));
        b = dequant8(make_uint2(code[i].z, code[i].w), widen_scale<SDT>(ONE ? s0[i] : s1[i]));
      }
      st_v8(p.emb + (t0 + tt_c[i]) * K + 16 * (int64_t)cq_c[i], a, b);
    }
  }
}

template <int SDT>
__device__ __forceinline__ void lookup_chunk_s(const ProjParams& p, int64_t t0, int64_t t1, int lane) {
  if (p.block >= 16)
    lookup_chunk<SDT, true>(p, t0, t1, lane);
  else
    lookup_chunk<SDT, false>(p, t0, t1, lane);
}

__device__ __forceinline__ void lookup_chunk_any(const ProjParams& p, int64_t t0, int64_t t1, int lane) {
  switch (p.scale_dtype) {
    case ENGRAM_SCALE_F32: lookup_chunk_s<ENGRAM_SCALE_F32>(p, t0, t1, lane); break;
    case ENGRAM_SCALE_BF16: lookup_chunk_s<ENGRAM_SCALE_BF16>(p, t0, t1, lane); break;
    case ENGRAM_SCALE_E8M0: lookup_chunk_s<ENGRAM_SCALE_E8M0>(p, t0, t1, lane); break;
    default: lookup_chunk_s<ENGRAM_SCALE_E4M3>(p, t0, t1, lane); break;
  }
}

// lane 0 of a lookup warp: wait until this CTA's loader has reached tile group `need` (or finished).
// A group lasts hundreds of microseconds at the block's shapes, so the warp polls every few
// microseconds: polling every 256 ns cost the projection about 1% (measured at 65,536 tokens).
__device__ __forceinline__ bool pace_wait(const volatile int* cur_group, int32_t need, const volatile int* abort) {
  const uint64_t t0 = tc::global_timer_ns();
  while (*cur_group < need) {
    if (*abort || tc::global_timer_ns() - t0 > tc::kWaitLimitNs) return false;
    __nanosleep(4000);
  }
  return true;
}

// the loader: wait until `need` chunks of a tile group are written (acquire: their rows are visible)
__device__ __forceinline__ bool ready_wait(const unsigned int* ctr, unsigned int need, const volatile int* abort) {
  const uint64_t t0 = tc::global_timer_ns();
  for (;;) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= need) return true;
    if (*abort || tc::global_timer_ns() - t0 > tc::kWaitLimitNs) return false;
    __nanosleep(128);
  }
}

__device__ __forceinline__ void red_release_add(unsigned int* ctr, unsigned int v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(ctr), "r"(v) : "memory");
}

// chunks of tile group g: [g * per_group, min(n_chunks, (g + 1) * per_group))
__device__ __forceinline__ unsigned int group_chunks(const ProjParams& p, int32_t g) {
  const int64_t per = p.group_tokens / p.chunk_tokens;
  const int64_t c0 = (int64_t)g * per;
  return (unsigned int)(min(p.n_chunks, c0 + per) - c0);
}

__device__ __forceinline__ void lookup_warp(const ProjParams& p, const volatile int* cur_group, volatile int* abort) {
  const int lane = threadIdx.x & 31;
  for (;;) {
    unsigned int chunk = 0;
    if (lane == 0) chunk = atomicAdd(&p.counters[0], 1u);
    chunk = __shfl_sync(0xffffffffu, chunk, 0);
    if ((int64_t)chunk >= p.n_chunks) break;
    const int64_t t0 = (int64_t)chunk * p.chunk_tokens;
    const int32_t g = (int32_t)(t0 / p.group_tokens);
    int ok = 1;
    if (lane == 0) {
      ok = pace_wait(cur_group, g - 1, abort) ? 1 : 0;
      if (!ok) raise_timeout(abort);
    }
    if (__shfl_sync(0xffffffffu, ok, 0) == 0) break;
    lookup_chunk_any(p, t0, min(p.T, t0 + (int64_t)p.chunk_tokens), lane);
    tc::fence_proxy_async_global();  // the rows are read next by TMA loads (the async proxy)
    __threadfence();
    __syncwarp();
    if (lane == 0) red_release_add(&p.counters[1 + g], 1u);
  }
}

template <int EPI, int CS, bool LA, int BN>
__global__ void __launch_bounds__(LA ? kThreadsLookup : kThreads, 1)
    proj_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmO, const ProjParams p) {
  using C = Cfg<CS, BN>;
  constexpr bool PAIR = C::kPairs;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // the same offset in every CTA of a cluster
  uint8_t* gbase = smem_raw + (base - raw);
  volatile int* abort = reinterpret_cast<volatile int*>(gbase + C::kAbortOff);
  volatile int* cur_group = reinterpret_cast<volatile int*>(gbase + C::kGroupOff);
  const uint32_t* tmem_slot = reinterpret_cast<const uint32_t*>(gbase + C::kTmemSlotOff);
  auto bar = [&](int i) { return base + C::kBarOff + 8u * (uint32_t)i; };
  auto full = [&](uint32_t s) { return bar((int)s); };
  auto empty = [&](uint32_t s) { return bar(C::kStages + (int)s); };
  auto acc_full = [&](uint32_t a) { return bar(2 * C::kStages + (int)a); };
  auto acc_empty = [&](uint32_t a) { return bar(2 * C::kStages + 2 + (int)a); };
  const uint32_t drain = bar(2 * C::kStages + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // place in the cluster: pair pr (of CS / 2), position q in the pair; q = 0 leads (issues the pair's
  // MMAs; its full and acc_empty barriers count for both CTAs of the pair)
  const uint32_t rank = CS > 1 ? tc::cluster_ctarank() : 0u;
  const uint32_t q = PAIR ? (rank & 1u) : 0u;
  const uint32_t pr = CS == 4 ? (rank >> 1) : 0u;
  const uint32_t lead = rank & ~1u;
  const bool leader = q == 0;
  const int64_t unit = (int64_t)(blockIdx.x / CS);  // cluster index
  const int64_t n_units = (int64_t)(gridDim.x / CS);
  // the loads and MMAs of a stage must have been read by every pair that writes into this CTA's copy
  // of it: with CS = 4 the other pair multicasts half of A into it
  constexpr uint32_t kEmptyArrivals = CS == 4 ? 2 : 1;
  constexpr uint16_t kAllCtas = (uint16_t)((1u << CS) - 1u);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      tc::mbar_init(full(s), 1);                // the leader's arrive + the bytes of its pair's loads
      tc::mbar_init(empty(s), kEmptyArrivals);  // a commit of every pair's leader
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(acc_full(a), 1);
      tc::mbar_init(acc_empty(a), PAIR ? 8 : 4);  // one arrival per epilogue warp of the pair (or CTA)
    }
    tc::mbar_init(drain, 1);
    *abort = 0;
    *cur_group = 0;
    tc::fence_barrier_init();
    tc::tma_prefetch_descriptor(&tmA);
    tc::tma_prefetch_descriptor(&tmB);
    tc::tma_prefetch_descriptor(&tmO);
  }
  // inputs may come from the previous kernel on the stream, and its tensor memory must be free
  pdl_wait();
  if (CS > 1) tc::cluster_sync();  // every CTA's barriers exist before anyone signals them
  if (warp == 1) {
    if (PAIR) {
      tc::tmem_alloc_pair(base + C::kTmemSlotOff, C::kTmemCols);
      tc::tmem_relinquish_alloc_permit_pair();
    } else {
      tc::tmem_alloc(base + C::kTmemSlotOff, C::kTmemCols);
      tc::tmem_relinquish_alloc_permit();
    }
  }
  tc::fence_before_thread_sync();
  __syncthreads();
  tc::fence_after_thread_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA loader (every CTA)
    int64_t issued = 0;
    uint32_t stage = 0, phase = 0;
    int32_t ready_group = -1;
    for (int64_t tile = unit; tile < p.n_tiles && !*abort; tile += n_units) {
      int32_t mt, nt;
      tile_coords(p, C::kGroup, tile, mt, nt);
      if (LA) {
        // the rows of this tile's group must be looked up before the first load of A reads them
        const int32_t g = (int32_t)(tile / ((int64_t)C::kGroup * p.n_ntile));
        if (g != ready_group) {
          *cur_group = g;  // this CTA's lookup warps may take chunks of group g + 1 from now on
          if (!ready_wait(p.counters + 1 + g, group_chunks(p, g), abort)) {
            raise_timeout(abort);
            break;
          }
          tc::fence_proxy_async_global();
          ready_group = g;
        }
      }
      const int32_t nb = nt * C::kNBlocks + (int32_t)pr;
      const int32_t arow0 = mt * C::kTileM + (int32_t)q * kBM + (int32_t)pr * C::kARows;
      const int32_t brow0 = nb * BN + (int32_t)q * C::kBRows;
      for (int kb = 0; kb < p.num_kb; ++kb) {
        if (!tc::mbar_wait(empty(stage), phase ^ 1u, abort)) {
          raise_timeout(abort);
          break;
        }
        // one box per 128-byte swizzle atom of K: atom j of A at a_dst + j * kAAtomBytes, of B after A
        const uint32_t a_dst = base + stage * C::kStageBytes;
        if (PAIR) {
          const uint32_t fb = tc::map_to_rank(full(stage), lead);
          if (leader) tc::mbar_arrive_expect_tx(full(stage), C::kTxBytes);
#pragma unroll
          for (int j = 0; j < kKAtoms; ++j) {
            const int x = kb * kBK + j * kAtomK;
            if (CS == 4)  // this CTA's half of its A block, to itself and its counterpart in the other pair
              tc::tma_load_2d_pair_multicast(a_dst + j * kAAtomBytes + pr * (C::kARows * kAtomK * 2), &tmA, fb, x,
                                             arow0, (uint16_t)((1u << q) | (1u << (q + 2))));
            else
              tc::tma_load_2d_pair(a_dst + j * kAAtomBytes, &tmA, fb, x, arow0);
            tc::tma_load_2d_pair(a_dst + kABytes + j * C::kBAtomBytes, &tmB, fb, x, brow0);
          }
        } else {
          tc::mbar_arrive_expect_tx(full(stage), C::kTxBytes);
#pragma unroll
          for (int j = 0; j < kKAtoms; ++j) {
            const int x = kb * kBK + j * kAtomK;
            tc::tma_load_2d(a_dst + j * kAAtomBytes, &tmA, full(stage), x, arow0);
            tc::tma_load_2d(a_dst + kABytes + j * C::kBAtomBytes, &tmB, full(stage), x, brow0);
          }
        }
        ++issued;
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (LA) *cur_group = 0x7fffffff;  // no more loads: the lookup warps take any chunk left
    // No copy may still be landing in shared memory when the CTA exits. A CTA of a pair counts its
    // loads on its leader's barriers, so it waits for the MMAs that read its last loads instead
    // (which implies they landed); a lone CTA waits for the loads themselves.
    for (int64_t i = issued - (issued < C::kStages ? issued : C::kStages); i < issued; ++i) {
      const uint32_t s = (uint32_t)(i % C::kStages), ph = (uint32_t)((i / C::kStages) & 1);
      if (!tc::mbar_wait(PAIR ? empty(s) : full(s), ph, nullptr))
        atomicOr(&g_device_status, (unsigned)ENGRAM_STATUS_TIMEOUT);
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // ---------------------------------------------------------------- MMA issuer (a pair's leader)
    uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
    bool ok = true;
    const uint16_t pair_ctas = (uint16_t)(3u << lead);
    int32_t local_tile = 0;
    for (int64_t tile = unit; ok && tile < p.n_tiles && !*abort; tile += n_units, ++local_tile) {
      if (!tc::mbar_wait(acc_empty(acc), acc_phase ^ 1u, abort)) {
        raise_timeout(abort);
        break;
      }
      tc::fence_after_thread_sync();
      const uint32_t d = tmem_base + acc * C::kAccCols;
      for (int kb = 0; kb < p.num_kb; ++kb) {
        if (!tc::mbar_wait(full(stage), phase, abort)) {
          raise_timeout(abort);
          ok = false;
          break;
        }
        tc::fence_after_thread_sync();
        const uint32_t a0 = base + stage * C::kStageBytes, b0 = a0 + kABytes;
#pragma unroll
        for (int k = 0; k < kBK / kUmmaK; ++k) {
          constexpr int kPerAtom = kAtomK / kUmmaK;  // MMAs per swizzle atom of K
          const uint32_t off = 2 * kUmmaK * (k % kPerAtom);
          const uint64_t ad = tc::sw128_kmajor_desc(a0 + (k / kPerAtom) * kAAtomBytes + off);
          const uint64_t bd = tc::sw128_kmajor_desc(b0 + (k / kPerAtom) * C::kBAtomBytes + off);
          if (PAIR)
            tc::mma_bf16_pair(d, ad, bd, C::kIdesc, (kb | k) != 0 ? 1u : 0u);
          else
            tc::mma_bf16(d, ad, bd, C::kIdesc, (kb | k) != 0 ? 1u : 0u);
        }
        // the stage returns to every loader that writes into it once these MMAs have read it
        if (PAIR)
          tc::commit_pair_multicast(empty(stage), kAllCtas);
        else
          tc::commit(empty(stage));
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      // the tile's accumulators are complete once every MMA above is
      if (local_tile != p.withhold) {
        if (PAIR)
          tc::commit_pair_multicast(acc_full(acc), pair_ctas);
        else
          tc::commit(acc_full(acc));
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // every MMA this thread issued has completed before tensor memory is freed
    if (PAIR)
      tc::commit_pair_multicast(drain, (uint16_t)(1u << rank));
    else
      tc::commit(drain);
    if (!tc::mbar_wait(drain, 0, nullptr)) atomicOr(&g_device_status, (unsigned)ENGRAM_STATUS_TIMEOUT);
  } else if (LA && warp >= 6) {
    // ---------------------------------------------------------------- lookup ahead (every CTA)
    lookup_warp(p, cur_group, abort);
  } else if (warp >= 2 && warp < 6) {
    // ---------------------------------------------------------------- epilogue (every CTA)
    const int quarter = warp & 3;  // tensor-memory lanes [32*quarter, 32*quarter + 32)
    const int r = quarter * 32 + lane;
    uint32_t acc = 0, acc_phase = 0;
    // the gate epilogue reads h: each thread prefetches its row of the next key tile into L2 one tile ahead
    auto prefetch_h = [&](int64_t t) {
      if (EPI != EPI_GATE || t >= p.n_tiles) return;
      int32_t pm, pn;
      tile_coords(p, C::kGroup, t, pm, pn);
      const int col = (pn * C::kNBlocks + (int)pr) * BN;
      if (col >= p.N) return;
      const uint16_t* hr = h_row(p, ((int64_t)pm * (C::kTileM / kBM) + q) * kBM + r, col);
      if (hr != nullptr) tc::prefetch_l2_bulk(hr, BN * 2);
    };
    prefetch_h(unit);
    for (int64_t tile = unit; tile < p.n_tiles; tile += n_units) {
      int32_t mt, nt;
      tile_coords(p, C::kGroup, tile, mt, nt);
      if (!warp_wait(acc_full(acc), acc_phase, abort)) break;
      tc::fence_after_thread_sync();
      prefetch_h(tile + n_units);
      const int64_t mb = (int64_t)mt * (C::kTileM / kBM) + q;  // this CTA's block of 128 rows
      const int64_t row = mb * kBM + r;
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * C::kAccCols;
      const int col0 = (nt * C::kNBlocks + (int)pr) * BN;  // a pair past the last column block stores nothing
      const uint32_t stage_base = base + C::kEpiOff + (uint32_t)quarter * 2u * kEpiChunkBytes;
      const int32_t y0 = (int32_t)(mb * kBM) + quarter * 32;  // TMA stores skip rows past T
      if (EPI == EPI_STORE) {
        if (col0 < p.N) store_tile_rows_tma<BN>(taddr, &tmO, stage_base, col0, y0);
      } else if (col0 < p.N) {
        const int key_cols = p.hc * p.dim;
        if (col0 < key_cols) {
          const int i = col0 / p.dim, j0 = col0 - i * p.dim;
          float sums[3];
          gate_tile_row<BN>(taddr, h_row(p, row, col0), p.qw + i * p.dim + j0, p.kw + i * p.dim + j0, sums);
          float* dst = p.part + (mb * (key_cols / BN) + col0 / BN) * 3 * kBM + r;
          dst[0] = sums[0];
          dst[kBM] = sums[1];
          dst[2 * kBM] = sums[2];
        } else {
          store_tile_rows_tma<BN>(taddr, &tmO, stage_base, col0 - key_cols, y0);
        }
      }
      tc::fence_before_thread_sync();
      __syncwarp();
      if (lane == 0) {
        if (PAIR)
          tc::mbar_arrive_cluster(tc::map_to_rank(acc_empty(acc), lead));
        else
          tc::mbar_arrive(acc_empty(acc));
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (lane == 0) tc::bulk_wait_group_0();  // this warp's output copies are done before the CTA exits
    __syncwarp();
  }
  pdl_trigger();
  tc::fence_before_thread_sync();
  __syncthreads();
  // no CTA of a cluster leaves while another may still signal its barriers or read its memory
  if (CS > 1) tc::cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc::fence_after_thread_sync();
    if (PAIR)
      tc::tmem_dealloc_pair(tmem_base, C::kTmemCols);
    else
      tc::tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

}  // namespace

// ------------------------------------------------------------------------------------------------
// host side

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime (no link to libcuda)
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// [rows][cols] bf16 row-major, moved in boxes of box_rows x box_cols: operands are read with 128-byte
// swizzling (reads past the matrix, ragged rows or K, are filled with zeros), outputs written from
// 64-byte swizzled staging chunks (writes past the matrix are dropped)
bool make_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows,
              uint32_t box_cols = kAtomK, CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

#ifndef ENGRAM_PROJ_CLUSTER
#define ENGRAM_PROJ_CLUSTER 2
#endif
// CTAs per cluster: 1, 2 (a pair) or 4 (two pairs sharing A). Sustained at the block shape on one box
// (power-limited, alternating rounds) pairs took 5.91 ms and four-CTA clusters 5.94 ms: the multicast
// saves L2 traffic but leaves 8 SMs idle, so pairs are the default.
constexpr int kCS = ENGRAM_PROJ_CLUSTER;
static_assert(kCS == 1 || kCS == 2 || kCS == 4, "cluster of 1, 2 or 4 CTAs");

ProjParams base_params(int64_t T, int32_t K, int32_t N) {
  ProjParams p = {};
  p.T = T;
  p.K = K;
  p.N = N;
  p.num_kb = (K + kBK - 1) / kBK;
  p.n_mtile = (int32_t)((T + Cfg<kCS>::kTileM - 1) / Cfg<kCS>::kTileM);
  p.bn = (int32_t)project_tile_cols(T);
  p.n_nblk = (N + p.bn - 1) / p.bn;
  p.n_ntile = (p.n_nblk + Cfg<kCS>::kNBlocks - 1) / Cfg<kCS>::kNBlocks;
  p.n_tiles = (int64_t)p.n_mtile * p.n_ntile;
  p.withhold = -1;
  return p;
}

// as many persistent clusters as can be resident at once, launched as a programmatic dependent like
// every kernel of the library
template <int EPI, bool LA, int BN>
cudaError_t launch_proj_bn(const uint16_t* emb, const uint16_t* w, const ProjParams& p, cudaStream_t s) {
  using C = Cfg<kCS, BN>;
  CUtensorMap ta, tb, to;
  // the output tensor: out [T][N], or the value rows [T][dim] of the gate epilogue
  const uint16_t* optr = EPI == EPI_STORE ? p.out : p.value;
  const uint64_t ocols = EPI == EPI_STORE ? (uint64_t)p.N : (uint64_t)p.dim;
  if (!make_map(&ta, emb, (uint64_t)p.T, (uint64_t)p.K, (uint32_t)C::kARows) ||
      !make_map(&tb, w, (uint64_t)p.N, (uint64_t)p.K, (uint32_t)C::kBRows) ||
      !make_map(&to, optr, (uint64_t)p.T, ocols, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  auto kern = proj_kernel<EPI, kCS, LA, BN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = ENGRAM_PDL;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kCS;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.blockDim = dim3(LA ? kThreadsLookup : kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  int units = 0;
  if (kCS > 1) {
    cfg.gridDim = dim3(kCS);
    e = cudaOccupancyMaxActiveClusters(&units, kern, &cfg);
  } else {
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&units, cudaDevAttrMultiProcessorCount, dev);
  }
  if (e != cudaSuccess) return e;
  if (units < 1) return cudaErrorInvalidConfiguration;
  const int64_t n = p.n_tiles < units ? p.n_tiles : units;
  cfg.gridDim = dim3((unsigned)(n * kCS));
  return cudaLaunchKernelEx(&cfg, kern, ta, tb, to, p);
}

template <int EPI, bool LA = false>
cudaError_t launch_proj(const uint16_t* emb, const uint16_t* w, const ProjParams& p, cudaStream_t s) {
  return p.bn == 128 ? launch_proj_bn<EPI, LA, 128>(emb, w, p, s) : launch_proj_bn<EPI, LA, 256>(emb, w, p, s);
}

// lookup ahead: the lookup arguments, the rows' workspace, and its counters zeroed on the stream
cudaError_t lookup_ahead_params(ProjParams& p, const LookupArgs& la, cudaStream_t s) {
  using C = Cfg<kCS>;
  static_assert((C::kGroup * C::kTileM) % kChunkTokens == 0, "a chunk of lookup work lies in one tile group");
  // chunks of up to kChunkTokens tokens, smaller when the call has fewer tokens than the lookup warps
  // could take in chunks of that size (a 256-token call on 152 SMs: 1-token chunks, 256 of them);
  // powers of two, so a chunk never straddles a tile group
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  int32_t ct = kChunkTokens;
  const int64_t warps = (int64_t)sms * kLookupWarps;  // one CTA per SM
  while (ct > 1 && p.T < (int64_t)ct * warps) ct >>= 1;
  p.chunk_tokens = ct;
  p.idx = la.idx;
  p.idx_stride = la.idx_stride;
  p.n_cols = la.n_cols;
  p.W = la.W;
  p.S = la.S;
  p.rows = la.rows;
  p.head_dim = la.head_dim;
  p.block = la.block;
  p.scale_dtype = la.scale_dtype;
  p.emb = la.emb;
  p.counters = la.counters;
  p.n_chunks = (p.T + ct - 1) / ct;
  p.group_tokens = C::kGroup * C::kTileM;
  return launch_fill_i32(reinterpret_cast<int32_t*>(la.counters), lookup_ahead_counters(p.T), 0, s);
}

}  // namespace

int64_t lookup_ahead_counters(int64_t T) {
  using C = Cfg<kCS>;
  const int64_t group_tokens = (int64_t)C::kGroup * C::kTileM;
  return 1 + (T + group_tokens - 1) / group_tokens;
}

cudaError_t launch_lookup_project(const LookupArgs& la, const uint16_t* wkv, int64_t T, int32_t N, uint16_t* out,
                                  cudaStream_t s) {
  ProjParams p = base_params(T, la.n_cols * la.head_dim, N);
  p.out = out;
  cudaError_t e = lookup_ahead_params(p, la, s);
  if (e != cudaSuccess) return e;
  return launch_proj<EPI_STORE, true>(la.emb, wkv, p, s);
}

cudaError_t launch_lookup_project_gate_sums(const uint16_t* x, const LookupArgs& la, const uint16_t* wkv,
                                            const uint16_t* qw, const uint16_t* kw, int64_t T, int32_t hc,
                                            int32_t dim, uint16_t* value, float* part, cudaStream_t s) {
  ProjParams p = base_params(T, la.n_cols * la.head_dim, (hc + 1) * dim);
  p.x = x;
  p.qw = qw;
  p.kw = kw;
  p.value = value;
  p.part = part;
  p.hc = hc;
  p.dim = dim;
  cudaError_t e = lookup_ahead_params(p, la, s);
  if (e != cudaSuccess) return e;
  return launch_proj<EPI_GATE, true>(la.emb, wkv, p, s);
}

cudaError_t launch_project(const uint16_t* emb, const uint16_t* w, int64_t T, int32_t K, int32_t N, uint16_t* out,
                           cudaStream_t s, int32_t withhold) {
  ProjParams p = base_params(T, K, N);
  p.out = out;
  p.withhold = withhold;
  return launch_proj<EPI_STORE>(emb, w, p, s);
}

#ifndef ENGRAM_PROJ_NARROW_T
#define ENGRAM_PROJ_NARROW_T 256  // calls of at most this many tokens use 128-column tiles
#endif
// 128-column tiles for calls of one row tile: a decode batch's projection (T = 256, N = 25,600) has
// only 100 tiles of 256 columns for 76 pairs, a full wave and a third; 200 narrower tiles fill the
// waves better: 38.9 against 41.2 us per call. From 512 tokens on the waves are as full either way and
// the wider tiles win (57.9 against 68.7 us at 512 tokens, even at 1,024): a narrow tile does half the
// work per MMA and per stage wait and re-reads its rows of A twice as often. Each output sums its K
// terms in the same order either way: the same bits.
int64_t project_tile_cols(int64_t T) { return T <= ENGRAM_PROJ_NARROW_T ? 128 : 256; }

int64_t project_gate_partials(int64_t T, int32_t hc, int32_t dim) {
  // whole (cluster) tiles: the second CTA of a pair's last tile writes its block even past T
  const int64_t tiles = (T + Cfg<kCS>::kTileM - 1) / Cfg<kCS>::kTileM;
  return tiles * (Cfg<kCS>::kTileM / kBM) * (int64_t)(hc * dim / project_tile_cols(T)) * 3 * kBM;
}

cudaError_t launch_project_gate_sums(const uint16_t* x, const uint16_t* emb, const uint16_t* wkv, const uint16_t* qw,
                                     const uint16_t* kw, int64_t T, int32_t K, int32_t hc, int32_t dim,
                                     uint16_t* value, float* part, cudaStream_t s) {
  ProjParams p = base_params(T, K, (hc + 1) * dim);
  p.x = x;
  p.qw = qw;
  p.kw = kw;
  p.value = value;
  p.part = part;
  p.hc = hc;
  p.dim = dim;
  return launch_proj<EPI_GATE>(emb, wkv, p, s);
}

namespace {
__device__ unsigned int g_device_status_taken;

__global__ void device_status_take_kernel(int clear) {
  g_device_status_taken = clear ? atomicExch(&g_device_status, 0u) : atomicOr(&g_device_status, 0u);
}
}  // namespace

// Read (and optionally clear, in one atomic step) the device status word, ordered after the work
// already on stream s; synchronises s.
cudaError_t device_status_take(unsigned int* flags, int clear, cudaStream_t s) {
  device_status_take_kernel<<<1, 1, 0, s>>>(clear);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess)
    e = cudaMemcpyFromSymbolAsync(flags, g_device_status_taken, sizeof(unsigned int), 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e;
}

}  // namespace engram
