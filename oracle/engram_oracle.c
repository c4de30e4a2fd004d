/*
 * Engram n-gram hash + fp8 row lookup: plain CPU oracle.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
 * baseline use this file. It shares no code, header or constant with the CUDA
 * library and is deliberately slow: one loop per step of the pages, in their
 * order, with no blocking, fusion or reordering.
 *
 * Sources (all on the "DeepSeek V4.1" pages):
 *   - blocks/stack-hashes page, the n-gram hash `forward(input_ids, start_pos,
 *     token_mask)`: token compression, masking, compressed-token cache,
 *     lookback with cumulative blocking, multiply / rolling XOR, floored mod
 *     by the bucket primes, column concatenation plus offsets.
 *   - blocks/stack-hashes page, `Transformer.forward`: the engram mask is the
 *     negated image mask.
 *   - engram-first/lookup page, `ParallelEngramEmbedding.forward`: out-of-range
 *     rows are read as row 0 and then zeroed; fp8 values are widened to fp32,
 *     multiplied block-wise by the scale widened to fp32 (`.float()`), and
 *     converted to bf16.
 *
 * Precision: the pages fix it (`.float()` on both operands, one multiply,
 * `.to(torch.bfloat16)`), so the dequant is one fp32 round-to-nearest multiply
 * followed by round-to-nearest-even to bf16. Build with -ffp-contract=off and
 * without fast-math so no FMA or flush-to-zero can creep in.
 *
 * Readings where the pages are silent (documented with the build):
 *   - the cache starts out (and is reset to) DEAD;
 *   - start_pos is a per-row value; rows never interact;
 *   - int64 products wrap mod 2^64 and `%` is floored (torch semantics);
 *   - an id outside [0, raw_vocab) is treated as a masked (DEAD) token and
 *     flagged; a row whose start position does not fit the cache writes
 *     nothing, gets hash -1 everywhere, and is flagged.
 *   - the scale dtype (`scale_dtype`, left open by the pages) is fp32, bf16,
 *     UE8M0 or E4M3; each widens to fp32 exactly, as `.float()` does, before
 *     the one fp32 multiply.
 *   - call row b uses cache row b unless a cache-row map is given, in which
 *     case it uses cache row cache_rows[b] (the pages index the cache by the
 *     batch row; the map only renames rows, so each sequence is still hashed
 *     exactly as the pages' `forward` hashes a batch row). A row mapped outside
 *     the cache writes nothing, gets hash -1 everywhere, and is flagged.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)

#define ORACLE_FLAG_BAD_START 1u
#define ORACLE_FLAG_BAD_ID 2u
#define ORACLE_FLAG_BAD_ROW 8u

#define ORACLE_SCALE_F32 0
#define ORACLE_SCALE_BF16 1
#define ORACLE_SCALE_E8M0 2
#define ORACLE_SCALE_E4M3 3

/* ---------------------------------------------------------------- scalar definitions */

/* OCP 8-bit E4M3 ("fn" variant): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
 * bits; exponent 0 is subnormal (m * 2^-9); S.1111.111 is NaN; no infinities. */
float oracle_fp8_e4m3_to_f32(uint8_t code) {
  const int sign = (code >> 7) & 1;
  const int e = (code >> 3) & 0xF;
  const int m = code & 0x7;
  double v;
  if (e == 0xF && m == 0x7) {
    v = NAN;
  } else if (e == 0) {
    v = ldexp((double)m, -9);
  } else {
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  }
  return (float)(sign ? -v : v);
}

/* bfloat16 is the upper half of an IEEE binary32: widening appends 16 zero bits (exact). */
float oracle_bf16_to_f32(uint16_t h) {
  const uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* OCP UE8M0: 8 exponent bits, no sign, no mantissa: 2^(e - 127); e = 255 is NaN. */
float oracle_e8m0_to_f32(uint8_t e) {
  if (e == 0xFF) return NAN;
  return (float)ldexp(1.0, (int)e - 127); /* 2^-127 is an fp32 subnormal, still exact */
}

/* bf16 = the upper half of an IEEE binary32, rounded to nearest, ties to even.
 * NaNs stay NaN (quiet bit set). */
uint16_t oracle_bf16_rne(float x) {
  uint32_t u;
  memcpy(&u, &x, sizeof u);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u) {
    return (uint16_t)((u >> 16) | 0x0040u);
  }
  const uint32_t lower = u & 0xFFFFu;
  uint32_t upper = u >> 16;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) {
    upper += 1u; /* carries into the exponent (and to infinity) as rounding requires */
  }
  return (uint16_t)upper;
}

/* Floored modulo: the result has the sign of p (p > 0 here), like torch's `%`. */
int64_t oracle_floor_mod(int64_t x, int64_t p) {
  int64_t r = x % p; /* C: truncated toward zero, |r| < p */
  if (r != 0 && ((r < 0) != (p < 0))) r += p;
  return r;
}

/* ---------------------------------------------------------------- n-gram hash */

/* One sequence: L tokens that sit at positions s .. s+L-1 of the cache row `cache_row`
 * (cache_len positions). ids/mask/hashes point at the sequence's first token; hashes is
 * [L][n_layers][C]. Returns the status flags it raised. */
static uint32_t hash_sequence(int64_t n_layers, int64_t max_ngram, int64_t n_heads, const int64_t* token_map,
                              int64_t raw_vocab, int64_t dead, int64_t pad_id, const int64_t* multipliers,
                              const int64_t* primes, const int64_t* offsets, int64_t* cache_row, int64_t cache_len,
                              const int64_t* ids, const uint8_t* mask, int64_t s, int64_t L, int64_t* hashes) {
  const int64_t C = (max_ngram - 1) * n_heads;
  uint32_t fl = 0;
  const int row_ok = (s >= 0 && s <= cache_len - L);
  if (!row_ok) {
    for (int64_t t = 0; t < L; ++t)
      for (int64_t j = 0; j < n_layers * C; ++j) hashes[t * n_layers * C + j] = -1;
    return ORACLE_FLAG_BAD_START;
  }

  /* compressed = token_map[input_ids]; masked tokens become DEAD */
  /* cache[b, s : s + L] = compressed */
  for (int64_t t = 0; t < L; ++t) {
    const int64_t id = ids[t];
    int64_t c;
    if (id < 0 || id >= raw_vocab) {
      fl |= ORACLE_FLAG_BAD_ID;
      c = dead;
    } else {
      c = token_map[id];
    }
    if (mask != NULL && !mask[t]) c = dead;
    cache_row[s + t] = c;
  }

  /* one token at a time: lookback with cumulative blocking, then the hash */
  for (int64_t t = 0; t < L; ++t) {
    const int64_t pos = s + t;
    int64_t tokens[64];
    int blocked = 0;
    for (int64_t shift = 0; shift < max_ngram; ++shift) {
      const int64_t src_pos = pos - shift < 0 ? 0 : pos - shift; /* clamp_min(0) */
      const int64_t source = cache_row[src_pos];
      blocked = blocked || (pos < shift) || (source == dead);
      tokens[shift] = blocked ? pad_id : source;
    }
    for (int64_t l = 0; l < n_layers; ++l) {
      /* products = tokens * multipliers (int64, wrapping) */
      uint64_t products[64];
      for (int64_t k = 0; k < max_ngram; ++k)
        products[k] = (uint64_t)tokens[k] * (uint64_t)multipliers[l * max_ngram + k];
      uint64_t rolling = products[0];
      for (int64_t i = 1; i < max_ngram; ++i) {
        rolling ^= products[i];
        for (int64_t h = 0; h < n_heads; ++h) {
          const int64_t p = primes[(l * (max_ngram - 1) + (i - 1)) * n_heads + h];
          const int64_t col = (i - 1) * n_heads + h;
          const int64_t x = (int64_t)rolling; /* two's complement reinterpretation */
          hashes[(t * n_layers + l) * C + col] = oracle_floor_mod(x, p) + offsets[l * C + col];
        }
      }
    }
  }
  return fl;
}

/* The cache row of call row b: cache_rows[b] when a map is given, else b. A row outside
 * [0, max_batch) gets hash -1 everywhere (L tokens from `hashes`) and returns -1. */
static int64_t cache_row_of(const int64_t* cache_rows, int64_t b, int64_t max_batch, int64_t L, int64_t NC,
                            int64_t* hashes) {
  const int64_t r = cache_rows ? cache_rows[b] : b;
  if (r >= 0 && r < max_batch) return r;
  for (int64_t i = 0; i < L * NC; ++i) hashes[i] = -1;
  return -1;
}

/* hashes[B][L][n_layers][C], C = (max_ngram - 1) * n_heads.
 * cache[max_batch][cache_len] int64 holds compressed tokens across calls; sequence b uses row b,
 * or row cache_rows[b] when cache_rows is not NULL (rows of one call must differ).
 * multipliers[n_layers][max_ngram], primes[n_layers][max_ngram-1][n_heads],
 * offsets[n_layers][C]. mask may be NULL (every token takes part). */
int oracle_engram_hash(int64_t n_layers, int64_t max_ngram, int64_t n_heads,
                       const int64_t* token_map, int64_t raw_vocab, int64_t dead, int64_t pad_id,
                       const int64_t* multipliers, const int64_t* primes, const int64_t* offsets,
                       int64_t* cache, int64_t max_batch, int64_t cache_len,
                       const int64_t* ids, const uint8_t* mask, const int64_t* start_pos, const int64_t* cache_rows,
                       int64_t B, int64_t L, int64_t* hashes, uint32_t* flags) {
  if (n_layers < 1 || max_ngram < 2 || max_ngram > 64 || n_heads < 1 || B < 0 || L < 0) return ORACLE_EINVAL;
  if (B > max_batch) return ORACLE_EINVAL;
  const int64_t C = (max_ngram - 1) * n_heads;
  uint32_t fl = 0;
  for (int64_t b = 0; b < B; ++b) {
    int64_t* h = hashes + b * L * n_layers * C;
    const int64_t r = cache_row_of(cache_rows, b, max_batch, L, n_layers * C, h);
    if (r < 0) {
      fl |= ORACLE_FLAG_BAD_ROW;
      continue;
    }
    fl |= hash_sequence(n_layers, max_ngram, n_heads, token_map, raw_vocab, dead, pad_id, multipliers, primes,
                        offsets, cache + r * cache_len, cache_len, ids + b * L, mask ? mask + b * L : NULL,
                        start_pos[b], L, h);
  }
  if (flags) *flags |= fl;
  return ORACLE_OK;
}

/* Packed sequences: sequence b holds tokens cu_seqlens[b] .. cu_seqlens[b+1]-1 of ids/mask/hashes
 * (hashes [T][n_layers][C]) and uses cache row b (or cache_rows[b]) from position start_pos[b]. */
int oracle_engram_hash_varlen(int64_t n_layers, int64_t max_ngram, int64_t n_heads,
                              const int64_t* token_map, int64_t raw_vocab, int64_t dead, int64_t pad_id,
                              const int64_t* multipliers, const int64_t* primes, const int64_t* offsets,
                              int64_t* cache, int64_t max_batch, int64_t cache_len,
                              const int64_t* ids, const uint8_t* mask, const int64_t* cu_seqlens,
                              const int64_t* start_pos, const int64_t* cache_rows, int64_t B, int64_t* hashes,
                              uint32_t* flags) {
  if (n_layers < 1 || max_ngram < 2 || max_ngram > 64 || n_heads < 1 || B < 0) return ORACLE_EINVAL;
  if (B > max_batch) return ORACLE_EINVAL;
  const int64_t C = (max_ngram - 1) * n_heads;
  uint32_t fl = 0;
  for (int64_t b = 0; b < B; ++b) {
    const int64_t begin = cu_seqlens[b], L = cu_seqlens[b + 1] - cu_seqlens[b];
    if (L < 0) return ORACLE_EINVAL;
    int64_t* h = hashes + begin * n_layers * C;
    const int64_t r = cache_row_of(cache_rows, b, max_batch, L, n_layers * C, h);
    if (r < 0) {
      fl |= ORACLE_FLAG_BAD_ROW;
      continue;
    }
    fl |= hash_sequence(n_layers, max_ngram, n_heads, token_map, raw_vocab, dead, pad_id, multipliers, primes,
                        offsets, cache + r * cache_len, cache_len, ids + begin, mask ? mask + begin : NULL,
                        start_pos[b], L, h);
  }
  if (flags) *flags |= fl;
  return ORACLE_OK;
}

/* ---------------------------------------------------------------- fp8 row lookup */

/* Scale i of a scale tensor stored as `scale_dtype`, widened to fp32. */
static float scale_at(const void* S, int64_t scale_dtype, int64_t i) {
  switch (scale_dtype) {
    case ORACLE_SCALE_BF16: return oracle_bf16_to_f32(((const uint16_t*)S)[i]);
    case ORACLE_SCALE_E8M0: return oracle_e8m0_to_f32(((const uint8_t*)S)[i]);
    case ORACLE_SCALE_E4M3: return oracle_fp8_e4m3_to_f32(((const uint8_t*)S)[i]);
    default: return ((const float*)S)[i];
  }
}

/* out[n_idx][D] bf16 bits. W[rows][D] E4M3 codes, S[rows][D / block] scales stored as
 * scale_dtype (ORACLE_SCALE_*). An index outside [0, rows) gives a row of +0. */
int oracle_engram_lookup(const int64_t* idx, int64_t n_idx, const uint8_t* W, const void* S, int64_t rows,
                         int64_t D, int64_t block, int64_t scale_dtype, uint16_t* out) {
  if (n_idx < 0 || D < 1 || block < 1 || D % block != 0) return ORACLE_EINVAL;
  if (scale_dtype < ORACLE_SCALE_F32 || scale_dtype > ORACLE_SCALE_E4M3) return ORACLE_EINVAL;
  const int64_t n_scales = D / block;
  for (int64_t i = 0; i < n_idx; ++i) {
    const int64_t r = idx[i];
    const int out_of_range = (r < 0 || r >= rows);
    const int64_t local = out_of_range ? 0 : r; /* masked_fill(mask, 0) */
    for (int64_t k = 0; k < D; ++k) {
      uint16_t y = 0;
      if (!out_of_range) {
        const float value = oracle_fp8_e4m3_to_f32(W[local * D + k]);
        const float scale = scale_at(S, scale_dtype, local * n_scales + k / block);
        const float prod = value * scale; /* one fp32 multiply, round to nearest */
        y = oracle_bf16_rne(prod);
      }
      out[i * D + k] = y; /* masked rows: +0 */
    }
  }
  return ORACLE_OK;
}
