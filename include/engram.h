/*
 * engram.h -- C ABI of the Engram n-gram hash + fp8 row lookup library (sm_103a).
 *
 * The operation is the Engram front end of the DeepSeek V4.1 block stack, as
 * printed on the "DeepSeek V4.1" pages:
 *   - blocks/stack-hashes page, the n-gram hash `forward(input_ids, start_pos,
 *     token_mask)`: compress raw ids through `token_map`, replace masked tokens
 *     by DEAD, store them in a per-batch cache at [start_pos, start_pos+L), look
 *     back max_ngram-1 positions with cumulative blocking (positions before 0
 *     and DEAD tokens turn that slot and every later slot into pad_id),
 *     multiply the slots by per-layer int64 multipliers, XOR them one lookback
 *     at a time, reduce each running value with a floored mod by per-(n-gram
 *     size, head) primes, and add per-column offsets. Result: int64 hash ids
 *     [B, L, n_layers, C] with C = (max_ngram-1) * n_heads.
 *   - engram-first/lookup page, `ParallelEngramEmbedding.forward` (world size
 *     1): gather fp8 E4M3 rows of a [rows, head_dim] table and their fp32
 *     per-block scales, multiply in fp32, round to bf16 (nearest-even); an index
 *     outside [0, rows) yields a row of +0.
 *
 * Conventions for every call:
 *   - Pointers named "device" must be CUDA device (or managed) memory of the
 *     current device; "host" pointers are ordinary host memory.
 *   - Every compute call is asynchronous on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream), allocates nothing, and never synchronises.
 *   - Arguments are checked on the host before anything is launched; on a
 *     non-zero return nothing was enqueued.
 *   - The library never reads beyond the sizes it is given and never faults on
 *     data values: out-of-range ids, start positions and table indices are
 *     handled as documented below and recorded in the state's status word.
 *   - Caller-owned buffers stay caller-owned; the library only reads inputs and
 *     tables and writes the outputs it is given.
 *   - A state's cache and status word are shared by every call on that state:
 *     calls that may run at the same time (on different streams) must not use
 *     the same cache rows; the library does not order them.
 */
#ifndef ENGRAM_H
#define ENGRAM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* engram_stream_t;

/* Opaque state: device copies of the layout, token_map and the compressed-token cache. */
typedef struct engram_state engram_state;

/* Return codes. */
#define ENGRAM_OK 0
#define ENGRAM_ERR_INVALID (-1)     /* null or misaligned pointer, negative size, inconsistent layout value */
#define ENGRAM_ERR_RANGE (-2)       /* B > max_batch, L > max_seq_len, layer out of range */
#define ENGRAM_ERR_CUDA (-3)        /* a CUDA runtime call or kernel launch failed */
#define ENGRAM_ERR_NOMEM (-4)       /* device allocation failed (engram_state_create only) */
#define ENGRAM_ERR_UNSUPPORTED (-5) /* a size beyond the library limits below */

/* Status flags accumulated on the device (read with engram_state_status). */
#define ENGRAM_STATUS_BAD_START 1u /* a row's start_pos was < 0 or start_pos + L > max_seq_len: that row wrote
                                      nothing to the cache, its hash ids are -1 and its looked-up rows are +0 */
#define ENGRAM_STATUS_BAD_ID 2u    /* an input id outside [0, raw_vocab): that token was treated as masked (DEAD) */
#define ENGRAM_STATUS_BAD_LENGTH 4u /* packed calls: a sequence's extent from cu_seqlens was negative, outside
                                       [0, T] or longer than max_len: that sequence was skipped entirely (no cache
                                       write, its hash ids and rows left unwritten) */
#define ENGRAM_STATUS_BAD_ROW 8u   /* a cache_rows entry outside [0, max_batch): that row (sequence) wrote nothing to
                                      the cache, its hash ids are -1 and its looked-up rows are +0 */
#define ENGRAM_STATUS_CHECK 16u    /* checked builds only (compiled with -DENGRAM_CHECKED=1): a hash or fused kernel
                                      skipped a memory access outside the call's buffers. A library bug, never a
                                      data error; release builds do not test for it */
#define ENGRAM_STATUS_TIMEOUT 32u  /* a tensor-core kernel (engram_project, engram_project_gate) gave up a wait that
                                      did not complete within a second: its outputs are undefined. A library or
                                      device fault, never a data error; read with engram_device_status */

/* Storage types of the scale tensors. The engram-first/lookup page leaves `scale_dtype` open and
 * widens the scale with `.float()`; each type below widens to fp32 exactly before the one fp32
 * multiply. Scales are stored like W: [rows][head_dim / block], each of the type's width. */
#define ENGRAM_SCALE_F32 0  /* IEEE binary32 */
#define ENGRAM_SCALE_BF16 1 /* bfloat16: the upper half of a binary32 */
#define ENGRAM_SCALE_E8M0 2 /* OCP UE8M0: 2^(e - 127); e = 255 is NaN */
#define ENGRAM_SCALE_E4M3 3 /* OCP E4M3 (fn), as the table codes */

/* Library limits. */
#define ENGRAM_MAX_LAYERS 8       /* n_layers */
#define ENGRAM_MAX_NGRAM 8        /* max_ngram (>= 2) */
#define ENGRAM_MAX_COLS_TOTAL 512 /* n_layers * (max_ngram - 1) * n_heads */
/* head_dim must be one of 16, 32, 64, 128, 256, 512; block must divide head_dim and be a multiple of 8. */
#define ENGRAM_GATE_MAX_COPIES 8  /* engram_gate: residual copies hc in {1, 2, 4, 8}; dim a multiple of 8 */
#define ENGRAM_MAX_SHARDS 64      /* engram_shard_pack: ranks a table is split over */

typedef struct engram_layout {
  int32_t n_layers;    /* engram layers hashed per call (the config's engram_layer_ids count) */
  int32_t max_ngram;   /* engram_max_ngram_size: n-gram sizes 2..max_ngram are hashed */
  int32_t n_heads;     /* engram_n_heads: one prime per (n-gram size, head) */
  int32_t head_dim;    /* fp8 values per table row (engram_head_dim) */
  int32_t block;       /* fp8 values per fp32 scale (fp8 block size) */
  int32_t max_batch;   /* cache rows: calls take B <= max_batch */
  int64_t max_seq_len; /* cache positions per row */
  int64_t raw_vocab;   /* entries of token_map (the tokenizer vocabulary) */
  int64_t dead;        /* DEAD sentinel stored for masked tokens; must fit int32 */
  int64_t pad_id;      /* token that fills blocked n-gram slots (engram_pad_id) */
  int32_t scale_dtype; /* storage type of the tables' scales, ENGRAM_SCALE_* (0: fp32) */
} engram_layout;

/*
 * Create a state: the hash module of the blocks/stack-hashes page. Its constructor holds the
 * table-independent parameters that the hash `forward` uses -- the token_map compression table,
 * the DEAD sentinel for masked tokens, pad_id for blocked n-gram slots, the per-layer multipliers,
 * the bucket primes and the per-column offsets -- and the compressed-token cache that `forward`
 * writes at [start_pos, start_pos + L) and reads back for the lookback. All of them are copied to
 * the device once; the cache [max_batch, max_seq_len] is allocated and filled with DEAD (the pages
 * do not show its initial contents; DEAD makes history that was never written read as blocked).
 *   token_map   host int64 [raw_vocab]; every value and `dead` must fit in int32
 *   multipliers host int64 [n_layers][max_ngram]
 *   primes      host int64 [n_layers][max_ngram-1][n_heads]; each in [1, 2^62)
 *   offsets     host int64 [n_layers][C], column = (n-2)*n_heads + head for n-gram size n;
 *               offset + prime - 1 must not overflow int64
 * Ownership: the host arrays are read during the call only; the state owns its device copies and
 * the cache until engram_state_destroy. On success *out receives the state; the call synchronises
 * `stream` once. Errors: ENGRAM_ERR_INVALID / _UNSUPPORTED for bad layout values, _NOMEM, _CUDA;
 * on error *out is NULL and nothing stays allocated.
 */
int engram_state_create(const engram_layout* layout, const int64_t* token_map, const int64_t* multipliers,
                        const int64_t* primes, const int64_t* offsets, engram_stream_t stream, engram_state** out);

/* Free the state's device memory (synchronises the device first). NULL is accepted. */
int engram_state_destroy(engram_state* state);

/* Refill the whole cache with DEAD, the state's starting contents (asynchronous on stream): the
 * cache of the hash `forward` (blocks/stack-hashes page) forgets every sequence, so positions below
 * a later call's start_pos read as blocked. Errors: _INVALID (NULL state, another current device),
 * _CUDA. */
int engram_cache_reset(engram_state* state, engram_stream_t stream);

/* Read the accumulated ENGRAM_STATUS_* flags into *flags (synchronises stream); clears them when
 * `clear` is non-zero. The pages have no counterpart: their hash `forward` assumes valid ids and
 * start positions (blocks/stack-hashes page); this library instead records the data errors it
 * handled without faulting. Reading and clearing is one atomic exchange on the device, ordered
 * after the work already enqueued on `stream`; a flag that a kernel on another stream raises
 * concurrently is kept for the next read. Errors: _INVALID, _CUDA. */
int engram_state_status(engram_state* state, engram_stream_t stream, uint32_t* flags, int clear);

/*
 * The n-gram hash (blocks/stack-hashes page, hash `forward`).
 *   ids        device int64 [B][L] raw token ids
 *   mask       device uint8 [B][L] (non-zero = token takes part) or NULL (all take part)
 *   start_pos  device int32 [B]: position of ids[b][0] in row b's cache row (a scalar start is a filled array)
 *   cache_rows device int32 [B] or NULL: row b reads and writes cache row cache_rows[b] (NULL: cache row b).
 *              The pages index the cache by the batch row; the map only renames rows, so a serving loop can
 *              keep each sequence in its own cache row whatever its place in the batch. The entries of one
 *              call must differ (two rows on one cache row would race); an entry outside [0, max_batch) skips
 *              that row and raises ENGRAM_STATUS_BAD_ROW.
 *   hashes     device int64 [B][L][n_layers][C], written
 * Writes cache[r][start_pos[b] + t] (r = row b's cache row) for every valid row. Rows never interact.
 * B == 0 or L == 0 is a no-op. Errors: _INVALID (null, misaligned), _RANGE (B > max_batch, L > max_seq_len),
 * _UNSUPPORTED (B * L > 2^40 or L > 2^32).
 */
int engram_hash(engram_state* state, const int64_t* ids, const uint8_t* mask, const int32_t* start_pos,
                const int32_t* cache_rows, int32_t B, int64_t L, int64_t* hashes, engram_stream_t stream);

/*
 * The fp8 row lookup of one table (engram-first/lookup page, `ParallelEngramEmbedding.forward`, world size 1).
 *   idx          device int64 [n_idx] row indices; an index outside [0, rows) gives a row of +0
 *   W            device fp8 E4M3 codes [rows][head_dim], 16-byte aligned
 *   S            device scales [rows][head_dim / block] stored as scale_dtype, aligned to its width
 *   scale_dtype  ENGRAM_SCALE_*
 *   out          device bf16 bits [n_idx][head_dim], 16-byte aligned, written
 * out[i][k] = bf16_rne(fp32(W[idx[i]][k]) * fp32(S[idx[i]][k / block])) (one fp32 round-to-nearest multiply).
 * n_idx == 0 is a no-op. Errors: _INVALID, _UNSUPPORTED (head_dim / block / scale_dtype).
 */
int engram_lookup(const int64_t* idx, int64_t n_idx, const uint8_t* W, const void* S, int64_t rows,
                  int32_t head_dim, int32_t block, int32_t scale_dtype, uint16_t* out, engram_stream_t stream);

/*
 * Hash and lookup in one launch, as one forward of the model does: `Transformer.forward`
 * (blocks/stack-hashes page) calls the hash module once for all engram layers and hands each
 * engram layer its slice [:, :, l, :] of the hash ids, and that layer's embedding
 * (`ParallelEngramEmbedding.forward`, engram-first/lookup page, world size 1) turns the slice into
 * rows of its own table. So: the hash of engram_hash (same cache update), then for every layer l
 * the lookup of its C columns in table l, with the row ids kept on chip.
 *   W, S, rows, out  host arrays of n_layers entries: per layer the device table, scales (stored as the
 *                    layout's scale_dtype), row count (as engram_lookup) and a device bf16 output
 *                    [B][L][C][head_dim]
 *   hashes           device int64 [B][L][n_layers][C] to also receive the hash ids, or NULL
 * Errors: as engram_hash and engram_lookup.
 */
int engram_hash_lookup(engram_state* state, const int64_t* ids, const uint8_t* mask, const int32_t* start_pos,
                       const int32_t* cache_rows, int32_t B, int64_t L, const uint8_t* const* W,
                       const void* const* S, const int64_t* rows, uint16_t* const* out, int64_t* hashes,
                       engram_stream_t stream);

/*
 * Packed (variable-length) sequences, for continuous batching: B sequences of different lengths are
 * concatenated into one token array (an extension: the pages' hash `forward`, blocks/stack-hashes
 * page, takes one [B, L] batch at one start position). Sequence b holds tokens cu_seqlens[b] .. cu_seqlens[b+1]-1,
 * sits at positions start_pos[b] .. of its cache row (b, or cache_rows[b]), and is hashed exactly as
 * engram_hash would hash it alone (blocks/stack-hashes page, hash `forward`, applied per sequence).
 *   ids         device int64 [T] raw token ids
 *   mask        device uint8 [T] or NULL
 *   cu_seqlens  device int32 [B+1], non-decreasing, cu_seqlens[0] = 0 and cu_seqlens[B] = T expected
 *   start_pos   device int32 [B]
 *   cache_rows  device int32 [B] or NULL: the cache row of sequence b, as in engram_hash
 *   max_len     host: an upper bound on every sequence's length (a longer one is skipped and flagged;
 *               max_len <= max_seq_len)
 *   hashes      device int64 [T][n_layers][C]
 * A sequence whose extent is inconsistent is skipped and flagged (ENGRAM_STATUS_BAD_LENGTH); a start
 * position that does not fit is handled as in engram_hash. Where cu_seqlens decreases, the sequence at
 * the decrease is flagged and skipped and which other sequences are processed is unspecified: once a
 * call raises ENGRAM_STATUS_BAD_LENGTH, treat every output of that call (hash ids, rows, and the
 * cache positions it was to write) as undefined, valid sequences included. Extents
 * must not overlap (tokens shared by two sequences would be written twice). B == 0, T == 0 or
 * max_len == 0 is a no-op. The launch has floor(T / tile) + B CTAs (tile: 4 to 64 tokens), each
 * taking one tile of one sequence, so its cost follows T, not B x max_len.
 * Errors: _INVALID (null, misaligned, negative sizes), _RANGE (B > max_batch, max_len > max_seq_len),
 * _UNSUPPORTED (T > 2^31 - 1).
 */
int engram_hash_varlen(engram_state* state, const int64_t* ids, const uint8_t* mask, const int32_t* cu_seqlens,
                       const int32_t* start_pos, const int32_t* cache_rows, int32_t B, int64_t T, int64_t max_len,
                       int64_t* hashes, engram_stream_t stream);

/*
 * Packed sequences, hash and lookup in one launch (as engram_hash_lookup: `Transformer.forward`'s
 * one hash call and each layer's `ParallelEngramEmbedding.forward`, applied per sequence): out[l] is device bf16
 * [T][C][head_dim] for layer l, hashes ([T][n_layers][C]) may be NULL. Other arguments and errors as
 * engram_hash_varlen and engram_hash_lookup.
 */
int engram_hash_lookup_varlen(engram_state* state, const int64_t* ids, const uint8_t* mask,
                              const int32_t* cu_seqlens, const int32_t* start_pos, const int32_t* cache_rows,
                              int32_t B, int64_t T, int64_t max_len, const uint8_t* const* W, const void* const* S,
                              const int64_t* rows, uint16_t* const* out, int64_t* hashes, engram_stream_t stream);

/*
 * The Engram gate (blocks/stack-hashes page, `Engram.forward`, after the `wkv` projection), in fp32:
 * for every token t and residual copy i,
 *   rstd = rsqrt(mean(h^2) + eps) * rsqrt(mean(key_i^2) + eps),  h = x[t][i]
 *   dot  = sum(h * q_weight[i] * k_weight[i] * key_i) * rstd * dim^-0.5
 *   gate = sigmoid(copysign(sqrt(max(|dot|, 1e-6)), dot)), and 0 where mask[t] == 0
 *   out[t][i] = bf16_rne(h + gate * value)
 *   x        device bf16 [T][hc][dim] (the residual copies)
 *   kv       device bf16 [T][(hc+1)*dim]: the projection output, hc keys then one shared value
 *   q_weight, k_weight  device bf16 [hc][dim]
 *   mask     device uint8 [T] (non-zero = the token's gate is open) or NULL
 *   out      device bf16 [T][hc][dim]; may be the same buffer as x
 * All bf16 pointers 16-byte aligned. T == 0 is a no-op. Errors: _INVALID, _UNSUPPORTED (hc, dim).
 */
int engram_gate(const uint16_t* x, const uint16_t* kv, const uint16_t* q_weight, const uint16_t* k_weight,
                const uint8_t* mask, int64_t T, int32_t hc, int32_t dim, float eps, uint16_t* out,
                engram_stream_t stream);

/*
 * The Engram `wkv` projection on the tensor cores (blocks/stack-hashes page, `Engram.forward`:
 * kv = wkv(embedding rows flattened over the hash columns)):
 *   out[t][n] = bf16_rne( sum_k emb[t][k] * w[n][k] )      for t < T, n < N
 * with bf16 inputs and fp32 accumulation (the sum is formed in an unspecified order).
 *   emb  device bf16 [T][K] (for the Engram block: a lookup output [T][C][head_dim], K = C * head_dim)
 *   w    device bf16 [N][K] (the weight as `Linear` stores it: out_features x in_features)
 *   out  device bf16 [T][N], written
 * All three 16-byte aligned; K and N multiples of 8 (rows stay 16-byte aligned), K >= 8, N >= 8.
 * T == 0 is a no-op. A kernel fault that stops progress raises ENGRAM_STATUS_TIMEOUT instead of
 * hanging (engram_device_status). Errors: _INVALID (null, misaligned, negative T), _UNSUPPORTED
 * (K or N not a multiple of 8 or below 8, T >= 2^31, N > 2^31 - 256), _CUDA.
 */
int engram_project(const uint16_t* emb, const uint16_t* w, int64_t T, int32_t K, int32_t N, uint16_t* out,
                   engram_stream_t stream);

/*
 * Test hook of engram_project's failure path (no counterpart in the pages): the same call, except
 * that in every cluster of CTAs the projection never signals that its tile number `tile` (counted
 * from 0 per cluster) is complete. That tile's epilogue then waits until its one-second limit runs
 * out, the kernel raises ENGRAM_STATUS_TIMEOUT (engram_device_status), stops, waits for its own
 * copies and MMAs in flight, frees its tensor memory and ends instead of hanging; the output is
 * undefined and the context stays usable. Errors: as engram_project, and _INVALID for tile < 0.
 */
int engram_project_withhold(const uint16_t* emb, const uint16_t* w, int64_t T, int32_t K, int32_t N, uint16_t* out,
                            int32_t tile, engram_stream_t stream);

/* Bytes of device workspace that engram_project_gate needs for T tokens (a multiple of 256). */
uint64_t engram_project_gate_workspace(int64_t T, int32_t hc, int32_t dim);

/*
 * The Engram block after the lookup, fused (blocks/stack-hashes page, `Engram.forward`): the `wkv`
 * projection kv = emb @ wkv^T (as engram_project, bf16 keys and value), then the gate of engram_gate
 * on it, in two launches that never write the keys to memory:
 *   1. the projection; the epilogue of each key tile turns its accumulators (rounded to bf16, the
 *      projection's output type) into per-row partial sums of h^2, key^2 and h*q_weight*k_weight*key
 *      over the tile's 256 columns, and each value tile stores its bf16 value rows;
 *   2. per token: the partial sums give the hc gates (as engram_gate), then
 *      out[t][i] = bf16_rne(h + gate * value).
 *   x         device bf16 [T][hc][dim] (the residual copies h)
 *   emb       device bf16 [T][K] (the lookup rows, flattened)
 *   wkv       device bf16 [(hc+1)*dim][K]: hc key blocks of dim rows, then the value block
 *   q_weight, k_weight  device bf16 [hc][dim]
 *   mask      device uint8 [T] (non-zero = the token's gate is open) or NULL
 *   workspace device memory of at least engram_project_gate_workspace(T, hc, dim) bytes, 256-byte
 *             aligned, owned by the caller; holds the value rows and the partial sums between the
 *             two launches, so calls that use one workspace must not overlap on the GPU
 *   out       device bf16 [T][hc][dim]; may be the same buffer as x
 * The result equals engram_gate(x, engram_project(emb, wkv), ...) up to the fp32 summation order.
 * hc in {1, 2, 4, 8}; dim a multiple of 256; K a multiple of 8, K >= 8. T == 0 is a no-op.
 * Errors: _INVALID (null, misaligned, workspace too small), _UNSUPPORTED (hc, dim, K, T >= 2^31), _CUDA.
 */
int engram_project_gate(const uint16_t* x, const uint16_t* emb, const uint16_t* wkv, const uint16_t* q_weight,
                        const uint16_t* k_weight, const uint8_t* mask, int64_t T, int32_t K, int32_t hc, int32_t dim,
                        float eps, void* workspace, uint64_t workspace_bytes, uint16_t* out, engram_stream_t stream);

/*
 * One layer's table, as engram_lookup takes it: fp8 E4M3 codes W [rows][head_dim] (16-byte
 * aligned), scales S [rows][head_dim / block] stored as scale_dtype (ENGRAM_SCALE_*; aligned to
 * their size). rows == 0 is an empty table (every row +0; W and S may then be NULL).
 */
typedef struct engram_table {
  const void* W;
  const void* S;
  int64_t rows;
  int32_t head_dim;
  int32_t block;
  int32_t scale_dtype;
} engram_table;

/* Bytes of device workspace that engram_lookup_project needs (a multiple of 256; 0 for T <= 0 or
 * n_cols * head_dim <= 0): the looked-up bf16 rows [T][n_cols * head_dim] and a few counters. */
uint64_t engram_lookup_project_workspace(int64_t T, int32_t n_cols, int32_t head_dim);

/*
 * The lookup and the `wkv` projection after it in one kernel (blocks/stack-hashes page,
 * `Engram.forward`: kv = wkv(embed(hash ids) flattened over the hash columns); the embedding is
 * `ParallelEngramEmbedding.forward` of the engram-first/lookup page):
 *   emb[t][c * head_dim + k] = the bf16 row of engram_lookup for table row idx[t * idx_stride + c]
 *   out[t][n] = bf16_rne( sum_k emb[t][k] * wkv[n][k] )        (fp32 accumulation)
 * equal bit for bit to engram_lookup followed by engram_project. Warps of every CTA of the projection
 * look the rows up into the workspace one tile group (4,096 tokens) ahead of the tensor-core loads
 * that read them, which read them back from L2; only the first group's lookup runs before the first
 * MMA. On GB300, in steady state, this is 0.5% faster than the two calls at 65,536 tokens and 0.4%
 * slower at 16,384 (the lookup inside the contraction still costs the tensor cores about its own
 * time). Inputs written by an earlier launch on the stream are read after it completes.
 *   idx         device int64: token t's n_cols row ids at idx[t * idx_stride + c] (8-byte aligned;
 *               idx_stride >= n_cols), e.g. one layer's slice of engram_hash's output (stride
 *               n_layers * C); ids outside [0, rows) give +0 rows
 *   table       host pointer to the layer's table; head_dim and block as engram_lookup
 *   wkv         device bf16 [N][n_cols * head_dim]; out  device bf16 [T][N], written
 *   workspace   device memory of engram_lookup_project_workspace(T, n_cols, head_dim) bytes, 256-byte
 *               aligned, owned by the caller; calls that use one workspace must not overlap on the GPU
 * N a multiple of 8, N >= 8. T == 0 is a no-op. A wait that does not end (a lookup warp or load that
 * stops progressing) raises ENGRAM_STATUS_TIMEOUT (engram_device_status) after one second instead of
 * hanging. Errors: _INVALID (null, misaligned, idx_stride < n_cols, workspace too small), _UNSUPPORTED
 * (head_dim, block, scale_dtype as engram_lookup; N; T >= 2^31), _CUDA.
 */
int engram_lookup_project(const int64_t* idx, int64_t idx_stride, int64_t T, int32_t n_cols,
                          const engram_table* table, const uint16_t* wkv, int32_t N, void* workspace,
                          uint64_t workspace_bytes, uint16_t* out, engram_stream_t stream);

/* Bytes of device workspace that engram_lookup_project_gate needs (a multiple of 256). */
uint64_t engram_lookup_project_gate_workspace(int64_t T, int32_t n_cols, int32_t head_dim, int32_t hc, int32_t dim);

/*
 * The whole Engram block for one layer from its hash ids (blocks/stack-hashes page, `Engram.forward`):
 * the lookup of engram_lookup_project inside the projection of engram_project_gate, whose epilogue
 * turns the key tiles into the gate's partial sums, then the gate's finishing pass:
 *   out[t][i] = bf16_rne(h + gate * value),  h = x[t][i]
 * equal bit for bit to engram_lookup, then engram_project_gate. Arguments as engram_lookup_project and
 * engram_project_gate (wkv [(hc + 1) * dim][n_cols * head_dim]; x, out [T][hc][dim]; out may be x);
 * workspace of engram_lookup_project_gate_workspace(T, n_cols, head_dim, hc, dim) bytes.
 * Errors: as engram_lookup_project, and _UNSUPPORTED for hc or dim as engram_project_gate.
 */
int engram_lookup_project_gate(const uint16_t* x, const int64_t* idx, int64_t idx_stride, int64_t T, int32_t n_cols,
                               const engram_table* table, const uint16_t* wkv, const uint16_t* q_weight,
                               const uint16_t* k_weight, const uint8_t* mask, int32_t hc, int32_t dim, float eps,
                               void* workspace, uint64_t workspace_bytes, uint16_t* out, engram_stream_t stream);

/* Read the status flags of the kernels that have no state object (ENGRAM_STATUS_TIMEOUT) for the
 * current device into *flags, ordered after the work already on `stream` (synchronises it); clears
 * them in the same atomic step when `clear` is non-zero. The pages have no counterpart: it reports
 * a failure that the library turns into a flag instead of a hang. Errors: _INVALID, _CUDA. */
int engram_device_status(engram_stream_t stream, uint32_t* flags, int clear);

/*
 * Row-sharded lookup over `world` ranks (engram-first/lookup page, `ParallelEngramEmbedding`: rank r
 * holds rows [r * part, (r + 1) * part) of the table, part = ceil(rows / world)). The pages look up
 * every index on every rank, zero the rows a rank does not own and all-reduce the mostly-zero result;
 * here each request travels only to the rank that owns its row, and only that row travels back:
 *   1. engram_shard_pack groups a rank's indices by owner;
 *   2. an all-to-all exchange (the caller's, e.g. NCCL) sends local_rows bucket r to rank r;
 *   3. each rank looks the rows it received up in its shard (engram_lookup, rows = its shard size);
 *   4. a second all-to-all returns them in the same order;
 *   5. engram_shard_unpack puts them at their positions, +0 rows where no rank owns the index.
 * The result equals engram_lookup on the whole table bit for bit.
 *
 * engram_shard_pack
 *   idx         device int64 [n]: global row ids (any values; those outside [0, rows) are owned by no rank)
 *   rows        the whole table's row count; world in [1, ENGRAM_MAX_SHARDS]
 *   counts      device int64 [world + 1], written: counts[r] = indices owned by rank r, counts[world] =
 *               indices owned by none
 *   local_rows  device int64 [n], written: bucket 0 (rank 0's rows), then bucket 1, ..., then the unowned
 *               indices; inside a bucket in index order; a rank's entries are rows of its shard
 *               (global id - r * part), the unowned entries keep their global id
 *   positions   device int64 [n], written: the index (into idx) of each entry of local_rows
 *   workspace   device memory of engram_shard_pack_workspace(n, world) bytes, 16-byte aligned; calls
 *               that use one workspace must not overlap on the GPU
 * n == 0 is a no-op (counts is not written).
 * Errors: _INVALID (null, misaligned, negative n or rows, workspace too small), _UNSUPPORTED (world,
 * n >= 2^31), _CUDA.
 */
uint64_t engram_shard_pack_workspace(int64_t n, int32_t world);
int engram_shard_pack(const int64_t* idx, int64_t n, int64_t rows, int32_t world, int64_t* counts,
                      int64_t* local_rows, int64_t* positions, void* workspace, uint64_t workspace_bytes,
                      engram_stream_t stream);

/*
 * engram_shard_pack without a workspace, for callers that may not allocate device memory where they
 * pack: a serving loop whose device memory is all handed out up front by its own pool, code running
 * while a stream is captured into a CUDA graph (where a plain cudaMalloc is not allowed), or a hot
 * path that must not take an allocation's latency. The pages have no counterpart: it is a
 * convenience of this library. Same arguments and results as engram_shard_pack, without workspace:
 * the scratch (one int32 per segment of 4096 indices and bucket) is a fixed 64 KB array inside the
 * library, which every device that loads the library holds until the process exits.
 *   limit   n <= floor(16384 / (world + 1)) * 4096 (7,454,720 indices at world 8; 1,028,096 at world
 *           64); a larger n returns ENGRAM_ERR_UNSUPPORTED and launches nothing
 *   set-up  the first call on each device looks up the array's device address there (with that
 *           device current); make that first call before any stream capture
 *   sharing every call on a device uses the same array, and the count pass overwrites every entry a
 *           call reads, so no entry has to start at zero; calls that overlap on the GPU (on different
 *           streams, or unordered) race on it and their results are undefined
 * The call allocates nothing and calls no allocating routine. Errors: as engram_shard_pack.
 */
int engram_shard_pack_static(const int64_t* idx, int64_t n, int64_t rows, int32_t world, int64_t* counts,
                             int64_t* local_rows, int64_t* positions, engram_stream_t stream);

/*
 * engram_shard_unpack: out[positions[i]] = rows[i] for i < m (the rows received back, in the packed
 * order of the owned buckets), and out[positions[i]] = +0 for m <= i < n (the unowned indices).
 *   rows       device bf16 [m][head_dim];  positions  device int64 [n] (from engram_shard_pack)
 *   m          sum of counts[0 .. world-1];  out  device bf16 [n][head_dim], written
 * head_dim a multiple of 8; rows and out 16-byte aligned. n == 0 is a no-op.
 * Errors: _INVALID (null, misaligned, m outside [0, n]), _UNSUPPORTED (head_dim), _CUDA.
 */
int engram_shard_unpack(const uint16_t* rows, const int64_t* positions, int64_t m, int64_t n, int32_t head_dim,
                        uint16_t* out, engram_stream_t stream);

/*
 * Set the L2 fetch granularity limit of the current device's context (cudaLimitMaxL2FetchGranularity:
 * the most bytes L2 fetches from DRAM for one missed sector, a hint; 0, 32, 64 or 128) and return the
 * previous value in *previous (may be NULL). Process-wide for that context and not stream-ordered:
 * call it while none of the process's kernels run, e.g. at set-up; it lasts until the context ends.
 * The library never calls it on its own. At the default (64 on GB300) every random read of up to 128
 * bytes fetches a whole 128-byte line, so a row's 4-byte fp32 scale costs as much DRAM traffic as its
 * 128 bytes of codes; at 32 it costs one 32-byte sector (the full-scale gather then moves ~19% fewer
 * DRAM bytes). Errors: _INVALID (another value), _CUDA.
 */
int engram_set_l2_fetch_granularity(int32_t bytes, int32_t* previous);

/* Layout the state was created with (host copy). */
int engram_state_layout(const engram_state* state, engram_layout* layout);

/* Static text for a return code. */
const char* engram_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* ENGRAM_H */
