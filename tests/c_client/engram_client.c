/*
 * A plain C client of libengram: no Python, no torch. It reads a tiny layout and its inputs from
 * raw files, creates a state, runs the fused hash + lookup, the standalone lookup and the lookup
 * inside the wkv projection through the C ABI (include/engram.h) with buffers from cudaMalloc, and
 * writes the results back as raw files.
 * tests/test_gpu_c_client.py builds and runs it and compares the results with the oracle.
 *
 * usage: engram_client DIR   (DIR holds the inputs listed in main() and receives the outputs)
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "engram.h"

static void* slurp(const char* dir, const char* name, size_t* n) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) { fprintf(stderr, "cannot open %s\n", path); exit(2); }
  fseek(f, 0, SEEK_END);
  *n = (size_t)ftell(f);
  fseek(f, 0, SEEK_SET);
  void* p = malloc(*n ? *n : 1);
  if (fread(p, 1, *n, f) != *n) { fprintf(stderr, "short read %s\n", path); exit(2); }
  fclose(f);
  return p;
}

static void spit(const char* dir, const char* name, const void* p, size_t n) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f || fwrite(p, 1, n, f) != n) { fprintf(stderr, "cannot write %s\n", path); exit(2); }
  fclose(f);
}

#define CK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_)); return 3; } } while (0)
#define EK(x) do { int r_ = (x); if (r_ != ENGRAM_OK) { fprintf(stderr, "%s: %s\n", #x, engram_strerror(r_)); return 4; } } while (0)

static void* to_dev(const void* h, size_t n) {
  void* d = NULL;
  if (cudaMalloc(&d, n ? n : 16) != cudaSuccess) return NULL;
  if (n && cudaMemcpy(d, h, n, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
  return d;
}

int main(int argc, char** argv) {
  if (argc != 2) { fprintf(stderr, "usage: %s DIR\n", argv[0]); return 1; }
  const char* dir = argv[1];
  size_t n;
  /* layout.bin: int64 [n_layers, max_ngram, n_heads, head_dim, block, max_batch, max_seq_len, dead, pad, B, L] */
  int64_t* p = (int64_t*)slurp(dir, "layout.bin", &n);
  engram_layout lay;
  lay.n_layers = (int32_t)p[0]; lay.max_ngram = (int32_t)p[1]; lay.n_heads = (int32_t)p[2];
  lay.head_dim = (int32_t)p[3]; lay.block = (int32_t)p[4]; lay.max_batch = (int32_t)p[5];
  lay.max_seq_len = p[6]; lay.dead = p[7]; lay.pad_id = p[8];
  lay.scale_dtype = ENGRAM_SCALE_F32;
  const int32_t B = (int32_t)p[9];
  const int64_t L = p[10];
  size_t n_tm, n_mu, n_pr, n_of, n_ids, n_sp, n_w, n_s;
  const int64_t* tm = (const int64_t*)slurp(dir, "token_map.bin", &n_tm);
  lay.raw_vocab = (int64_t)(n_tm / 8);
  const int64_t* mu = (const int64_t*)slurp(dir, "multipliers.bin", &n_mu);
  const int64_t* pr = (const int64_t*)slurp(dir, "primes.bin", &n_pr);
  const int64_t* of = (const int64_t*)slurp(dir, "offsets.bin", &n_of);
  const int64_t* ids = (const int64_t*)slurp(dir, "ids.bin", &n_ids);
  const int32_t* sp = (const int32_t*)slurp(dir, "start.bin", &n_sp);
  const uint8_t* W = (const uint8_t*)slurp(dir, "W.bin", &n_w);   /* one layer's table, used for every layer */
  const float* S = (const float*)slurp(dir, "S.bin", &n_s);
  const int64_t rows = (int64_t)(n_w / (size_t)lay.head_dim);
  const int64_t C = (int64_t)(lay.max_ngram - 1) * lay.n_heads;

  engram_state* st = NULL;
  EK(engram_state_create(&lay, tm, mu, pr, of, NULL, &st));
  void* d_ids = to_dev(ids, n_ids);
  void* d_sp = to_dev(sp, n_sp);
  void* d_W = to_dev(W, n_w);
  void* d_S = to_dev(S, n_s);
  if (!d_ids || !d_sp || !d_W || !d_S) { fprintf(stderr, "device copy failed\n"); return 3; }
  const size_t hash_bytes = (size_t)B * L * lay.n_layers * C * 8;
  const size_t out_bytes = (size_t)B * L * C * lay.head_dim * 2;
  void* d_hash = NULL;
  CK(cudaMalloc(&d_hash, hash_bytes));
  const uint8_t* Wl[ENGRAM_MAX_LAYERS];
  const void* Sl[ENGRAM_MAX_LAYERS];
  int64_t Rl[ENGRAM_MAX_LAYERS];
  uint16_t* Ol[ENGRAM_MAX_LAYERS];
  for (int l = 0; l < lay.n_layers; ++l) {
    Wl[l] = (const uint8_t*)d_W; Sl[l] = d_S; Rl[l] = rows;
    CK(cudaMalloc((void**)&Ol[l], out_bytes));
  }
  /* call row b uses cache row B-1-b: the reversed map must not change the hash ids */
  int32_t* h_rows = (int32_t*)malloc((size_t)B * sizeof(int32_t));
  for (int32_t b = 0; b < B; ++b) h_rows[b] = B - 1 - b;
  void* d_rows = to_dev(h_rows, (size_t)B * sizeof(int32_t));
  if (!d_rows) { fprintf(stderr, "device copy failed\n"); return 3; }
  EK(engram_hash_lookup(st, (const int64_t*)d_ids, NULL, (const int32_t*)d_sp, (const int32_t*)d_rows, B, L, Wl, Sl,
                        Rl, Ol, (int64_t*)d_hash, NULL));
  /* the standalone lookup of layer 0's hash ids must give layer 0's rows again */
  int64_t* h_hash = (int64_t*)malloc(hash_bytes);
  CK(cudaMemcpy(h_hash, d_hash, hash_bytes, cudaMemcpyDeviceToHost));
  const int64_t n_idx = (int64_t)B * L * C;
  int64_t* idx0 = (int64_t*)malloc((size_t)n_idx * 8);
  for (int64_t t = 0; t < (int64_t)B * L; ++t)
    for (int64_t c = 0; c < C; ++c) idx0[t * C + c] = h_hash[(t * lay.n_layers + 0) * C + c];
  void* d_idx0 = to_dev(idx0, (size_t)n_idx * 8);
  uint16_t* d_rows0 = NULL;
  CK(cudaMalloc((void**)&d_rows0, out_bytes));
  EK(engram_lookup((const int64_t*)d_idx0, n_idx, (const uint8_t*)d_W, d_S, rows, lay.head_dim, lay.block,
                   ENGRAM_SCALE_F32, d_rows0, NULL));
  /* the lookup inside the wkv projection, on layer 0's slice of the hash ids (row stride n_layers * C) */
  size_t n_wkv;
  const uint16_t* wkv = (const uint16_t*)slurp(dir, "wkv.bin", &n_wkv);
  const int64_t K = C * lay.head_dim;
  const int32_t N = (int32_t)(n_wkv / 2 / (size_t)K);
  void* d_wkv = to_dev(wkv, n_wkv);
  if (!d_wkv) { fprintf(stderr, "device copy failed\n"); return 3; }
  engram_table tb;
  tb.W = d_W;
  tb.S = d_S;
  tb.rows = rows;
  tb.head_dim = lay.head_dim;
  tb.block = lay.block;
  tb.scale_dtype = ENGRAM_SCALE_F32;
  const uint64_t ws_bytes = engram_lookup_project_workspace((int64_t)B * L, (int32_t)C, lay.head_dim);
  void* d_ws = NULL;
  CK(cudaMalloc(&d_ws, ws_bytes));
  const size_t kv_bytes = (size_t)B * L * N * 2;
  uint16_t* d_kv = NULL;
  CK(cudaMalloc((void**)&d_kv, kv_bytes));
  EK(engram_lookup_project((const int64_t*)d_hash, (int64_t)lay.n_layers * C, (int64_t)B * L, (int32_t)C, &tb,
                           (const uint16_t*)d_wkv, N, d_ws, ws_bytes, d_kv, NULL));
  uint32_t dflags = 1;
  EK(engram_device_status(NULL, &dflags, 1));
  uint32_t flags = 0;
  EK(engram_state_status(st, NULL, &flags, 1));
  CK(cudaDeviceSynchronize());
  void* h_out = malloc(out_bytes);
  spit(dir, "hashes.out", h_hash, hash_bytes);
  for (int l = 0; l < lay.n_layers; ++l) {
    char name[64];
    snprintf(name, sizeof name, "rows%d.out", l);
    CK(cudaMemcpy(h_out, Ol[l], out_bytes, cudaMemcpyDeviceToHost));
    spit(dir, name, h_out, out_bytes);
  }
  CK(cudaMemcpy(h_out, d_rows0, out_bytes, cudaMemcpyDeviceToHost));
  spit(dir, "lookup0.out", h_out, out_bytes);
  spit(dir, "status.out", &flags, sizeof flags);
  void* h_kv = malloc(kv_bytes);
  CK(cudaMemcpy(h_kv, d_kv, kv_bytes, cudaMemcpyDeviceToHost));
  spit(dir, "kv0.out", h_kv, kv_bytes);
  spit(dir, "device_status.out", &dflags, sizeof dflags);
  EK(engram_state_destroy(st));
  printf("ok\n");
  return 0;
}
