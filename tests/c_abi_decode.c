/*
 * A C program that uses only include/pagedkv.h and the CUDA runtime: it creates a bf16 pool,
 * appends every token of a small batch through pkv_reshape_and_cache, decodes with
 * pkv_paged_attention_decode, and prints the output's bf16 bit patterns, one per line.
 * Inputs (q, K, V bit patterns, block tables, lengths) are read from a binary file written
 * by the test, which compares the printed output with the oracle.
 *
 * Input file layout (little-endian): int32 B, Hq, Hkv, D, num_blocks, max_blocks, N
 * (tokens); float scale; int32 context_lens[B]; int32 block_tables[B * max_blocks];
 * int32 slot_mapping[N]; uint16 q[B * Hq * D]; uint16 key[N * Hkv * D];
 * uint16 value[N * Hkv * D].
 */
#include <cuda_runtime_api.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "pagedkv.h"

#define CHECK_CUDA(x)                                                 \
  do {                                                                \
    cudaError_t e_ = (x);                                             \
    if (e_ != cudaSuccess) {                                          \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));        \
      return 2;                                                       \
    }                                                                 \
  } while (0)
#define CHECK_PKV(x)                                                  \
  do {                                                                \
    pkv_status s_ = (x);                                              \
    if (s_ != PKV_OK) {                                               \
      fprintf(stderr, "%s: %s\n", #x, pkv_status_string(s_));         \
      return 3;                                                       \
    }                                                                 \
  } while (0)

static void* read_n(FILE* f, size_t bytes) {
  void* p = malloc(bytes ? bytes : 1);
  if (p && bytes && fread(p, 1, bytes, f) != bytes) {
    free(p);
    return NULL;
  }
  return p;
}

static void* to_device(const void* host, size_t bytes) {
  void* d = NULL;
  if (cudaMalloc(&d, bytes ? bytes : 16) != cudaSuccess) return NULL;
  if (bytes && cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
  return d;
}

int main(int argc, char** argv) {
  if (argc != 2) {
    fprintf(stderr, "usage: %s input.bin\n", argv[0]);
    return 1;
  }
  FILE* f = fopen(argv[1], "rb");
  if (!f) return 1;
  int32_t hdr[7];
  float scale;
  if (fread(hdr, sizeof hdr, 1, f) != 1 || fread(&scale, sizeof scale, 1, f) != 1) return 1;
  const int B = hdr[0], Hq = hdr[1], Hkv = hdr[2], D = hdr[3], NB = hdr[4], MB = hdr[5], N = hdr[6];
  int32_t* lens = read_n(f, sizeof(int32_t) * B);
  int32_t* tables = read_n(f, sizeof(int32_t) * B * MB);
  int32_t* slots = read_n(f, sizeof(int32_t) * N);
  uint16_t* q = read_n(f, 2 * (size_t)B * Hq * D);
  uint16_t* key = read_n(f, 2 * (size_t)N * Hkv * D);
  uint16_t* value = read_n(f, 2 * (size_t)N * Hkv * D);
  fclose(f);
  if (!lens || !tables || !slots || !q || !key || !value) return 1;
  int max_len = 0;
  for (int b = 0; b < B; ++b) max_len = lens[b] > max_len ? lens[b] : max_len;

  size_t kv_bytes = 0, scale_bytes = 0;
  CHECK_PKV(pkv_pool_bytes(NB, Hkv, D, PKV_KV_BF16, &kv_bytes, &scale_bytes));
  void *k_cache = NULL, *v_cache = NULL;
  CHECK_CUDA(cudaMalloc(&k_cache, kv_bytes));
  CHECK_CUDA(cudaMalloc(&v_cache, kv_bytes));
  pkv_pool* pool = NULL;
  CHECK_PKV(pkv_pool_create(NB, Hkv, D, PKV_BLOCK_SIZE, PKV_KV_BF16, k_cache, v_cache, NULL, NULL, &pool));

  void* d_key = to_device(key, 2 * (size_t)N * Hkv * D);
  void* d_value = to_device(value, 2 * (size_t)N * Hkv * D);
  void* d_slots = to_device(slots, sizeof(int32_t) * N);
  void* d_q = to_device(q, 2 * (size_t)B * Hq * D);
  void* d_tables = to_device(tables, sizeof(int32_t) * B * MB);
  void* d_lens = to_device(lens, sizeof(int32_t) * B);
  void* d_out = NULL;
  CHECK_CUDA(cudaMalloc(&d_out, 2 * (size_t)B * Hq * D));
  if (!d_key || !d_value || !d_slots || !d_q || !d_tables || !d_lens) return 2;

  CHECK_PKV(pkv_reshape_and_cache(pool, d_key, d_value, d_slots, N, NULL));
  size_t ws_bytes = 0;
  CHECK_PKV(pkv_decode_workspace_bytes(pool, B, Hq, max_len, NULL, &ws_bytes));
  void* ws = NULL;
  if (ws_bytes) CHECK_CUDA(cudaMalloc(&ws, ws_bytes));
  CHECK_PKV(pkv_paged_attention_decode(pool, d_q, d_tables, MB, d_lens, B, Hq, max_len, scale, d_out,
                                       ws, ws_bytes, NULL));
  uint32_t flags = 0;
  CHECK_PKV(pkv_get_device_error(pool, &flags, NULL));
  if (flags) {
    fprintf(stderr, "device error flags %u\n", flags);
    return 4;
  }
  uint16_t* out = malloc(2 * (size_t)B * Hq * D);
  CHECK_CUDA(cudaMemcpy(out, d_out, 2 * (size_t)B * Hq * D, cudaMemcpyDeviceToHost));
  for (size_t i = 0; i < (size_t)B * Hq * D; ++i) printf("%u\n", (unsigned)out[i]);
  CHECK_PKV(pkv_pool_destroy(pool));
  return 0;
}
