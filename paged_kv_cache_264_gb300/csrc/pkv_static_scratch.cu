// pkv_static_scratch.cu -- a decode entry point that allocates nothing.
//
// pkv_paged_attention_decode needs device scratch (the split-K partials) that its
// caller allocates.  Some callers cannot allocate device memory where they decode: a
// plugin hosted by another runtime that owns the whole device-memory budget and hands
// its plugins no allocator, or a latency-critical serving loop that must not call
// cudaMalloc (which can synchronise the device and takes allocator locks).  For them,
// pkv_paged_attention_decode_static_scratch runs the same decode with its scratch in a
// fixed array that lives in this library's device image.
//
// The array is PKV_STATIC_SCRATCH_BYTES (16 MiB).  Every GPU that loads the library
// holds it until the process exits.  All calls on one device share it and it keeps the
// last call's contents; nothing in it has to start at zero, because each call writes
// every partial it later reads.  Two calls whose kernels overlap on the GPU (different
// streams, or different host threads) race on the array and must be serialised.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/pagedkv.h"
#include "pkv_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[PKV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;
thread_local char g_msg[160] = "no error";

// Device address of the scratch array on device `dev`, which is current.  The host-side
// name of the array is only a stand-in, so the address is looked up once per device
// (with that device current) and cached.
pkv_status scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) {
    std::snprintf(g_msg, sizeof g_msg, "device %d is beyond the %d devices this call serves", dev,
                  kMaxDevices);
    return PKV_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || !p) {
      std::snprintf(g_msg, sizeof g_msg, "cudaGetSymbolAddress(static scratch): %s",
                    cudaGetErrorString(e));
      return PKV_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" {

PKV_API const char* pkv_static_scratch_error(void) { return g_msg; }

PKV_API pkv_status pkv_paged_attention_decode_static_scratch(
    const pkv_pool* pool, const void* q, const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* context_lens, int num_seqs, int num_q_heads, int max_context_len, float scale,
    void* out, void* stream) {
  std::snprintf(g_msg, sizeof g_msg, "no error");
  size_t need = 0;
  pkv_status st = pkv_decode_workspace_bytes(pool, num_seqs, num_q_heads, max_context_len,
                                             nullptr, &need);
  if (st != PKV_OK) {
    std::snprintf(g_msg, sizeof g_msg, "%s (batch shape)", pkv_status_string(st));
    return st;
  }
  // The scratch address and the kernels belong to the current device: it must be the
  // pool's, or the kernels would pair one GPU's scratch with another GPU's pool.
  int dev = -1;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    std::snprintf(g_msg, sizeof g_msg, "cudaGetDevice: %s", cudaGetErrorString(e));
    return PKV_ERR_CUDA;
  }
  if (dev != pkv::pool_device(pool)) {
    std::snprintf(g_msg, sizeof g_msg, "device %d is current but the pool lives on device %d", dev,
                  pkv::pool_device(pool));
    return PKV_ERR_INVALID_ARG;
  }
  if (need > PKV_STATIC_SCRATCH_BYTES) {
    std::snprintf(g_msg, sizeof g_msg,
                  "decode needs %zu bytes of scratch; the static scratch holds %zu",
                  need, static_cast<size_t>(PKV_STATIC_SCRATCH_BYTES));
    return PKV_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  if (need > 0) {
    st = scratch_address(dev, &scratch);
    if (st != PKV_OK) return st;
  }
  st = pkv_paged_attention_decode(pool, q, block_tables, max_blocks_per_seq, context_lens,
                                  num_seqs, num_q_heads, max_context_len, scale, out, scratch,
                                  need > 0 ? static_cast<size_t>(PKV_STATIC_SCRATCH_BYTES) : 0,
                                  stream);
  if (st != PKV_OK)
    std::snprintf(g_msg, sizeof g_msg, "%s%s", pkv_status_string(st),
                  st == PKV_ERR_CUDA ? " (pkv_last_cuda_error() has the CUDA text)" : "");
  return st;
}

}  // extern "C"
