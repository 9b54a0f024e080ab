// pkv_internal.h -- structures shared by the C-ABI layer and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

struct pkv_pool;  // the C ABI's opaque pool descriptor (include/pagedkv.h)

namespace pkv {

constexpr int kBlockSize = 16;                      // tokens per physical block
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // bounded waits give up after 2 s
constexpr int kMaxSchedSeqs = 4096;  // largest batch scheduled by the persistent grid
constexpr int kNoWindow = 1 << 30;   // window value meaning "no window" (contexts are shorter)

// Partitions of a sequence's nblk blocks for partition size P (decode kernels, partition
// reduce and host plan alike).  They start at multiples of P, so that an item's slice of the
// block table can be requested before its context length is known, and the last one also
// takes a remainder of at most P / 4 blocks instead of leaving it to an item of its own
// (with its own partial to merge): a partition holds up to partition_cap(P) blocks.
__host__ __device__ constexpr int partition_count(int nblk, int P) {
  return nblk - P / 4 <= P ? 1 : (nblk - P / 4 + P - 1) / P;
}
__host__ __device__ constexpr int partition_cap(int P) { return P + P / 4; }
static_assert(partition_count(64, 64) == 1 && partition_count(80, 64) == 1 && partition_count(81, 64) == 2 &&
                  partition_count(1024, 64) == 16 && partition_count(7, 1) == 7 && partition_count(5, 4) == 1,
              "partition_count");

// Device error word bits (mirror PKV_DEVERR_* of the public header).
constexpr uint32_t kErrBlockId = 0x1u;
constexpr uint32_t kErrContextLen = 0x2u;
constexpr uint32_t kErrSlot = 0x4u;
constexpr uint32_t kErrTimeout = 0x8u;

enum class KvType : int { kBf16 = 0, kInt8 = 1, kFp8 = 2 };

struct CacheParams {
  const void* key;              // bf16 [N, Hkv, D]
  const void* value;            // bf16 [N, Hkv, D]
  const int32_t* slot_mapping;  // [N]
  void* k_cache;                // [NB, Hkv, 16, D]
  void* v_cache;
  float* k_scale;               // [NB, Hkv, 16] (int8 only)
  float* v_scale;
  uint32_t* err;
  int64_t num_tokens;
  int64_t num_blocks;
  int kv_heads;
  int head_dim;
};

struct DecodeParams {
  const void* q;                // bf16 [B, k, Hq, D]  (k = num_queries)
  const void* k_cache;          // [NB, Hkv, 16, D]
  const void* v_cache;
  const float* k_scale;         // [NB, Hkv, 16] (int8 only)
  const float* v_scale;
  const int32_t* block_tables;  // [B, max_blocks_per_seq]
  const int32_t* context_lens;  // [B]
  void* out;                    // bf16 [B, k, Hq, D]
  float* ws_acc;                // [B, k, Hq, max_parts, D]   (split only)
  float* ws_ml;                 // [B, k, Hq, max_parts, 2]   (split only): running max (log2 units), sum
  uint32_t* err;
  unsigned* sched;              // [2] work ticket and finished-CTA counters (zero between calls)
  int persistent;               // 1: persistent grid taking items from the ticket counter
  int grid;                     // CTAs to launch in persistent mode
  int64_t num_blocks;
  int max_blocks_per_seq;
  int num_seqs;
  int num_q_heads;
  int kv_heads;
  int group;                    // query heads per kv head (num_q_heads / kv_heads), any >= 1
  int group_log2;               // log2(group) when group is a power of two, else -1
  int num_queries;              // k >= 1 query tokens per sequence, the last k positions
  int chunks;                   // column chunks per kv head: group * k columns are served in
                                // chunks of the variant's column slots, one work unit each
  int window;                   // each query sees its last `window` tokens (kNoWindow: all)
  int head_dim;
  int max_context_len;
  int partition_blocks;         // P: blocks per work item
  int max_parts;                // ceil(ceil(max_context_len / 16) / P)
  float scale_log2;             // softmax scale * log2(e)
};

// Launch a kernel with programmatic stream serialisation (see griddep_wait in
// pkv_device.cuh): its launch may overlap the tail of the previous kernel in the stream.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Kernel launchers (defined next to their kernels).  Each returns the launch status.
cudaError_t launch_cache_bf16(const CacheParams& p, cudaStream_t stream);
cudaError_t launch_cache_int8(const CacheParams& p, cudaStream_t stream);
cudaError_t launch_cache_fp8(const CacheParams& p, cudaStream_t stream);
cudaError_t launch_copy_blocks(const CacheParams& p, const int32_t* pairs, int n, int elem_bytes,
                               cudaStream_t stream);
// The decode kernels serve, per (sequence, kv head), a tile of query columns: column c is
// query token c / group of head kvh * group + c % group.  `cols` is the column slot count
// of the variant to launch: the smallest built power of two >= group * num_queries, or the
// largest built one, the columns then served in chunks of that many.
cudaError_t launch_decode_bf16(const DecodeParams& p, int cols, cudaStream_t stream);
cudaError_t launch_decode_int8(const DecodeParams& p, int cols, cudaStream_t stream);
cudaError_t launch_decode_fp8(const DecodeParams& p, int cols, cudaStream_t stream);
cudaError_t launch_lse_reduce(const DecodeParams& p, cudaStream_t stream);

// Tensor-core decode (2, 4, 8 or 16 column slots): tk/tv are 2-D tensor maps of the K and
// V pools (rows of head_dim elements, 128-byte boxes of 16 rows, 128-byte swizzle).
bool mma_supported(KvType kv, int head_dim, int cols);
// Ring shape (stages x blocks per stage) index for requested values (0 = default); -1 if
// that shape is not built.
int mma_ring_shape(KvType kv, int head_dim, int stages, int blocks_per_stage);
cudaError_t launch_decode_mma(const DecodeParams& p, const CUtensorMap* tk, const CUtensorMap* tv,
                              KvType kv, int cols, int shape, cudaStream_t stream);
// gen: the variant with the general masks (several query tokens or a window).
int mma_ctas_per_sm(KvType kv, int head_dim, int cols, int shape, bool gen);
// Whether a tensor-core call takes the general-mask variant: some query has a causal cut
// or a window, or the tile is 16 columns wide (plain decode of a group of more than 8
// heads; the 16-column tiles are built with the general masks only).
inline bool mma_needs_general(int num_queries, int window, int cols) {
  return num_queries > 1 || window != kNoWindow || cols > 8;
}

// The CUDA device a pool was created on (-1 for NULL).
int pool_device(const pkv_pool* pool);

// Resident CTAs per SM of the CUDA-core decode kernel variant (0 if not built).
int decode_ctas_per_sm(KvType kv, int head_dim, int cols);

}  // namespace pkv
