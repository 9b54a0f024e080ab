// pkv_api.cu -- the C ABI declared in include/pagedkv.h: argument validation, the
// decode plan (partition size), workspace layout and kernel dispatch.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>

#include "../../include/pagedkv.h"
#include "pkv_internal.h"

namespace pkv {
int ctas_per_sm_bf16(int head_dim, int cols);
int ctas_per_sm_int8(int head_dim, int cols);
int ctas_per_sm_fp8(int head_dim, int cols);
}  // namespace pkv

struct pkv_pool {
  int64_t num_blocks;
  int kv_heads;
  int head_dim;
  pkv_kv_dtype dtype;
  void* k_cache;
  void* v_cache;
  float* k_scale;
  float* v_scale;
  uint32_t* d_err;  // library-owned device error word
  int device;
  int sm_count;
  bool has_tmaps;    // tensor maps below are valid (the tensor-core kernel can run)
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
};

namespace {

std::atomic<uint64_t> g_launches{0};
thread_local char g_cuda_msg[256] = "no error";

pkv_status cuda_fail(cudaError_t e, const char* where) {
  std::snprintf(g_cuda_msg, sizeof g_cuda_msg, "%s: %s (%d)", where, cudaGetErrorString(e),
                static_cast<int>(e));
  return PKV_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_dtype(pkv_kv_dtype d) { return d == PKV_KV_BF16 || d == PKV_KV_INT8 || d == PKV_KV_FP8_E4M3; }
bool scaled_dtype(pkv_kv_dtype d) { return d == PKV_KV_INT8 || d == PKV_KV_FP8_E4M3; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

constexpr int kMaxQueries = 16;  // query tokens per sequence in one call

// Query tokens per sequence that the options ask for (0 or absent: 1); -1 if invalid.
int num_queries_of(const pkv_decode_options* opt) {
  if (!opt || opt->num_queries == 0) return 1;
  return opt->num_queries >= 1 && opt->num_queries <= kMaxQueries ? opt->num_queries : -1;
}

// Smallest power of two >= n (n >= 1).
int pow2_at_least(int n) {
  int c = 1;
  while (c < n) c <<= 1;
  return c;
}

constexpr int kMaxPartitionBlocks = 1024;
constexpr int kItemBlocksCudaCore = 128;   // blocks per work item, before shrinking to fill the GPU
constexpr int kItemBlocksTensorCore = 64;

struct Plan {
  int kernel;  // PKV_KERNEL_CUDA_CORE or PKV_KERNEL_TENSOR_CORE
  int cols;    // query-column slots of the kernel variant
  int chunks;  // column chunks per kv head: cols * chunks >= group * num_queries
  int num_queries;
  int window;  // tokens each query sees back from its own position (pkv::kNoWindow: all)
  int shape;   // tensor-core ring shape index
  int persistent;
  int ctas_per_sm;
  int partition_blocks;
  int max_parts;
  int kernels;
  size_t ws_bytes;
  size_t ws_ml_offset;
};

pkv_status make_plan(const pkv_pool* pool, int num_seqs, int num_q_heads, int max_context_len,
                     const pkv_decode_options* opt, Plan* plan) {
  const int group = num_q_heads / pool->kv_heads;
  const int nq = num_queries_of(opt);
  if (nq < 1) return PKV_ERR_INVALID_ARG;
  if (max_context_len < nq) return PKV_ERR_INVALID_ARG;
  const int window = opt ? opt->window : 0;
  if (window < 0) return PKV_ERR_INVALID_ARG;
  plan->window = (window == 0 || window >= pkv::kNoWindow) ? pkv::kNoWindow : window;
  // Blocks one sequence's work can span: the whole context, or with a window the blocks
  // that hold the window of its first query up to its newest token.
  int64_t max_nblk = ceil_div(max_context_len, pkv::kBlockSize);
  // With a window shorter than the longest context, every sequence longer than the window
  // spans this same bound (or one block less): the window, not the lengths, sets the work.
  bool window_bound = false;
  if (plan->window != pkv::kNoWindow) {
    const int64_t span = ceil_div(int64_t(plan->window) + nq - 1, pkv::kBlockSize) + 1;
    if (span < max_nblk) {
      max_nblk = span;
      window_bound = true;
    }
  }
  const auto kv = static_cast<pkv::KvType>(pool->dtype);
  // Query columns per (sequence, kv head): the group's heads times the query tokens.  The
  // tensor-core kernel holds 2 to 16 column slots, the CUDA-core kernel 1 to 8; wider tiles
  // are served in chunks of the largest slot count, each chunk its own work unit (it reads
  // the kv head's blocks again, mostly from L2 since the chunks of a head run together).
  const int ncols = group * nq;
  const int mma_cols = ncols > 16 ? 16 : pow2_at_least(ncols < 2 ? 2 : ncols);
  const int cc_cols = ncols > 8 ? 8 : pow2_at_least(ncols);
  const bool mma_ok = pool->has_tmaps && pkv::mma_supported(kv, pool->head_dim, mma_cols);
  const int want = opt ? opt->kernel : PKV_KERNEL_AUTO;
  if (want != PKV_KERNEL_AUTO && want != PKV_KERNEL_CUDA_CORE && want != PKV_KERNEL_TENSOR_CORE)
    return PKV_ERR_INVALID_ARG;
  if (want == PKV_KERNEL_TENSOR_CORE && !mma_ok) return PKV_ERR_UNSUPPORTED;
  // Automatic choice: the tensor-core kernel wherever it is built, one query column (MHA
  // decode) included -- measured on GB300 it beats the FMA kernel there too (LLaMA-2-7B
  // shape: 154 us against 161 us).
  if (want == PKV_KERNEL_TENSOR_CORE || (want == PKV_KERNEL_AUTO && mma_ok))
    plan->kernel = PKV_KERNEL_TENSOR_CORE;
  else
    plan->kernel = PKV_KERNEL_CUDA_CORE;
  plan->cols = plan->kernel == PKV_KERNEL_TENSOR_CORE ? mma_cols : cc_cols;
  plan->chunks = static_cast<int>(ceil_div(ncols, plan->cols));
  plan->num_queries = nq;
  const int sched = opt ? opt->schedule : PKV_SCHEDULE_AUTO;
  if (sched != PKV_SCHEDULE_AUTO && sched != PKV_SCHEDULE_GRID && sched != PKV_SCHEDULE_PERSISTENT)
    return PKV_ERR_INVALID_ARG;
  plan->persistent = 0;  // decided below, once the partition size is known
  plan->shape = 0;
  const int want_stages = opt ? opt->stages : 0;
  const int want_bps = opt ? opt->blocks_per_stage : 0;
  if (plan->kernel == PKV_KERNEL_TENSOR_CORE) {
    plan->shape = pkv::mma_ring_shape(kv, pool->head_dim, want_stages, want_bps);
    if (plan->shape < 0) return PKV_ERR_UNSUPPORTED;
  } else if (want_stages || want_bps) {
    return PKV_ERR_UNSUPPORTED;
  }
  const bool gen = pkv::mma_needs_general(nq, plan->window, plan->cols);
  int per_sm = plan->kernel == PKV_KERNEL_TENSOR_CORE
                   ? pkv::mma_ctas_per_sm(kv, pool->head_dim, plan->cols, plan->shape, gen)
                   : pkv::decode_ctas_per_sm(kv, pool->head_dim, plan->cols);
  if (plan->kernel == PKV_KERNEL_TENSOR_CORE && per_sm == 0 && !want_stages && !want_bps) {
    // The default ring shape has no variant for this tile (a 16-column merge record needs
    // a deeper ring): take the next built shape.
    for (int sh = 1; sh < 4 && per_sm == 0; ++sh) {
      per_sm = pkv::mma_ctas_per_sm(kv, pool->head_dim, plan->cols, sh, gen);
      if (per_sm > 0) plan->shape = sh;
    }
  }
  if (plan->kernel == PKV_KERNEL_TENSOR_CORE && per_sm == 0) return PKV_ERR_UNSUPPORTED;
  plan->ctas_per_sm = per_sm > 0 ? per_sm : 1;
  int P;
  const int64_t resident = int64_t(pool->sm_count) * plan->ctas_per_sm;
  const int64_t units = int64_t(num_seqs) * pool->kv_heads * plan->chunks;
  bool one_wave = false;
  if (opt && opt->partition_blocks > 0) {
    P = opt->partition_blocks;
  } else if (window_bound && units > 0 && units <= resident) {
    // The window bounds every work unit to about the same number of blocks, and the units
    // fit on the GPU at once: split each into as many equal items as still run in one
    // wave, all concurrently, so that none starts late.  Measured on GB300 (8 sequences of
    // 32768 tokens, 32 kv heads, 4096-token window, 256 units, 3 CTAs per SM): one item
    // per unit on the grid 81.9 us; 2 items (512 CTAs, a second partial wave) 99.2 us;
    // 3 items 84.9 us; the earlier plan (5 items of 52 blocks, persistent) 89.0 us.
    int64_t parts = resident / units;
    if (parts < ceil_div(max_nblk, kMaxPartitionBlocks)) parts = ceil_div(max_nblk, kMaxPartitionBlocks);
    P = static_cast<int>(ceil_div(max_nblk, parts));
    one_wave = true;
  } else {
    // Measured on GB300: items of 128 blocks (CUDA-core kernel, bf16 pools) or 64 blocks
    // (tensor-core kernel, which consumes a block faster, and CUDA-core kernel on INT8/FP8
    // pools, whose items carry half the bytes: 409.6 against 428.0 us on the 256-sequence
    // INT8 batch) balance fewer partials against load balance.  The tensor-core kernel takes
    // 128-block items too when that leaves every sequence in one item (no partials, no
    // reduce kernel) and for 16-column tiles (twice the work per block).
    P = plan->kernel == PKV_KERNEL_TENSOR_CORE || pool->dtype != PKV_KV_BF16 ? kItemBlocksTensorCore
                                                                            : kItemBlocksCudaCore;
    if (plan->kernel == PKV_KERNEL_TENSOR_CORE && (max_nblk <= 128 || plan->cols == 16)) P = 128;
    // Shrink the partition while the batch would not fill the GPU twice over.
    while (P > 4 && units * ceil_div(max_nblk, P) < 2 * resident) P /= 2;
  }
  if (P > kMaxPartitionBlocks) P = kMaxPartitionBlocks;
  if (P > max_nblk) P = static_cast<int>(max_nblk);
  if (P < 1) P = 1;
  if (!(opt && opt->partition_blocks > 0)) {
    // Same number of partitions, equal sizes: the longest sequences split into items of
    // equal work instead of full items and a short remainder (a 257-block window with
    // 64-block items would leave a 1-block item).
    P = static_cast<int>(ceil_div(max_nblk, ceil_div(max_nblk, P)));
  }
  plan->partition_blocks = P;
  plan->max_parts = pkv::partition_count(static_cast<int>(max_nblk), P);
  // Persistent CTAs pay off when the grid would hold idle slots, i.e. when sequences split
  // into different numbers of partitions; with one partition each, or one wave of equal
  // items under a window bound, the grid is exact.
  if (num_seqs <= pkv::kMaxSchedSeqs) {
    if (sched == PKV_SCHEDULE_PERSISTENT) plan->persistent = 1;
    else if (sched == PKV_SCHEDULE_AUTO) plan->persistent = plan->max_parts > 1 && !one_wave;
  }
  plan->kernels = plan->max_parts > 1 ? 2 : 1;
  plan->ws_bytes = 0;
  plan->ws_ml_offset = 0;
  if (plan->max_parts > 1) {
    const size_t rows = size_t(num_seqs) * nq * num_q_heads * plan->max_parts;
    const size_t acc = rows * pool->head_dim * sizeof(float);
    plan->ws_ml_offset = (acc + 255) / 256 * 256;
    plan->ws_bytes = plan->ws_ml_offset + rows * 2 * sizeof(float);
  }
  return PKV_OK;
}

// cuTensorMapEncodeTiled from the driver, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// A 2-D tensor map over a [rows, head_dim] pool: 128-byte boxes of 16 rows, 128-byte
// swizzle.  Token rows of 64 bytes (INT8/FP8 at head_dim 64) are mapped two to a 128-byte
// row: the pool seen as [rows / 2, 128 bytes], boxes of 8 such rows (one 16-token tile).
// Returns false when the layout does not qualify (rows neither whole 128-byte spans nor
// 64 bytes, more than 2^31 rows, or no driver entry point).
bool make_pool_tensor_map(CUtensorMap* map, void* base, pkv_kv_dtype dtype, int head_dim,
                          int64_t rows) {
  const int esz = scaled_dtype(dtype) ? 1 : 2;
  const int row_bytes = head_dim * esz;
  const bool pairs = row_bytes == 64;
  if ((row_bytes % 128 != 0 && !pairs) || rows >= (int64_t(1) << 31)) return false;
  auto encode = tensor_map_encoder();
  if (!encode) return false;
  const int64_t map_rows = pairs ? rows / 2 : rows;  // rows is a multiple of 16
  const int64_t map_cols = pairs ? 128 / esz : head_dim;
  const cuuint64_t dims[2] = {cuuint64_t(map_cols), cuuint64_t(map_rows)};
  const cuuint64_t strides[1] = {cuuint64_t(map_cols) * esz};
  const cuuint32_t box[2] = {cuuint32_t(128 / esz), cuuint32_t(pairs ? pkv::kBlockSize / 2 : pkv::kBlockSize)};
  const cuuint32_t elem_strides[2] = {1, 1};
  const CUresult r = encode(
      map, scaled_dtype(dtype) ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
      2, base, dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

pkv_status check_decode_shape(const pkv_pool* pool, int num_seqs, int num_q_heads,
                              int max_context_len) {
  if (!pool) return PKV_ERR_INVALID_ARG;
  if (num_seqs < 0 || num_q_heads < 1 || max_context_len < 1) return PKV_ERR_INVALID_ARG;
  if (max_context_len >= pkv::kNoWindow) return PKV_ERR_INVALID_ARG;
  if (num_q_heads % pool->kv_heads != 0) return PKV_ERR_INVALID_ARG;
  return PKV_OK;
}

}  // namespace

namespace pkv {
int pool_device(const pkv_pool* pool) { return pool ? pool->device : -1; }

int decode_ctas_per_sm(KvType kv, int head_dim, int cols) {
  // [dtype][head_dim 64/128][column slots]; 0 = not yet queried.  Threads may fill an entry
  // concurrently; they store the same value.
  static std::atomic<int> cache[3][2][9];
  const int di = head_dim == 128 ? 1 : 0;
  const int ki = static_cast<int>(kv);
  if (cols < 1 || cols > 8) return 0;
  std::atomic<int>& slot = cache[ki][di][cols];
  int n = slot.load(std::memory_order_relaxed);
  if (n == 0) {
    n = kv == KvType::kInt8  ? ctas_per_sm_int8(head_dim, cols)
        : kv == KvType::kFp8 ? ctas_per_sm_fp8(head_dim, cols)
                             : ctas_per_sm_bf16(head_dim, cols);
    slot.store(n, std::memory_order_relaxed);
  }
  return n;
}

}  // namespace pkv

extern "C" {

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_WORKSPACE: return "workspace too small";
    case PKV_ERR_CAPACITY: return "out of blocks, sequence slots or table capacity";
  }
  return "unknown status";
}

const char* pkv_last_cuda_error(void) { return g_cuda_msg; }

const char* pkv_version(void) { return "0.1.0"; }

uint64_t pkv_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

pkv_status pkv_pool_bytes(int64_t num_blocks, int kv_heads, int head_dim, pkv_kv_dtype dtype,
                          size_t* kv_bytes_each, size_t* scale_bytes_each) {
  if (num_blocks < 1 || kv_heads < 1 || head_dim < 1) return PKV_ERR_INVALID_ARG;
  if (!valid_dtype(dtype)) return PKV_ERR_INVALID_ARG;
  const size_t esz = scaled_dtype(dtype) ? 1 : 2;
  const size_t rows = size_t(num_blocks) * kv_heads * pkv::kBlockSize;
  if (kv_bytes_each) *kv_bytes_each = rows * head_dim * esz;
  if (scale_bytes_each) *scale_bytes_each = scaled_dtype(dtype) ? rows * sizeof(float) : 0;
  return PKV_OK;
}

pkv_status pkv_pool_create(int64_t num_blocks, int kv_heads, int head_dim, int block_size,
                           pkv_kv_dtype dtype, void* k_cache, void* v_cache, float* k_scale,
                           float* v_scale, pkv_pool** out) {
  if (!out) return PKV_ERR_INVALID_ARG;
  *out = nullptr;
  if (num_blocks < 1 || kv_heads < 1 || head_dim < 1) return PKV_ERR_INVALID_ARG;
  if (!valid_dtype(dtype)) return PKV_ERR_INVALID_ARG;
  if (!k_cache || !v_cache || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_INVALID_ARG;
  if (scaled_dtype(dtype)) {
    if (!k_scale || !v_scale || !aligned16(k_scale) || !aligned16(v_scale)) return PKV_ERR_INVALID_ARG;
  } else if (k_scale || v_scale) {
    return PKV_ERR_INVALID_ARG;
  }
  if (block_size != pkv::kBlockSize) return PKV_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
  // Block ids are int32 in the page table; tile offsets are computed in 64 bits.
  if (num_blocks > INT32_MAX) return PKV_ERR_INVALID_ARG;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  uint32_t* d_err = nullptr;
  e = cudaMalloc(&d_err, 16);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(error word)");
  e = cudaMemset(d_err, 0, 16);
  if (e != cudaSuccess) {
    cudaFree(d_err);
    return cuda_fail(e, "cudaMemset(error word)");
  }
  pkv_pool* pool = new (std::nothrow) pkv_pool;
  if (!pool) {
    cudaFree(d_err);
    return PKV_ERR_INVALID_ARG;
  }
  pool->num_blocks = num_blocks;
  pool->kv_heads = kv_heads;
  pool->head_dim = head_dim;
  pool->dtype = dtype;
  pool->k_cache = k_cache;
  pool->v_cache = v_cache;
  pool->k_scale = k_scale;
  pool->v_scale = v_scale;
  pool->d_err = d_err;
  pool->device = dev;
  pool->sm_count = sms;
  const int64_t rows = num_blocks * kv_heads * pkv::kBlockSize;
  pool->has_tmaps = make_pool_tensor_map(&pool->tmap_k, k_cache, dtype, head_dim, rows) &&
                    make_pool_tensor_map(&pool->tmap_v, v_cache, dtype, head_dim, rows);
  *out = pool;
  return PKV_OK;
}

pkv_status pkv_pool_destroy(pkv_pool* pool) {
  if (!pool) return PKV_OK;
  cudaFree(pool->d_err);
  delete pool;
  return PKV_OK;
}

pkv_status pkv_reshape_and_cache(const pkv_pool* pool, const void* key, const void* value,
                                 const int32_t* slot_mapping, int64_t num_tokens, void* stream) {
  if (!pool || num_tokens < 0) return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!key || !value || !slot_mapping || !aligned16(key) || !aligned16(value))
    return PKV_ERR_INVALID_ARG;
  pkv::CacheParams p{};
  p.key = key;
  p.value = value;
  p.slot_mapping = slot_mapping;
  p.k_cache = pool->k_cache;
  p.v_cache = pool->v_cache;
  p.k_scale = pool->k_scale;
  p.v_scale = pool->v_scale;
  p.err = pool->d_err;
  p.num_tokens = num_tokens;
  p.num_blocks = pool->num_blocks;
  p.kv_heads = pool->kv_heads;
  p.head_dim = pool->head_dim;
  auto s = static_cast<cudaStream_t>(stream);
  cudaError_t e = pool->dtype == PKV_KV_INT8     ? pkv::launch_cache_int8(p, s)
                   : pool->dtype == PKV_KV_FP8_E4M3 ? pkv::launch_cache_fp8(p, s)
                                                    : pkv::launch_cache_bf16(p, s);
  if (e != cudaSuccess) return cuda_fail(e, "reshape_and_cache launch");
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return PKV_OK;
}

pkv_status pkv_copy_blocks(const pkv_pool* pool, const int32_t* pairs, int num_pairs, void* stream) {
  if (!pool || num_pairs < 0) return PKV_ERR_INVALID_ARG;
  if (num_pairs == 0) return PKV_OK;
  if (!pairs || num_pairs > 65535) return PKV_ERR_INVALID_ARG;
  pkv::CacheParams p{};
  p.k_cache = pool->k_cache;
  p.v_cache = pool->v_cache;
  p.k_scale = pool->k_scale;
  p.v_scale = pool->v_scale;
  p.err = pool->d_err;
  p.num_blocks = pool->num_blocks;
  p.kv_heads = pool->kv_heads;
  p.head_dim = pool->head_dim;
  cudaError_t e = pkv::launch_copy_blocks(p, pairs, num_pairs, scaled_dtype(pool->dtype) ? 1 : 2,
                                          static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "copy_blocks launch");
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return PKV_OK;
}

pkv_status pkv_decode_workspace_bytes(const pkv_pool* pool, int num_seqs, int num_q_heads,
                                      int max_context_len, const pkv_decode_options* options,
                                      size_t* bytes) {
  if (!bytes) return PKV_ERR_INVALID_ARG;
  pkv_status st = check_decode_shape(pool, num_seqs, num_q_heads, max_context_len);
  if (st != PKV_OK) return st;
  Plan plan;
  st = make_plan(pool, num_seqs, num_q_heads, max_context_len, options, &plan);
  if (st != PKV_OK) return st;
  *bytes = plan.ws_bytes;
  return PKV_OK;
}

pkv_status pkv_decode_plan(const pkv_pool* pool, int num_seqs, int num_q_heads,
                           int max_context_len, const pkv_decode_options* options,
                           int* partition_blocks, int* max_partitions, int* kernels_per_call,
                           int* kernel) {
  pkv_status st = check_decode_shape(pool, num_seqs, num_q_heads, max_context_len);
  if (st != PKV_OK) return st;
  Plan plan;
  st = make_plan(pool, num_seqs, num_q_heads, max_context_len, options, &plan);
  if (st != PKV_OK) return st;
  if (partition_blocks) *partition_blocks = plan.partition_blocks;
  if (max_partitions) *max_partitions = plan.max_parts;
  if (kernels_per_call) *kernels_per_call = plan.kernels;
  if (kernel) *kernel = plan.kernel;
  return PKV_OK;
}

pkv_status pkv_paged_attention_decode_ex(const pkv_pool* pool, const void* q,
                                         const int32_t* block_tables, int max_blocks_per_seq,
                                         const int32_t* context_lens, int num_seqs,
                                         int num_q_heads, int max_context_len, float scale,
                                         void* out, void* workspace, size_t workspace_bytes,
                                         const pkv_decode_options* options, void* stream) {
  pkv_status st = check_decode_shape(pool, num_seqs, num_q_heads, max_context_len);
  if (st != PKV_OK) return st;
  if (num_seqs == 0) return PKV_OK;
  if (!q || !block_tables || !context_lens || !out || !aligned16(q) || !aligned16(out))
    return PKV_ERR_INVALID_ARG;
  if (max_blocks_per_seq < 1) return PKV_ERR_INVALID_ARG;
  if (int64_t(max_context_len) > int64_t(max_blocks_per_seq) * pkv::kBlockSize)
    return PKV_ERR_INVALID_ARG;
  if (!(scale == scale)) return PKV_ERR_INVALID_ARG;  // NaN
  Plan plan;
  st = make_plan(pool, num_seqs, num_q_heads, max_context_len, options, &plan);
  if (st != PKV_OK) return st;
  if (plan.ws_bytes > 0) {
    if (!workspace || workspace_bytes < plan.ws_bytes) return PKV_ERR_WORKSPACE;
    if (!aligned16(workspace)) return PKV_ERR_INVALID_ARG;
  }

  pkv::DecodeParams p{};
  p.q = q;
  p.k_cache = pool->k_cache;
  p.v_cache = pool->v_cache;
  p.k_scale = pool->k_scale;
  p.v_scale = pool->v_scale;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.out = out;
  p.ws_acc = plan.ws_bytes ? static_cast<float*>(workspace) : nullptr;
  p.ws_ml = plan.ws_bytes
                ? reinterpret_cast<float*>(static_cast<char*>(workspace) + plan.ws_ml_offset)
                : nullptr;
  p.err = pool->d_err;
  p.sched = pool->d_err + 1;
  p.persistent = plan.persistent;
  {
    const int64_t items = int64_t(plan.max_parts) * num_seqs * pool->kv_heads * plan.chunks;
    const int64_t resident = int64_t(pool->sm_count) * plan.ctas_per_sm;
    p.grid = static_cast<int>(items < resident ? items : resident);
  }
  p.num_blocks = pool->num_blocks;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.kv_heads = pool->kv_heads;
  p.group = num_q_heads / pool->kv_heads;
  p.group_log2 = -1;
  for (int l = 0; l < 31; ++l)
    if ((1 << l) == p.group) p.group_log2 = l;
  p.num_queries = plan.num_queries;
  p.window = plan.window;
  p.chunks = plan.chunks;
  p.head_dim = pool->head_dim;
  p.max_context_len = max_context_len;
  p.partition_blocks = plan.partition_blocks;
  p.max_parts = plan.max_parts;
  p.scale_log2 = scale * 1.4426950408889634f;

  auto s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (plan.kernel == PKV_KERNEL_TENSOR_CORE)
    e = pkv::launch_decode_mma(p, &pool->tmap_k, &pool->tmap_v,
                               static_cast<pkv::KvType>(pool->dtype), plan.cols, plan.shape, s);
  else
    e = pool->dtype == PKV_KV_INT8       ? pkv::launch_decode_int8(p, plan.cols, s)
        : pool->dtype == PKV_KV_FP8_E4M3 ? pkv::launch_decode_fp8(p, plan.cols, s)
                                         : pkv::launch_decode_bf16(p, plan.cols, s);
  if (e != cudaSuccess) return cuda_fail(e, "paged_attention_decode launch");
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (plan.max_parts > 1) {
    e = pkv::launch_lse_reduce(p, s);
    if (e != cudaSuccess) return cuda_fail(e, "partition reduce launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
  }
  return PKV_OK;
}

pkv_status pkv_paged_attention_decode(const pkv_pool* pool, const void* q,
                                      const int32_t* block_tables, int max_blocks_per_seq,
                                      const int32_t* context_lens, int num_seqs, int num_q_heads,
                                      int max_context_len, float scale, void* out,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  return pkv_paged_attention_decode_ex(pool, q, block_tables, max_blocks_per_seq, context_lens,
                                       num_seqs, num_q_heads, max_context_len, scale, out,
                                       workspace, workspace_bytes, nullptr, stream);
}

pkv_status pkv_get_device_error(const pkv_pool* pool, uint32_t* flags, void* stream) {
  if (!pool || !flags) return PKV_ERR_INVALID_ARG;
  auto s = static_cast<cudaStream_t>(stream);
  uint32_t h = 0;
  cudaError_t e = cudaMemcpyAsync(&h, pool->d_err, sizeof h, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(error word)");
  e = cudaMemsetAsync(pool->d_err, 0, sizeof h, s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(error word)");
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  *flags = h;
  return PKV_OK;
}

}  // extern "C"
